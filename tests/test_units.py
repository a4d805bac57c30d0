"""The persistent kernels' work schedule, checked on the host (no GPU).

gemm_plan_work_unit runs the schedule functions the kernels call for every
unit of work, compiled for the host.  For planned problems these tests list
every cluster's units and check what the product's correctness and balance
rest on:

* every (tile, K block) pair is computed exactly once;
* tile indices map one to one onto (batch, m block, n block) inside D;
* a tile split along K (stream-K) has one contributor, K blocks [0, x), and
  one finisher, [x, nk), in neighbouring clusters c-1 and c, which share the
  contributor's partial slot c-1; the contributor is the first unit of its
  cluster and the finisher the last of its cluster's stream-K units, so a
  finisher never waits on a cluster that is itself waiting;
* clusters get equal shares: data-parallel tiles differ by at most one, and
  stream-K ranges by at most one K block;
* raster groups: a wave's tiles walk m blocks first inside a group.
"""
import random

import pytest

import dense_gemm_blackwell_gb300 as dg

GB300 = dg.GemmDeviceProps(sm_count=152, smem_optin_bytes=232448, cc_major=10, cc_minor=3)


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()


def plan(M, N, K, **kw):
    desc = dg.make_desc(M, N, K, **kw)
    s, info = dg.gemm_plan_query(desc, GB300)
    assert s == dg.GEMM_OK, (M, N, K, kw, dg.gemm_status_string(s))
    return desc, info


def units_of(desc, info):
    """{cluster: [unit dict, ...]} in processing order."""
    G = info.grid // info.cta_group
    out = {}
    for c in range(G):
        lst = []
        for i in range(100000):
            s, u = dg.gemm_plan_work_unit(desc, info, c, i)
            assert s == dg.GEMM_OK
            if u.tile < 0:
                break
            lst.append(u.as_dict())
        out[c] = lst
    return out


def check_schedule(desc, info, group=None):
    M, N, K, batch = desc.M, desc.N, desc.K, max(desc.batch, 1)
    nk = -(-K // info.tile_k)
    mb_n, nb_n = -(-M // info.tile_m), -(-N // info.tile_n)
    T = batch * mb_n * nb_n
    assert info.num_tiles == T
    G = info.grid // info.cta_group
    sched = units_of(desc, info)

    covered = {}
    coords = {}
    for c, lst in sched.items():
        for u in lst:
            t = u["tile"]
            assert 0 <= t < T
            assert 0 <= u["k_block_begin"] < u["k_block_end"] <= nk, u
            for kb in range(u["k_block_begin"], u["k_block_end"]):
                assert (t, kb) not in covered, ("computed twice", t, kb)
                covered[(t, kb)] = c
            xy = (u["batch"], u["m_block"], u["n_block"])
            assert 0 <= xy[0] < batch and 0 <= xy[1] < mb_n and 0 <= xy[2] < nb_n, u
            assert coords.setdefault(t, xy) == xy
    assert len(covered) == T * nk, "some (tile, K block) pair is never computed"
    assert len(set(coords.values())) == T, "two tiles map onto the same block of D"

    # stream-K pairs
    sk = info.stream_k_tiles
    by_tile = {}
    for c, lst in sched.items():
        for i, u in enumerate(lst):
            by_tile.setdefault(u["tile"], []).append((c, i, u))
    for t, parts in by_tile.items():
        if len(parts) == 1:
            c, i, u = parts[0]
            assert u["role"] == 0 and (u["k_block_begin"], u["k_block_end"]) == (0, nk)
            continue
        assert sk > 0 and t >= T - sk and len(parts) == 2, (t, parts)
        (c0, i0, u0), (c1, i1, u1) = sorted(parts, key=lambda p: p[2]["k_block_begin"])
        assert u0["role"] == 1 and u1["role"] == 2, (u0, u1)
        assert u0["k_block_end"] == u1["k_block_begin"]
        assert c1 == c0 + 1 and u0["slot"] == u1["slot"] == c0
        assert i0 == 0, "a contributor publishes before its cluster does anything else"
        n_sk = sum(1 for u in sched[c1] if u["tile"] >= T - sk)
        assert i1 == n_sk - 1, "a finisher is its cluster's last stream-K unit"

    # balance
    dp = [sum(1 for u in lst if u["tile"] < T - sk) for lst in sched.values()]
    assert max(dp) - min(dp) <= 1
    if sk:
        kbs = [sum(u["k_block_end"] - u["k_block_begin"] for u in lst if u["tile"] >= T - sk)
               for lst in sched.values()]
        assert max(kbs) - min(kbs) <= 1 and sum(kbs) == sk * nk
        assert min(kbs) >= nk, "every stream-K range is at least one tile long"

    # raster: inside a group, consecutive tiles step m first
    if group:
        for t in range(T - 1):
            b0, m0, n0 = coords[t]
            b1, m1, n1 = coords[t + 1]
            if b0 == b1 and m0 // group == m1 // group and n1 == n0:
                assert m1 == m0 + 1
    return sched


def test_headline_wide_tiles_data_parallel():
    """8192^3 bf16: 512 tiles of 256 x 512 on 76 pairs, raster groups of 16."""
    desc, info = plan(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    assert (info.tile_m, info.tile_n, info.stream_k_tiles) == (256, 512, 0)
    sched = check_schedule(desc, info, group=16)
    counts = sorted(len(v) for v in sched.values())
    assert counts[0] == 6 and counts[-1] == 7        # 512 = 6 * 76 + 56
    # the first wave covers 16 m blocks x 4 (and part of a fifth) n blocks
    first = [sched[c][0] for c in range(76)]
    assert {u["m_block"] for u in first} == set(range(16))


def test_stream_k_region_256_wide():
    """1024 tiles of 256 x 256 on 76 pairs: the last wave plus one full wave
    (76 + 36 tiles) are split along K, the rest run whole."""
    desc, info = plan(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, tile_n=256)
    assert info.stream_k_tiles == 76 + 1024 % 76
    check_schedule(desc, info, group=8)


def test_stream_k_only():
    """80 tiles of 256 x 512 on 76 pairs: every tile is in the stream-K region."""
    desc, info = plan(2048, 5120, 2048, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, tile_n=512)
    assert info.stream_k_tiles == info.num_tiles == 80
    sched = check_schedule(desc, info)
    assert all(u["tile"] >= 0 for lst in sched.values() for u in lst)


def test_batched_and_block_scaled():
    desc, info = plan(256, 256, 256, batch=512, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F16)
    assert info.kernel == dg.GEMM_KERNEL_PERSISTENT
    sched = check_schedule(desc, info)
    assert {u["batch"] for lst in sched.values() for u in lst} == set(range(512))
    desc, info = plan(8192, 8192, 8192, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16,
                      scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    assert info.kernel == dg.GEMM_KERNEL_FP8_BLOCK
    check_schedule(desc, info, group=8)


def test_ragged_and_raster_overrides():
    for kw in (dict(M=1000, N=3000, K=1000, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16),
               dict(M=4000, N=1000, K=5000, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32, raster_group=3),
               dict(M=6000, N=6000, K=700, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                    flags=dg.GEMM_FLAG_CTA_GROUP_1, raster_group=5)):
        desc, info = plan(**kw)
        check_schedule(desc, info, group=kw.get("raster_group"))


def test_random_shapes():
    """Seeded random shapes, CTA groups, tile widths and stage depths."""
    rng = random.Random(7)
    n = 0
    while n < 40:
        M, N, K = (rng.choice([1, 17, 128, 255, 256, 1000, 2048, 3333, 4096]) for _ in range(3))
        kw = dict(dtype_a=rng.choice([dg.GEMM_BF16, dg.GEMM_F16]), dtype_d=dg.GEMM_F32,
                  flags=rng.choice([0, dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2,
                                    dg.GEMM_FLAG_NO_SINGLE_CTA]),
                  max_ctas=rng.choice([0, 0, 8, 30]))
        desc = dg.make_desc(M, N, K, **kw)
        s, info = dg.gemm_plan_query(desc, GB300)
        if s != dg.GEMM_OK or info.kernel != dg.GEMM_KERNEL_PERSISTENT:
            continue
        check_schedule(desc, info)
        n += 1


def test_argument_errors():
    desc, info = plan(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    G = info.grid // info.cta_group
    assert dg.gemm_plan_work_unit(desc, info, G, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    assert dg.gemm_plan_work_unit(desc, info, -1, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    assert dg.gemm_plan_work_unit(desc, info, 0, -1)[0] == dg.GEMM_ERR_INVALID_ARG
    s, u = dg.gemm_plan_work_unit(desc, info, 0, 7)     # cluster 0 has 7 tiles: 0..6
    assert s == dg.GEMM_OK and u.tile == -1
    # an info that is not this desc's plan
    other = dg.make_desc(4096, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    assert dg.gemm_plan_work_unit(other, info, 0, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    zero_n = dg.make_desc(8192, 0, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    assert dg.gemm_plan_work_unit(zero_n, info, 0, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    bad_sk = dg.GemmPlanInfo.from_buffer_copy(info)
    bad_sk.stream_k_tiles = 5                      # fewer than the 76 clusters
    assert dg.gemm_plan_work_unit(desc, bad_sk, 0, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    desc, info = plan(128, 64, 64, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32)
    assert info.kernel == dg.GEMM_KERNEL_SINGLE_CTA
    assert dg.gemm_plan_work_unit(desc, info, 0, 0)[0] == dg.GEMM_ERR_UNSUPPORTED
