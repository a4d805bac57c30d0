"""The persistent kernels' work schedule, checked on the host (no GPU).

gemm_plan_work_unit runs the schedule functions the kernels call for every
unit of work, compiled for the host.  For planned problems these tests list
every cluster's units and check what the product's correctness and balance
rest on:

* every (tile, K block) pair is computed exactly once;
* tile indices map one to one onto (batch, m block, n block) inside D;
* a tile split along K (stream-K) is held by consecutive clusters c0 .. c:
  contributors (K blocks [0, x1), [x1, x2), ...) in c0 .. c-1, each writing
  its own partial slot, and the finisher (the tile's last K blocks) in c,
  which reads slots c-1 down to c0; with ranges at least one tile long that
  is one contributor, c-1.  A contributor is the first unit of its cluster
  and a finisher the last of its cluster's stream-K units, so a finisher
  never waits on a cluster that is itself waiting;
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
            assert u["slot"] == u["slot_first"] == 0
            continue
        assert sk > 0 and t >= T - sk, (t, parts)
        if sk >= G:
            assert len(parts) == 2, (t, parts)
        parts = sorted(parts, key=lambda p: p[2]["k_block_begin"])
        c0 = parts[0][0]
        for n, (c, i, u) in enumerate(parts):
            assert c == c0 + n, "a tile's parts sit in consecutive clusters"
            if n:
                assert u["k_block_begin"] == parts[n - 1][2]["k_block_end"]
            if n + 1 < len(parts):
                assert u["role"] == 1 and u["slot"] == u["slot_first"] == c, u
                assert i == 0, "a contributor publishes before its cluster does anything else"
            else:
                assert u["role"] == 2 and u["slot"] == c - 1 and u["slot_first"] == c0, u
                n_sk = sum(1 for v in sched[c] if v["tile"] >= T - sk)
                assert i == n_sk - 1, "a finisher is its cluster's last stream-K unit"

    # balance
    dp = [sum(1 for u in lst if u["tile"] < T - sk) for lst in sched.values()]
    assert max(dp) - min(dp) <= 1
    if sk:
        kbs = [sum(u["k_block_end"] - u["k_block_begin"] for u in lst if u["tile"] >= T - sk)
               for lst in sched.values()]
        assert max(kbs) - min(kbs) <= 1 and sum(kbs) == sk * nk
        if sk >= G:
            assert min(kbs) >= nk, "every stream-K range is at least one tile long"
        else:
            assert sk == T and min(kbs) >= 1, "fewer tiles than clusters: every tile split, no empty range"

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
    desc, info = plan(2048, 5120, 4096, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, tile_n=512)
    assert info.stream_k_tiles == info.num_tiles == 80
    sched = check_schedule(desc, info)
    assert all(u["tile"] >= 0 for lst in sched.values() for u in lst)


@pytest.mark.parametrize("M,N,K,kw,tiles,grid,most_parts", [
    (128, 8192, 8192, {}, 64, 128, 2),        # 64 tiles 128 wide: 2 ranges of 64 K atoms each
    (512, 512, 8192, {}, 8, 64, 4),           # long K: 8 pair tiles 128 wide, 4 ranges each
    (128, 8192, 8192, {"tile_n": 256}, 32, 128, 4),
    (512, 512, 8192, {"tile_n": 256}, 4, 32, 4),
    (512, 512, 8192, {"flags": dg.GEMM_FLAG_CTA_GROUP_1, "tile_n": 256}, 8, 32, 4),
    (64, 64, 65536, {}, 1, 8, 8),             # one tile: 8 ranges (the cap)
    (256, 256, 16384, {"tile_n": 256}, 1, 16, 8),
    (1024, 2048, 8192, {"flags": dg.GEMM_FLAG_CTA_GROUP_2, "tile_n": 512}, 16, 128, 4),   # 16 pair tiles
    # a cap below tiles x splits: ranges straddle tiles, middle contributors
    (128, 2048, 4096, {"max_ctas": 13, "tile_n": 256}, 8, 13, 3),
    (200, 1000, 4160, {"max_ctas": 11, "tile_n": 256}, 8, 11, 3),
])
def test_few_tiles_split_along_k(M, N, K, kw, tiles, grid, most_parts):
    """Fewer tiles than clusters: the grid grows past the tile count and every
    tile is split along K, several clusters per tile, one finisher each."""
    desc, info = plan(M, N, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, **kw)
    assert (info.num_tiles, info.grid, info.stream_k_tiles) == (tiles, grid, tiles)
    sched = check_schedule(desc, info)
    parts = {}
    for lst in sched.values():
        for u in lst:
            parts[u["tile"]] = parts.get(u["tile"], 0) + 1
    assert max(parts.values()) == most_parts
    assert all(lst for lst in sched.values()), "no cluster idles"
    if "max_ctas" not in kw:
        assert len(set(parts.values())) == 1, "equal ranges per tile"


@pytest.mark.parametrize("M,N,K,cg,tile_n", [
    (128, 8192, 8192, 1, 128), (256, 4096, 4096, 1, 128), (1536, 1536, 6144, 2, 128), (512, 512, 8192, 2, 128),
    (3000, 1000, 4000, 1, 256), (2048, 2048, 8192, 2, 256), (2048, 2048, 2048, 1, 256), (8192, 8192, 8192, 2, 512),
])
def test_default_tile_width(M, N, K, cg, tile_n):
    """256-wide tiles for fewer than half of the clusters narrow to 128."""
    desc, info = plan(M, N, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    assert (info.cta_group, info.tile_n) == (cg, tile_n)


@pytest.mark.parametrize("M,N,K", [(8192, 1024, 8192), (1024, 8192, 8192), (2048, 2048, 8192)])
def test_near_full_wave_not_split(M, N, K):
    """Tiles for more than half of the clusters: an uneven spread (about 1.2
    clusters per tile) measured slower than none, so the grid stays one
    cluster per tile."""
    desc, info = plan(M, N, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    assert info.stream_k_tiles == 0 and info.grid == info.num_tiles * info.cta_group


def test_residency_cap_leaves_uneven_ranges():
    """A grid smaller than tiles x splits (as a residency cap can leave it):
    the schedule still covers every K block once, with ranges across tiles."""
    desc, info = plan(512, 512, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    for G in (9, 13, 31):
        capped = dg.GemmPlanInfo.from_buffer_copy(info)
        capped.grid = G * info.cta_group
        check_schedule(desc, capped)


def test_few_tiles_short_k_and_opt_out_stay_data_parallel():
    # 16 K atoms per tile: too short to split
    desc, info = plan(128, 8192, 1024, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    assert (info.tile_n, info.num_tiles, info.grid, info.stream_k_tiles) == (128, 64, 64, 0)
    check_schedule(desc, info)
    desc, info = plan(128, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, flags=dg.GEMM_FLAG_NO_STREAM_K)
    assert (info.num_tiles, info.grid, info.stream_k_tiles) == (64, 64, 0)
    desc, info = plan(512, 512, 8192, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F16, flags=dg.GEMM_FLAG_ACCUM_F16)
    assert info.stream_k_tiles == 0 and info.grid == info.num_tiles * info.cta_group


@pytest.mark.parametrize("K,tile_n,sk", [(1024, 256, 0), (2048, 256, 0), (3072, 512, 0), (4096, 512, 0)])
def test_short_k_tile_width_and_stream_k(K, tile_n, sk):
    """Short K: 256-wide pair tiles (two accumulators) rather than 512-wide, and
    no stream-K region until a tile holds 48 K atoms."""
    desc, info = plan(8192, 8192, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    assert (info.cta_group, info.tile_n, info.stream_k_tiles) == (2, tile_n, sk)
    desc, info = plan(8192, 8192, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, tile_n=256)
    assert info.stream_k_tiles == (0 if K < 3072 else 76 + 1024 % 76)
    check_schedule(desc, info)


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


def test_random_few_tile_shapes():
    """Seeded skinny and long-K shapes, so that most plans split tiles over
    several clusters: the split count stays within 2..8, each range keeps at
    least 32 K atoms (16-bit: 64-element atoms), the grid never exceeds the
    SMs, and the whole schedule passes the invariants above."""
    rng = random.Random(11)
    split = 0
    for _ in range(60):
        M = rng.choice([1, 64, 100, 128, 256, 384, 512, 1024])
        N = rng.choice([64, 128, 200, 512, 1000, 2048, 4096, 8192])
        K = rng.choice([2048, 4096, 6000, 8192, 16384, 65536])
        kw = dict(dtype_a=rng.choice([dg.GEMM_BF16, dg.GEMM_F16]), dtype_d=rng.choice([dg.GEMM_F32, dg.GEMM_BF16]),
                  flags=dg.GEMM_FLAG_NO_SINGLE_CTA)
        desc = dg.make_desc(M, N, K, **kw)
        s, info = dg.gemm_plan_query(desc, GB300)
        assert s == dg.GEMM_OK, (M, N, K)
        G = info.grid // info.cta_group
        assert info.grid <= GB300.sm_count and info.grid % info.cta_group == 0
        if 0 < info.stream_k_tiles == info.num_tiles < G:
            split += 1
            s_per_tile = G // info.num_tiles
            assert G == s_per_tile * info.num_tiles and 2 <= s_per_tile <= 8, (M, N, K, info.as_dict())
            atoms = -(-K // 64)
            assert atoms // s_per_tile >= 32, (M, N, K, s_per_tile)
        check_schedule(desc, info)
    assert split >= 20, split


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
    bad_sk.stream_k_tiles = 5                      # fewer than the 76 clusters, and not every tile
    assert dg.gemm_plan_work_unit(desc, bad_sk, 0, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    # every tile split, but fewer K blocks than clusters: some range would be empty
    desc1, info1 = plan(64, 64, 65536, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    few = dg.make_desc(64, 64, 64 * 7, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    assert dg.gemm_plan_work_unit(few, info1, 0, 0)[0] == dg.GEMM_ERR_INVALID_ARG
    desc, info = plan(128, 64, 64, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32)
    assert info.kernel == dg.GEMM_KERNEL_SINGLE_CTA
    assert dg.gemm_plan_work_unit(desc, info, 0, 0)[0] == dg.GEMM_ERR_UNSUPPORTED
