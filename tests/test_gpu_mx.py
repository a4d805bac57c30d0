"""GPU parity of the hardware block-scaled path (MXFP8, MXFP4, NVFP4) against
the CPU oracle.

"Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling": the
tensor core multiplies each block of a row of A and of B by its own scale
inside tcgen05.mma (.kind::mxf8f6f4, .kind::mxf4, .kind::mxf4nvf4), the
scales read from tensor memory after a tcgen05.cp from shared memory ("TMEM
-- the accumulator's new home", section "Block-scaled MMA").  Both sides read
the same element and scale bytes; the oracle sums the exact products in fp64,
the GPU in fp32.  Integer-valued elements with power-of-two scales keep every
sum exact, so those runs must match bit for bit; quantised N(0,1) inputs must
stay within 2e-3 of sum |a||b| (the products themselves are exact on both
sides, so only fp32 accumulation separates them: the 16-bit inputs' bound).
"""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_16BIT, compare, dump_on_failure

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32}
IN = {"e4m3": dg.GEMM_E4M3, "e5m2": dg.GEMM_E5M2, "e2m1": dg.GEMM_E2M1}
MODE = {"mx": dg.GEMM_SCALE_MX_E8M0_32, "nv": dg.GEMM_SCALE_NV_E4M3_16}


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def run_mx(prob, out, **kw):
    wl = prob.wl
    mode = wl.extra["scale_mode"]
    D = torch.full((wl.M, wl.N), float("nan"), dtype=TDT[out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=IN[wl.dtype_in], dtype_b=IN[wl.extra["dtype_b"]],
                        dtype_d=CODE[out], scale_mode=MODE[mode], **kw)
    ts = torch.tensor(prob.tensor_scales, dtype=torch.float32, device="cuda") if mode == "nv" else None
    with dg.Plan(desc) as plan:
        plan.run_mx(prob.A.cuda(), prob.B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda(), ts)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role, rec.stage, rec.tile)
        info = plan.info.as_dict()
    assert info["kernel"] == dg.GEMM_KERNEL_MX
    return D, info


def oracle_mx(prob, rows=None):
    wl = prob.wl
    return oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in,
                            dtype_b=wl.extra["dtype_b"], scale_a=prob.scale_a, scale_b=prob.scale_b,
                            scale_mode=wl.extra["scale_mode"], tensor_scales=prob.tensor_scales, rows=rows)


def check(prob, out, exact, **kw):
    D, info = run_mx(prob, out, **kw)
    dref, s = oracle_mx(prob)
    got = D.double().cpu().numpy()
    r = compare(got, dref[0], s[0], out, TOL_16BIT, exact=exact)
    if not r["ok"]:
        dump_on_failure("mx_%s_%s_cg%d" % (prob.wl.name, out, info["cta_group"]), got=got, dref=dref[0], sabs=s[0])
    assert r["ok"], (r, info)
    return info


# ragged M, N and K in every case: a partial 128-row block, a partial tile
# column, a K tail inside the last 128-byte atom (partial scale blocks)
SMALL = {"mxfp8_8192": dict(M=300, N=520, K=400), "mxfp4_8192": dict(M=300, N=520, K=416),
         "nvfp4_8192": dict(M=300, N=520, K=448)}


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_block_scaled_integers_bit_exact(name, cg_flag):
    prob = inputs.make(name, dist="ints", seed=51, **SMALL[name])
    info = check(prob, "f32", exact=True, flags=cg_flag)
    assert info["cta_group"] == (1 if cg_flag == dg.GEMM_FLAG_CTA_GROUP_1 else 2)


@pytest.mark.parametrize("out", ["bf16", "f16"])
@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_block_scaled_integers_16bit_out(name, out):
    prob = inputs.make(name, dist="ints", seed=52, **SMALL[name])
    check(prob, out, exact=True)


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_block_scaled_quantised_normal(name, cg_flag):
    prob = inputs.make(name, seed=53, **SMALL[name])
    check(prob, "bf16", exact=False, flags=cg_flag)


def test_mxfp8_e5m2_pairing_bit_exact():
    prob = inputs.make("mxfp8_8192", dist="ints", seed=54, dtype_b="e5m2", **SMALL["mxfp8_8192"])
    check(prob, "f32", exact=True)


def test_block_scaled_many_tiles_few_ctas():
    """More tiles than clusters: the single accumulator and the scale slots cycle."""
    prob = inputs.make("mxfp8_8192", dist="ints", seed=55, M=1024, N=1280, K=640)
    check(prob, "f32", exact=True, max_ctas=6, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    prob = inputs.make("nvfp4_8192", dist="ints", seed=56, M=1024, N=1280, K=768)
    check(prob, "f32", exact=True, max_ctas=5, flags=dg.GEMM_FLAG_CTA_GROUP_1)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_full_size_integers_bit_exact(name):
    """The benchmark's plan at 8192^3 on seeded rows plus both edge rows of every 128-row block."""
    prob = inputs.make(name, dist="ints")
    D, info = run_mx(prob, "bf16")
    assert (info["cta_group"], info["tile_n"], info["grid"]) == (2, 256, 152), info
    rows = inputs.sample_rows(prob.wl.M, 1, n_random=48, seed=5, tile_m=128)
    dref, s = oracle_mx(prob, rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, "bf16", TOL_16BIT, exact=True)
    assert r["ok"], (name, r, info)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_full_size_quantised_normal_sampled(name):
    prob = inputs.make(name)
    D, info = run_mx(prob, "bf16")
    rows = inputs.sample_rows(prob.wl.M, 1, n_random=32, seed=6, tile_m=256)
    dref, s = oracle_mx(prob, rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, "bf16", TOL_16BIT)
    assert r["ok"], (name, r, info)


def test_wrong_entry_points_are_refused():
    prob = inputs.make("mxfp8_8192", dist="ints", seed=57, M=256, N=256, K=256)
    desc = dg.make_desc(256, 256, 256, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_F32,
                        scale_mode=dg.GEMM_SCALE_MX_E8M0_32)
    A, B, sa, sb = prob.A.cuda(), prob.B.cuda(), prob.scale_a.cuda(), prob.scale_b.cuda()
    D = torch.zeros(256, 256, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    with dg.Plan(desc) as plan:
        assert dg.gemm_run(plan.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                           stream) == dg.GEMM_ERR_INVALID_ARG
        ts = torch.ones(2, device="cuda")
        assert dg.gemm_run_mx(plan.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), sa.data_ptr(), sb.data_ptr(),
                              ts.data_ptr(), stream) == dg.GEMM_ERR_INVALID_ARG   # tensor scales are NVFP4's
        assert dg.gemm_run_mx(plan.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), sa.data_ptr() + 8,
                              sb.data_ptr(), None, stream) == dg.GEMM_ERR_ALIGNMENT
    assert dg.gemm_run_noalloc(desc, A.data_ptr(), B.data_ptr(), D.data_ptr(), None, None, stream,
                               None) == dg.GEMM_ERR_UNSUPPORTED


def _batched(name, batch, seed0, **shape):
    """A batch of independent problems with the workload's recipe: operands
    stacked, tiled scales one batch entry after the other."""
    probs = [inputs.make(name, dist="ints", seed=seed0 + i, **shape) for i in range(batch)]
    return (probs, torch.stack([p.A for p in probs]), torch.stack([p.B for p in probs]),
            torch.cat([p.scale_a for p in probs]), torch.cat([p.scale_b for p in probs]))


@pytest.mark.parametrize("name,cg_flag", [("mxfp8_8192", dg.GEMM_FLAG_CTA_GROUP_2),
                                          ("mxfp4_8192", dg.GEMM_FLAG_CTA_GROUP_1),
                                          ("nvfp4_8192", dg.GEMM_FLAG_CTA_GROUP_2)])
def test_batched_block_scaled_bit_exact(name, cg_flag):
    """Three batch entries: 3-D operand maps and the scale maps' batch dimension."""
    shape = dict(M=300, N=260, K=256)
    probs, A, B, SA, SB = _batched(name, 3, 61, **shape)
    wl = probs[0].wl
    mode = wl.extra["scale_mode"]
    D = torch.full((3, wl.M, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=3, dtype_a=IN[wl.dtype_in], dtype_d=dg.GEMM_F32,
                        scale_mode=MODE[mode], flags=cg_flag)
    ts = torch.tensor(probs[0].tensor_scales, dtype=torch.float32, device="cuda") if mode == "nv" else None
    with dg.Plan(desc) as plan:
        plan.run_mx(A.cuda(), B.cuda(), D, SA.cuda(), SB.cuda(), ts)
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, _ = oracle.gemm(A, B, M=wl.M, N=wl.N, K=wl.K, batch=3, dtype_a=wl.dtype_in, dtype_b=wl.dtype_in,
                          scale_a=SA, scale_b=SB, scale_mode=mode, tensor_scales=probs[0].tensor_scales)
    assert np.array_equal(D.double().cpu().numpy(), dref)


def test_empty_and_k_zero():
    """K = 0 writes zeros (no scale pointers are read); M = 0 is a no-op."""
    for M, N, K in [(300, 64, 0), (0, 64, 64)]:
        D = torch.full((max(M, 1), N), 7.0, device="cuda")
        desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_F32, scale_mode=dg.GEMM_SCALE_MX_E8M0_32,
                            lda=64, ldb=64, ldd=N)
        dummy = torch.zeros(1024, dtype=torch.uint8, device="cuda")
        with dg.Plan(desc) as plan:
            plan.run_mx(dummy, dummy, D, dummy, dummy)
            torch.cuda.synchronize()
        assert (D == 0).all() if (K == 0 and M) else (D == 7.0).all()


def _random_cases(n=12, seed=2027):
    import random
    rng = random.Random(seed)
    cases = []
    for i in range(n):
        name = rng.choice(["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
        kq = 16 if name == "mxfp8_8192" else 32            # rows of K must be 16-byte multiples
        cases.append(dict(name=name, M=rng.randint(1, 700), N=8 * rng.randint(1, 90), K=kq * rng.randint(1, 40),
                          cg=rng.choice([dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2]),
                          out=rng.choice(["f32", "bf16", "f16"]), ctas=rng.choice([0, 4, 10]), seed=100 + i))
    return cases


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "%s-%dx%dx%d" % (c["name"], c["M"], c["N"], c["K"]))
def test_random_shapes_bit_exact(case):
    """Seeded random shapes: any M, N a multiple of 8, K a multiple of 16 (8-bit) or
    32 (4-bit), either CTA group, every output type, capped grids."""
    prob = inputs.make(case["name"], dist="ints", seed=case["seed"], M=case["M"], N=case["N"], K=case["K"])
    check(prob, case["out"], exact=True, flags=case["cg"], max_ctas=case["ctas"])


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("mn_a,mn_b", [(True, False), (False, True), (True, True)])
def test_mxfp8_mn_major_bit_exact(cg_flag, mn_a, mn_b):
    """MXFP8 operands stored [k][m] (or [k][n]) reach the block-scaled MMA through
    the descriptors' MN-major layout; the scales stay per row and K block."""
    prob = inputs.make("mxfp8_8192", M=384, N=640, K=400, dist="ints", seed=59)
    wl = prob.wl
    A = prob.A.transpose(0, 1).contiguous() if mn_a else prob.A
    B = prob.B.transpose(0, 1).contiguous() if mn_b else prob.B
    D = torch.full((wl.M, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_F32,
                        scale_mode=dg.GEMM_SCALE_MX_E8M0_32, flags=cg_flag,
                        major_a=dg.GEMM_MN_MAJOR if mn_a else dg.GEMM_K_MAJOR,
                        major_b=dg.GEMM_MN_MAJOR if mn_b else dg.GEMM_K_MAJOR)
    with dg.Plan(desc) as plan:
        plan.run_mx(A.cuda(), B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda())
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, _ = oracle.gemm(A, B, M=wl.M, N=wl.N, K=wl.K, dtype_a="e4m3", dtype_b="e4m3",
                          major_a="mn" if mn_a else "k", major_b="mn" if mn_b else "k",
                          scale_a=prob.scale_a, scale_b=prob.scale_b, scale_mode="mx")
    assert np.array_equal(D.double().cpu().numpy(), dref[0])

