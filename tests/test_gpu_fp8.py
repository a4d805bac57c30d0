"""GPU parity of the block-scaled e4m3 path against the CPU oracle.

The oracle dequantises every element (q * its block's scale) and sums the
products in fp64; the GPU multiplies e4m3 codes on the tensor core per
128-deep block and applies sA[m][kb] * sB[n/128][kb] to each block's fp32
partial.  Integer codes with scales in {1/2, 1, 2} keep every intermediate
exact, so those runs must match bit for bit; block-quantised N(0,1) inputs
must stay within 2e-2 of sum |a||b| ("Hopper and Blackwell GEMM", FP8 and
FP4 with block scaling).
"""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_FP8, compare, dump_on_failure

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32}


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def run_fp8(prob, out, **kw):
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    sa, sb = prob.scale_a.cuda(), prob.scale_b.cuda()
    D = torch.full((wl.M, wl.N), float("nan"), dtype=TDT[out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_E4M3, dtype_d=CODE[out],
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128, **kw)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D, sa, sb)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role, rec.stage, rec.tile)
        info = plan.info.as_dict()
    assert info["kernel"] == dg.GEMM_KERNEL_FP8_BLOCK
    return D, info


def oracle_fp8(prob, rows=None):
    wl = prob.wl
    return oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="e4m3", dtype_b="e4m3",
                            scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy(), rows=rows)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("out", ["bf16", "f32", "f16"])
def test_fp8_integers_bit_exact(cg_flag, out, tile_n):
    """Both tile widths (2 or 4 TMEM partial buffers, 128 or 64 columns per
    promotion warp) on both CTA groups."""
    prob = inputs.make("fp8_block8192", M=520, N=600, K=400, dist="ints", seed=31)
    D, info = run_fp8(prob, out, flags=cg_flag, tile_n=tile_n)
    assert info["tile_n"] == tile_n and info["tmem_stages"] == 512 // tile_n
    dref, s = oracle_fp8(prob)
    got = D.double().cpu().numpy()
    r = compare(got, dref[0], s[0], out, TOL_FP8, exact=True)
    if not r["ok"]:
        dump_on_failure("fp8_%s_cg%d" % (out, info["cta_group"]), got=got, dref=dref[0], sabs=s[0])
    assert r["ok"], (r, info)


@pytest.mark.parametrize("cg_flag,tile_n", [(dg.GEMM_FLAG_CTA_GROUP_1, 256), (dg.GEMM_FLAG_CTA_GROUP_2, 128),
                                            (dg.GEMM_FLAG_CTA_GROUP_2, 256), (dg.GEMM_FLAG_CTA_GROUP_1, 128)])
def test_fp8_quantised_normal(cg_flag, tile_n):
    prob = inputs.make("fp8_block8192", M=300, N=520, K=512, seed=32)
    D, info = run_fp8(prob, "bf16", flags=cg_flag, tile_n=tile_n)
    dref, s = oracle_fp8(prob)
    r = compare(D.double().cpu().numpy(), dref[0], s[0], "bf16", TOL_FP8)
    assert r["ok"], (r, info)


def test_fp8_many_tiles_few_ctas():
    prob = inputs.make("fp8_block8192", M=1024, N=1024, K=256, dist="ints", seed=33)
    D, info = run_fp8(prob, "f32", max_ctas=4, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    dref, s = oracle_fp8(prob)
    assert compare(D.double().cpu().numpy(), dref[0], s[0], "f32", TOL_FP8, exact=True)["ok"]


@pytest.mark.slow
def test_fp8_full_size_sampled():
    prob = inputs.make("fp8_block8192")
    D, info = run_fp8(prob, "bf16")
    rows = inputs.sample_rows(prob.wl.M, 1, n_random=48, seed=2, tile_m=info["tile_m"])
    dref, s = oracle_fp8(prob, rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, "bf16", TOL_FP8)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("mn_a,mn_b", [(True, False), (False, True), (True, True)])
def test_fp8_mn_major_bit_exact(cg_flag, mn_a, mn_b):
    """fp8 reaches tcgen05 in either majorness (cuBLASDx "API Card: Blackwell
    Pipeline (tcgen05)", precision and arrangement notes): an MN-major operand
    is stored [k][m] (or [k][n]) and loaded as 128-element x 128-k boxes."""
    prob = inputs.make("fp8_block8192", M=512, N=640, K=400, dist="ints", seed=35)
    wl = prob.wl
    A, B = prob.A, prob.B
    if mn_a:
        A = A.transpose(-1, -2).contiguous()
    if mn_b:
        B = B.transpose(-1, -2).contiguous()
    D = torch.full((wl.M, wl.N), float("nan"), dtype=torch.float32, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_F32,
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128, flags=cg_flag, tile_n=256,
                        major_a=dg.GEMM_MN_MAJOR if mn_a else dg.GEMM_K_MAJOR,
                        major_b=dg.GEMM_MN_MAJOR if mn_b else dg.GEMM_K_MAJOR)
    with dg.Plan(desc) as plan:
        plan.run(A.cuda(), B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda())
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
        info = plan.info.as_dict()
    assert info["kernel"] == dg.GEMM_KERNEL_FP8_BLOCK
    dref, sabs = oracle.gemm(A, B, M=wl.M, N=wl.N, K=wl.K, dtype_a="e4m3", dtype_b="e4m3",
                             major_a="mn" if mn_a else "k", major_b="mn" if mn_b else "k",
                             scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy())
    got = D.double().cpu().numpy()
    r = compare(got, dref[0], sabs[0], "f32", TOL_FP8, exact=True)
    if not r["ok"]:
        dump_on_failure("fp8_mn_%d%d_cg%d" % (mn_a, mn_b, info["cta_group"]), got=got, dref=dref[0], sabs=sabs[0])
    assert r["ok"], (r, info)


@pytest.mark.slow
def test_fp8_full_size_integers_bit_exact():
    """The benchmark's plan (SM-pair 256 x 256 tiles over the whole grid) on
    integer codes with scales in {1/2, 1, 2}: each block product, each scaled
    partial and each running sum is exact in fp32 (below 2^21 in units of
    1/4), so D must equal the oracle's single rounding bit for bit, on seeded
    rows plus the first and last row of every 128-row block."""
    prob = inputs.make("fp8_block8192", dist="ints")
    D, info = run_fp8(prob, "bf16")
    assert info["cta_group"] == 2 and info["tile_n"] == 256, info
    rows = inputs.sample_rows(prob.wl.M, 1, n_random=64, seed=4, tile_m=128)
    dref, s = oracle_fp8(prob, rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, "bf16", TOL_FP8, exact=True)
    if not r["ok"]:
        dump_on_failure("fp8_full_exact", got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)

