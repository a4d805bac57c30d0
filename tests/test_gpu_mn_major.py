"""GPU parity with MN-major operands in the persistent kernel.

"row_major / col_major" arrangements of A and B reach the tensor core in
either majorness for 16-bit inputs (cuBLASDx "API Card: Blackwell Pipeline
(tcgen05)", Descriptor).  An MN-major operand is stored [k][m] (or [k][n]):
the kernel loads it as 64-element x 64-k boxes and describes it to the MMA
with the MN-major 128-byte-swizzle layout.  Integer inputs: bit-exact.
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


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def run_mn(prob, out, mn_a, mn_b, **kw):
    wl = prob.wl
    A, B = prob.A, prob.B                       # logical [b][M][K], [b][N][K]
    batched = wl.batch > 1
    if mn_a:
        A = A.transpose(-1, -2).contiguous()    # stored [b][K][M]
    if mn_b:
        B = B.transpose(-1, -2).contiguous()    # stored [b][K][N]
    Ad, Bd = A.cuda(), B.cuda()
    shape = (wl.batch, wl.M, wl.N) if batched else (wl.M, wl.N)
    D = torch.full(shape, float("nan"), dtype=TDT[out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=CODE[wl.dtype_in], dtype_d=CODE[out],
                        major_a=dg.GEMM_MN_MAJOR if mn_a else dg.GEMM_K_MAJOR,
                        major_b=dg.GEMM_MN_MAJOR if mn_b else dg.GEMM_K_MAJOR, **kw)
    with dg.Plan(desc) as plan:
        plan.run(Ad, Bd, D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
        info = plan.info.as_dict()
    assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT
    dref, sabs = oracle.gemm(A, B, M=wl.M, N=wl.N, K=wl.K, batch=wl.batch, dtype_a=wl.dtype_in,
                             dtype_b=wl.dtype_in, major_a="mn" if mn_a else "k", major_b="mn" if mn_b else "k")
    got = D.double().cpu().numpy().reshape(dref.shape)
    return got, dref, sabs, info


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("mn_a,mn_b", [(True, False), (False, True), (True, True)])
def test_mn_major_integers_bit_exact(cg_flag, mn_a, mn_b):
    prob = inputs.make("square8192_bf16", M=600, N=712, K=1040, dist="ints", seed=81)
    got, dref, s, info = run_mn(prob, "f32", mn_a, mn_b, flags=cg_flag)
    r = compare(got, dref, s, "f32", TOL_16BIT, exact=True)
    if not r["ok"]:
        dump_on_failure("mn_%d%d_cg%d" % (mn_a, mn_b, info["cta_group"]), got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_mn_major_random_16bit_out_and_stream_k(out):
    prob = inputs.make("square4096_bf16", M=1024, N=1024, K=4096, seed=82)
    got, dref, s, info = run_mn(prob, out, True, True, flags=dg.GEMM_FLAG_CTA_GROUP_2, max_ctas=10)
    assert info["stream_k_tiles"] > 0
    assert compare(got, dref, s, out, TOL_16BIT)["ok"]


def test_mn_major_batched_f16():
    prob = inputs.make("batched256_f16", M=256, N=192, K=136, batch=5, dist="ints", seed=83)
    got, dref, s, info = run_mn(prob, "f16", True, True, flags=dg.GEMM_FLAG_NO_SINGLE_CTA)
    assert compare(got, dref, s, "f16", TOL_16BIT, exact=True)["ok"]


def test_mn_major_matches_k_major_bitwise():
    """Same logical product, same plan shape: MN-major and K-major operands give identical D."""
    prob = inputs.make("square4096_bf16", M=768, N=768, K=1024, seed=84)
    g1, _, _, _ = run_mn(prob, "f32", False, False, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    g2, _, _, _ = run_mn(prob, "f32", True, True, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    assert np.array_equal(g1, g2)
