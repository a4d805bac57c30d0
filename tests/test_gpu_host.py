"""GPU parity of gemm_run_host: operands in pinned host memory.

Large problems are split into row panels (or batch-entry panels): B first,
then each panel's rows of A are copied in on one stream while earlier panels
multiply on the caller's stream and copy their rows of D out on another.
Every case checks the whole of D against the oracle, with device buffers
filled with NaN first so that a row no panel wrote cannot pass.
"""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_16BIT, TOL_FP8, compare, dump_on_failure

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32, "e4m3": dg.GEMM_E4M3}


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def run_host(prob, out, mn_a=False, **kw):
    wl = prob.wl
    A = prob.A.transpose(-1, -2).contiguous() if mn_a else prob.A
    hA, hB = A.pin_memory(), prob.B.pin_memory()
    shape = (wl.batch, wl.M, wl.N) if wl.batch > 1 else (wl.M, wl.N)
    hD = torch.full(shape, float("nan"), dtype=TDT[out]).pin_memory()
    dA, dB = torch.empty_like(A, device="cuda"), torch.empty_like(prob.B, device="cuda")
    dD = torch.full(shape, float("nan"), dtype=TDT[out], device="cuda")
    scaled = prob.scale_a is not None
    hsa = prob.scale_a.pin_memory() if scaled else None
    hsb = prob.scale_b.pin_memory() if scaled else None
    dsa = torch.empty_like(prob.scale_a, device="cuda") if scaled else None
    dsb = torch.empty_like(prob.scale_b, device="cuda") if scaled else None
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=CODE[wl.dtype_in], dtype_d=CODE[out],
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128 if scaled else 0,
                        major_a=dg.GEMM_MN_MAJOR if mn_a else dg.GEMM_K_MAJOR, **kw)
    with dg.Plan(desc) as plan:
        for _ in range(2):   # the second call reuses the plan's panels and copy streams
            plan.run_host(hA, hB, hD, dA, dB, dD, hsa, hsb, dsa, dsb)
            s, rec = plan.sync_status()
            assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
    kw_o = dict(scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy()) if scaled else {}
    dref, sabs = oracle.gemm(A, prob.B, M=wl.M, N=wl.N, K=wl.K, batch=wl.batch, dtype_a=wl.dtype_in,
                             dtype_b=wl.dtype_in, major_a="mn" if mn_a else "k", **kw_o)
    return hD.double().numpy().reshape(dref.shape), dref, sabs


@pytest.mark.parametrize("mn_a", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_host_row_panels_bit_exact(mn_a, out):
    """M = 4096 gives four row panels of 1024 (2-D copies; for MN-major A the
    panel is a column range of the stored [K][M] array)."""
    prob = inputs.make("square8192_bf16", M=4096, N=1024, K=320, dist="ints", seed=91)
    got, dref, s = run_host(prob, out, mn_a=mn_a)
    r = compare(got, dref, s, out, TOL_16BIT, exact=True)
    if not r["ok"]:
        dump_on_failure("host_rows_%s_%d" % (out, mn_a), got=got, dref=dref, sabs=s)
    assert r["ok"], r


def test_host_ragged_row_panels_random():
    """M = 3000: panel edges on 256-row bands, a ragged last panel."""
    prob = inputs.make("square8192_bf16", M=3000, N=776, K=1000, seed=92)
    got, dref, s = run_host(prob, "f32")
    assert compare(got, dref, s, "f32", TOL_16BIT)["ok"]


def test_host_batch_panels_bit_exact():
    """256 batch entries of 128x128x192 -> four panels of 64 entries."""
    prob = inputs.make("batched256_f16", M=128, N=128, K=192, batch=256, dist="ints", seed=93)
    got, dref, s = run_host(prob, "f16")
    assert compare(got, dref, s, "f16", TOL_16BIT, exact=True)["ok"]


def test_host_block_scaled_panels_bit_exact():
    """Block-scaled fp8: each panel also copies its rows of A's scales."""
    prob = inputs.make("fp8_block8192", M=2048, N=768, K=512, dist="ints", seed=94)
    got, dref, s = run_host(prob, "bf16")
    r = compare(got, dref, s, "bf16", TOL_FP8, exact=True)
    assert r["ok"], r


def test_host_small_single_piece():
    """Below two panels' worth of rows the call copies, multiplies and copies back in one piece."""
    prob = inputs.make("square8192_bf16", M=512, N=512, K=256, dist="ints", seed=95)
    got, dref, s = run_host(prob, "f32")
    assert compare(got, dref, s, "f32", TOL_16BIT, exact=True)["ok"]


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_host_first_block_quarters_bit_exact(out):
    """M >= 4096 and N >= 2048: a first block of 40 % of the rows against B's
    four column quarters, then the remaining rows in panels."""
    prob = inputs.make("square8192_bf16", M=4352, N=2304, K=256, dist="ints", seed=96)
    got, dref, s = run_host(prob, out)
    r = compare(got, dref, s, out, TOL_16BIT, exact=True)
    if not r["ok"]:
        dump_on_failure("host_quarters_%s" % out, got=got, dref=dref, sabs=s)
    assert r["ok"], r


def test_host_first_block_quarters_block_scaled():
    """The same schedule with fp8 operands: each quarter of B brings its rows of B's scales."""
    prob = inputs.make("fp8_block8192", M=4096, N=2048, K=384, dist="ints", seed=97)
    got, dref, s = run_host(prob, "bf16")
    assert compare(got, dref, s, "bf16", TOL_FP8, exact=True)["ok"]
