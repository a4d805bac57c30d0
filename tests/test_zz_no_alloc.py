"""gemm_run_noalloc: the allocation-free entry point, for callers that cannot
call cudaMalloc (their device memory is owned by a framework's caching pool, or
they cannot afford the synchronisation an allocation may imply).  Its kernels
keep their error record in a library-owned static device array instead of a
plan's cudaMalloc'd record.

Checked through the C ABI on two calls in a row (the second call finds the
record left by the first and must clear it): against the CPU oracle, within
the parity tolerance of the other tests for random inputs and bit for bit for
integer-valued inputs, and against the plan-based gemm_run, which must give the
same bytes (both run the same data-parallel tiles).  This file is collected
last on purpose; it also passes when run alone.
"""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_16BIT, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


CASES = [
    # (workload, overrides, out dtype, flags): the persistent pair kernel and the single-CTA kernel
    ("square8192_bf16", dict(M=1024, N=768, K=512, seed=21), "f32", dg.GEMM_FLAG_CTA_GROUP_2),
    ("single_cta", dict(seed=22), "f32", 0),
    ("batched256_f16", dict(batch=6, seed=23), "f16", 0),
]
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
CODE = {"f32": dg.GEMM_F32, "bf16": dg.GEMM_BF16, "f16": dg.GEMM_F16}
IN_CODE = {"bf16": dg.GEMM_BF16, "f16": dg.GEMM_F16}


@pytest.mark.parametrize("dist", ["random", "ints"])
@pytest.mark.parametrize("name,over,out,flags", CASES)
def test_noalloc_matches_oracle_on_two_calls(name, over, out, flags, dist):
    if dist == "ints":
        over = dict(over, dist="ints")
    prob = inputs.make(name, **over)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    shape = (wl.batch, wl.M, wl.N) if wl.batch > 1 else (wl.M, wl.N)
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=IN_CODE[wl.dtype_in], dtype_d=CODE[out],
                        flags=flags)
    stream = torch.cuda.current_stream().cuda_stream
    dref, sabs = oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, batch=wl.batch,
                                  dtype_a=wl.dtype_in, dtype_b=wl.dtype_in)
    # the plan-based path on the same data-parallel tiles, for a byte comparison
    D_plan = torch.empty(shape, dtype=TDT[out], device="cuda")
    with dg.Plan(dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=IN_CODE[wl.dtype_in],
                              dtype_d=CODE[out], flags=flags | dg.GEMM_FLAG_NO_STREAM_K)) as plan:
        plan.run(A, B, D_plan)
        assert plan.sync_status()[0] == dg.GEMM_OK
    for call in range(2):
        D = torch.full(shape, float("nan"), dtype=TDT[out], device="cuda")
        rec = dg.GemmDeviceError()
        s = dg.gemm_run_noalloc(desc, A.data_ptr(), B.data_ptr(), D.data_ptr(), None, None, stream, rec)
        assert s == dg.GEMM_OK, (call, dg.gemm_status_string(s))
        assert rec.code == 0
        got = D.double().cpu().numpy().reshape(sabs.shape)
        r = compare(got, dref, sabs, out, TOL_16BIT, exact=(dist == "ints"))
        assert r["ok"], (call, dist, r)
        assert torch.equal(D, D_plan), call


def test_noalloc_enqueue_only_then_sync():
    """status_out = NULL: the call returns once enqueued; stream order still holds."""
    prob = inputs.make("square8192_bf16", M=512, N=512, K=256, dist="ints", seed=24)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.empty(wl.M, wl.N, dtype=torch.float32, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    s = dg.gemm_run_noalloc(desc, A.data_ptr(), B.data_ptr(), D.data_ptr(), None, None,
                            torch.cuda.current_stream().cuda_stream, None)
    assert s == dg.GEMM_OK
    torch.cuda.synchronize()
    dref, _ = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="bf16", dtype_b="bf16")
    assert (D.double().cpu().numpy() == dref[0]).all()
