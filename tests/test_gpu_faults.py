"""Device-side failure detection without a GPU fault.

A test-only plan flag makes the TMA producer of CTA 0 skip its first copy, so
the full barrier of that ring slot never completes.  Every wait in the kernel
is bounded (here by a 20 ms limit): the consumer's wait runs out, the kernel
records GEMM_ERR_TIMEOUT with the waiting role, every role leaves its loop and
drains what it issued, tensor memory is freed and the kernel returns.  The
host reads the record with gemm_sync_status; the context stays usable, which
the exact product that follows shows.  Nothing traps, faults or spins forever.
"""
import time

import numpy as np
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_FP8, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


@pytest.mark.parametrize("cg_flag,ctas", [(dg.GEMM_FLAG_CTA_GROUP_1, 0), (dg.GEMM_FLAG_CTA_GROUP_2, 0),
                                          (dg.GEMM_FLAG_CTA_GROUP_2, 6)])
def test_dropped_copy_times_out_and_context_survives(cg_flag, ctas):
    prob = inputs.make("square8192_bf16", M=1024, N=1024, K=1024, dist="ints", seed=41)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.zeros(wl.M, wl.N, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                        flags=cg_flag | dg.GEMM_FLAG_TEST_DROP_LOAD, wait_timeout_ns=20_000_000, max_ctas=ctas)
    with dg.Plan(desc) as plan:
        t0 = time.time()
        plan.run(A, B, D)
        status, rec = plan.sync_status()
        elapsed = time.time() - t0
        assert status == dg.GEMM_ERR_TIMEOUT
        assert rec.code == dg.GEMM_ERR_TIMEOUT and rec.role in (1, 2, 3)
        assert elapsed < 5.0
        # the record is cleared once read
        assert plan.sync_status()[0] == dg.GEMM_OK

    # the same context computes an exact product afterwards
    desc_ok = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, flags=cg_flag)
    with dg.Plan(desc_ok) as plan:
        plan.run(A, B, D)
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, _ = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="bf16", dtype_b="bf16")
    assert np.array_equal(D.double().cpu().numpy(), dref[0])


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
def test_fp8_dropped_copy_times_out_and_context_survives(cg_flag):
    """Same for the block-scaled kernel, whose full barriers also count the
    promotion warps' partial releases: the abort path must still drain."""
    prob = inputs.make("fp8_block8192", M=1024, N=1024, K=1024, seed=43)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    SA, SB = prob.scale_a.cuda(), prob.scale_b.cuda()
    D = torch.zeros(wl.M, wl.N, dtype=torch.bfloat16, device="cuda")
    common = dict(dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16, scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    desc = dg.make_desc(wl.M, wl.N, wl.K, flags=cg_flag | dg.GEMM_FLAG_TEST_DROP_LOAD,
                        wait_timeout_ns=20_000_000, **common)
    with dg.Plan(desc) as plan:
        t0 = time.time()
        plan.run(A, B, D, SA, SB)
        status, rec = plan.sync_status()
        elapsed = time.time() - t0
        assert status == dg.GEMM_ERR_TIMEOUT
        assert rec.code == dg.GEMM_ERR_TIMEOUT and rec.role in (1, 2, 3)
        assert elapsed < 5.0
        assert plan.sync_status()[0] == dg.GEMM_OK

    desc_ok = dg.make_desc(wl.M, wl.N, wl.K, flags=cg_flag, **common)
    with dg.Plan(desc_ok) as plan:
        plan.run(A, B, D, SA, SB)
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, sabs = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="e4m3", dtype_b="e4m3",
                             scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy())
    assert compare(D.double().cpu().numpy(), dref[0], sabs[0], "bf16", TOL_FP8)["ok"]


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
def test_mx_dropped_copy_times_out_and_context_survives(cg_flag):
    """Same for the hardware block-scaled kernel, whose full barriers also
    count the scale producer's bytes."""
    prob = inputs.make("mxfp8_8192", M=1024, N=1024, K=1024, dist="ints", seed=44)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    SA, SB = prob.scale_a.cuda(), prob.scale_b.cuda()
    D = torch.zeros(wl.M, wl.N, device="cuda")
    common = dict(dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_F32, scale_mode=dg.GEMM_SCALE_MX_E8M0_32)
    desc = dg.make_desc(wl.M, wl.N, wl.K, flags=cg_flag | dg.GEMM_FLAG_TEST_DROP_LOAD,
                        wait_timeout_ns=20_000_000, **common)
    with dg.Plan(desc) as plan:
        t0 = time.time()
        plan.run_mx(A, B, D, SA, SB)
        status, rec = plan.sync_status()
        elapsed = time.time() - t0
        assert status == dg.GEMM_ERR_TIMEOUT
        assert rec.code == dg.GEMM_ERR_TIMEOUT and rec.role in (1, 2, 3)
        assert elapsed < 5.0
        assert plan.sync_status()[0] == dg.GEMM_OK

    desc_ok = dg.make_desc(wl.M, wl.N, wl.K, flags=cg_flag, **common)
    with dg.Plan(desc_ok) as plan:
        plan.run_mx(A, B, D, SA, SB)
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, _ = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="e4m3", dtype_b="e4m3",
                          scale_a=prob.scale_a, scale_b=prob.scale_b, scale_mode="mx")
    assert np.array_equal(D.double().cpu().numpy(), dref[0])
