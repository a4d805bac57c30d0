"""GPU: the caller's padding around the operands and the output.

Leading dimensions may exceed the logical sizes.  The product must read only
the first K elements of each K-major operand row and write only the first N
elements of each row of D.  Two facts about the tensor copies make this worth
testing: a TMA load zero-fills exactly at the tensor's edge, element by element,
but a TMA store writes whole 16-byte granules of a row.  So a D row whose
N x element bytes is not a multiple of 16 ends inside a granule whose tail is
the caller's padding; every epilogue writes that edge chunk with plain stores.

Integer-valued inputs keep every sum exact; the oracle reads the same padded
buffers through the same leading dimensions.  Padding is NaN on both sides:
a NaN that reached D, or a padding element that the GPU overwrote, fails.
"""
import numpy as np
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_16BIT, TOL_FP8, compare

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32}
NAN_E4M3 = 0x7F


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def pad_rows(x, ld, fill_bytes=None):
    """x [..., rows, cols] copied into rows of `ld` elements; the padding is NaN
    (floats) or the given byte value (8-bit codes)."""
    shape = x.shape[:-1] + (ld,)
    if x.element_size() == 1:
        out = torch.full(shape, fill_bytes, dtype=torch.uint8).view(x.dtype)
    else:
        out = torch.full(shape, float("nan"), dtype=x.dtype)
    out[..., : x.shape[-1]] = x
    return out.contiguous()


def new_d(batch, M, ldd, out):
    rows = batch * M
    return torch.full((rows, ldd), float("nan"), dtype=TDT[out], device="cuda")


def check_d(D, dref, sabs, batch, M, N, ldd, out, tol):
    got_all = D.double().cpu().numpy().reshape(batch, M, ldd)
    pad = got_all[:, :, N:]
    assert np.isnan(pad).all(), "D padding written: %d elements" % int((~np.isnan(pad)).sum())
    got = got_all[:, :, :N]
    r = compare(got, dref.reshape(batch, M, N), sabs.reshape(batch, M, N), out, tol, exact=True)
    assert r["ok"], r


# (M, N, K, ldd, out, batch, desc flags, tile_n): every N x element bytes is off a
# 16-byte multiple, so the last chunk of each row ends inside a granule
OUT_CASES = [
    (640, 1002, 320, 1004, "f32", 1, 0, 0),
    (777, 1003, 320, 1008, "bf16", 1, 0, 0),
    (777, 1005, 256, 1016, "f16", 1, dg.GEMM_FLAG_CTA_GROUP_1, 0),
    (1024, 1002, 512, 1004, "f32", 1, dg.GEMM_FLAG_CTA_GROUP_2, 512),
    (640, 1002, 320, 1004, "f32", 1, dg.GEMM_FLAG_EPILOGUE_DIRECT, 0),
    (300, 1002, 256, 1004, "f32", 3, 0, 0),
    (100, 60, 64, 64, "f16", 1, 0, 0),                      # single-CTA kernel
]


@pytest.mark.parametrize("M,N,K,ldd,out,batch,flags,tile_n", OUT_CASES)
def test_output_padding_untouched(M, N, K, ldd, out, batch, flags, tile_n):
    prob = inputs.make("square8192_bf16", M=M, N=N, K=K, batch=batch, dist="ints", seed=61)
    D = new_d(batch, M, ldd, out)
    desc = dg.make_desc(M, N, K, batch=batch, dtype_a=dg.GEMM_BF16, dtype_d=CODE[out], ldd=ldd,
                        stride_d=M * ldd, flags=flags, tile_n=tile_n)
    with dg.Plan(desc) as plan:
        plan.run(prob.A.cuda(), prob.B.cuda(), D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    dref, sabs = oracle.gemm(prob.A, prob.B, M=M, N=N, K=K, batch=batch, dtype_a="bf16", dtype_b="bf16")
    check_d(D, dref, sabs, batch, M, N, ldd, out, TOL_16BIT)


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("N,ldd,out", [(1003, 1008, "bf16"), (1002, 1004, "f32")])
def test_output_padding_untouched_fp8_block(N, ldd, out, cg_flag):
    M, K = 512, 384
    prob = inputs.make("fp8_block8192", M=M, N=N, K=K, dist="ints", seed=62)
    D = new_d(1, M, ldd, out)
    desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_E4M3, dtype_d=CODE[out], ldd=ldd,
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128, flags=cg_flag, tile_n=256)
    with dg.Plan(desc) as plan:
        plan.run(prob.A.cuda(), prob.B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda())
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    dref, sabs = oracle.gemm(prob.A, prob.B, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3",
                             scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy())
    check_d(D, dref, sabs, 1, M, N, ldd, out, TOL_FP8)


@pytest.mark.parametrize("name,N,ldd,out", [("mxfp8_8192", 1003, 1008, "bf16"), ("nvfp4_8192", 1002, 1004, "f32"),
                                            ("mxfp4_8192", 1005, 1016, "f16")])
def test_output_padding_untouched_block_scaled(name, N, ldd, out):
    M, K = 384, 512
    prob = inputs.make(name, M=M, N=N, K=K, dist="ints", seed=63)
    wl = prob.wl
    mode = {"mx": dg.GEMM_SCALE_MX_E8M0_32, "nv": dg.GEMM_SCALE_NV_E4M3_16}[wl.extra["scale_mode"]]
    code = {"e4m3": dg.GEMM_E4M3, "e2m1": dg.GEMM_E2M1}[wl.dtype_in]
    D = new_d(1, M, ldd, out)
    desc = dg.make_desc(M, N, K, dtype_a=code, dtype_d=CODE[out], ldd=ldd, scale_mode=mode,
                        flags=dg.GEMM_FLAG_CTA_GROUP_2)
    ts = torch.tensor(prob.tensor_scales, dtype=torch.float32, device="cuda") if wl.extra["scale_mode"] == "nv" else None
    with dg.Plan(desc) as plan:
        plan.run_mx(prob.A.cuda(), prob.B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda(), ts)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    dref, sabs = oracle.gemm(prob.A, prob.B, M=M, N=N, K=K, dtype_a=wl.dtype_in, dtype_b=wl.extra["dtype_b"],
                             scale_a=prob.scale_a, scale_b=prob.scale_b, scale_mode=wl.extra["scale_mode"],
                             tensor_scales=prob.tensor_scales)
    check_d(D, dref, sabs, 1, M, N, ldd, out, TOL_16BIT)


# (label, workload, dtype code, oracle dtype, K, lda): K x element bytes off a 16-byte
# multiple, so each operand row's last K elements share a granule with padding
OPERAND_CASES = [
    ("bf16", "square8192_bf16", dg.GEMM_BF16, "bf16", 1001, 1008),
    ("bf16 pair 512-wide", "square8192_bf16", dg.GEMM_BF16, "bf16", 1001, 1008),
    ("fp8 block-scaled", "fp8_block8192", dg.GEMM_E4M3, "e4m3", 1000, 1008),
]


@pytest.mark.parametrize("label,name,code,odt,K,ld", OPERAND_CASES)
def test_operand_padding_not_read(label, name, code, odt, K, ld):
    M, N = 512, 1024
    prob = inputs.make(name, M=M, N=N, K=K, dist="ints", seed=64)
    A = pad_rows(prob.A, ld, NAN_E4M3)
    B = pad_rows(prob.B, ld, NAN_E4M3)
    D = new_d(1, M, N, "f32")
    fp8 = code == dg.GEMM_E4M3
    kw = dict(flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=512) if "512" in label else {}
    desc = dg.make_desc(M, N, K, dtype_a=code, dtype_d=dg.GEMM_F32, lda=ld, ldb=ld,
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128 if fp8 else dg.GEMM_SCALE_NONE, **kw)
    with dg.Plan(desc) as plan:
        if fp8:
            plan.run(A.cuda(), B.cuda(), D, prob.scale_a.cuda(), prob.scale_b.cuda())
        else:
            plan.run(A.cuda(), B.cuda(), D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    extra = dict(scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy()) if fp8 else {}
    dref, sabs = oracle.gemm(A, B, M=M, N=N, K=K, dtype_a=odt, dtype_b=odt, lda=ld, ldb=ld, **extra)
    check_d(D, dref, sabs, 1, M, N, N, "f32", TOL_FP8 if fp8 else TOL_16BIT)


def test_operand_padding_not_read_tf32():
    """fp32 operands read at tf32 precision: K = 1001 (4004 bytes per row)."""
    M, N, K, ld = 384, 640, 1001, 1004
    g = torch.Generator().manual_seed(65)
    A0 = torch.randint(-3, 4, (M, K), generator=g).float()
    B0 = torch.randint(-3, 4, (N, K), generator=g).float()
    A, B = pad_rows(A0, ld), pad_rows(B0, ld)
    D = new_d(1, M, N, "f32")
    desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_TF32, dtype_d=dg.GEMM_F32, lda=ld, ldb=ld)
    with dg.Plan(desc) as plan:
        plan.run(A.cuda(), B.cuda(), D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    dref, sabs = oracle.gemm(A, B, M=M, N=N, K=K, dtype_a="f32", dtype_b="f32", lda=ld, ldb=ld)
    check_d(D, dref, sabs, 1, M, N, N, "f32", 4e-3)
