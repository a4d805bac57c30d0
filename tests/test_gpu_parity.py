"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Small cases are compared element by element over the whole output; they span
several tiles and ragged tails in M, N and K.  Full-size workloads (the sizes
the benchmark times, in the same launch configuration) are compared on sampled
rows: seeded random rows plus the first and last row of every tile edge, each
over every column.  Integer-valued inputs must match bit for bit.
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


def run_gpu(prob, out_dtype, **desc_kw):
    """D via the C ABI for the host tensors of `prob` (A [b][M][K], B [b][N][K])."""
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    shape = (wl.batch, wl.M, wl.N) if wl.batch > 1 else (wl.M, wl.N)
    D = torch.full(shape, float("nan"), dtype=TDT[out_dtype], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=CODE[wl.dtype_in], dtype_d=CODE[out_dtype],
                        **desc_kw)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role, rec.stage, rec.tile)
        info = plan.info.as_dict()
    return D, info


def oracle_rows(prob, rows=None):
    wl = prob.wl
    return oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, batch=wl.batch,
                            dtype_a=wl.dtype_in, dtype_b=wl.dtype_in, rows=rows)


def check_full(prob, out_dtype, exact=False, **desc_kw):
    D, info = run_gpu(prob, out_dtype, **desc_kw)
    dref, s = oracle_rows(prob)
    got = D.double().cpu().numpy().reshape(dref.shape)
    r = compare(got, dref, s, out_dtype, TOL_16BIT, exact=exact)
    if not r["ok"]:
        dump_on_failure("%s_%dx%dx%dx%d" % (out_dtype, prob.wl.batch, prob.wl.M, prob.wl.N, prob.wl.K),
                        got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)
    return r, info


# ------------------------------------------------------------------ single CTA

def test_single_cta_example_integers_bit_exact():
    prob = inputs.make("single_cta_ints")
    r, info = check_full(prob, "f32", exact=True)
    assert info["kernel"] == dg.GEMM_KERNEL_SINGLE_CTA


def test_single_cta_example_uniform():
    prob = inputs.make("single_cta")
    D, info = run_gpu(prob, "f32")
    a, b = prob.A.cuda(), prob.B.cuda()
    # the walk-through's own check
    torch.testing.assert_close(D, a.float() @ b.float().T, rtol=2e-4, atol=2e-4)
    dref, s = oracle_rows(prob)
    assert compare(D.double().cpu().numpy().reshape(dref.shape), dref, s, "f32", TOL_16BIT)["ok"]


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_single_cta_ragged_batched(out):
    prob = inputs.make("single_cta", M=100, N=40, K=104, batch=3, seed=9)   # rows of 208 B: 16-B multiples
    prob.wl.dtype_in = "bf16"
    prob.A, prob.B = prob.A.float().bfloat16(), prob.B.float().bfloat16()
    check_full(prob, out)


def test_single_cta_mn_major():
    g = torch.Generator().manual_seed(10)
    M, N, K = 80, 56, 90   # MN-major rows are M (resp. N) long: 160 B and 112 B
    a = torch.randint(-3, 4, (M, K), generator=g).half()
    b = torch.randint(-3, 4, (N, K), generator=g).half()
    at, bt = a.t().contiguous().cuda(), b.t().contiguous().cuda()     # [K][M], [K][N]
    D = torch.empty(M, N, dtype=torch.float32, device="cuda")
    desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32, major_a=dg.GEMM_MN_MAJOR,
                        major_b=dg.GEMM_MN_MAJOR, lda=at.stride(0), ldb=bt.stride(0))
    with dg.Plan(desc) as plan:
        plan.run(at, bt, D)
        assert plan.sync_status()[0] == dg.GEMM_OK
    dref, _ = oracle.gemm(a, b, M=M, N=N, K=K, dtype_a="f16", dtype_b="f16")
    assert np.array_equal(D.double().cpu().numpy(), dref[0])


# ------------------------------------------------------------------ persistent, small

@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
def test_persistent_integers_bit_exact(cg_flag):
    prob = inputs.make("square8192_bf16", M=520, N=600, K=336, dist="ints", seed=11)   # K tail of 16
    r, info = check_full(prob, "f32", exact=True, flags=cg_flag)
    assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT
    assert info["cta_group"] == (1 if cg_flag == dg.GEMM_FLAG_CTA_GROUP_1 else 2)


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("dtype_in,out", [("bf16", "f32"), ("bf16", "bf16"), ("f16", "f16"), ("f16", "f32")])
def test_persistent_ragged(cg_flag, dtype_in, out):
    prob = inputs.make("square4096_bf16", M=300, N=520, K=200, seed=12)
    if dtype_in == "f16":
        prob.wl.dtype_in = "f16"
        prob.A, prob.B = prob.A.float().half(), prob.B.float().half()
    check_full(prob, out, flags=cg_flag)


@pytest.mark.parametrize("mode", [dg.GEMM_FLAG_EPILOGUE_DIRECT, dg.GEMM_FLAG_EPILOGUE_TMA])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_epilogue_modes_ragged(mode, out):
    """Direct row stores and TMA-staged stores write the same D, ragged edges included."""
    prob = inputs.make("square8192_bf16", M=600, N=712, K=3136, dist="ints", seed=19)
    r, info = check_full(prob, out, exact=True, flags=dg.GEMM_FLAG_CTA_GROUP_2 | mode)
    assert info["epilogue"] == (1 if mode == dg.GEMM_FLAG_EPILOGUE_DIRECT else 0)
    r, info = check_full(prob, out, exact=True, flags=dg.GEMM_FLAG_CTA_GROUP_2 | mode, max_ctas=8)
    assert info["stream_k_tiles"] > 0


@pytest.mark.parametrize("tile_n", [64, 128, 192, 256])
def test_persistent_tile_widths(tile_n):
    prob = inputs.make("square8192_bf16", M=384, N=700, K=256, dist="ints", seed=13)
    check_full(prob, "f32", exact=True, tile_n=tile_n, flags=dg.GEMM_FLAG_CTA_GROUP_1)


def test_persistent_few_ctas_many_tiles():
    """More tiles than CTAs: every CTA loops over tiles, both TMEM buffers cycle."""
    prob = inputs.make("square8192_bf16", M=1024, N=1024, K=128, dist="ints", seed=14)
    check_full(prob, "f32", exact=True, max_ctas=4, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    check_full(prob, "f32", exact=True, max_ctas=3, flags=dg.GEMM_FLAG_CTA_GROUP_1)


@pytest.mark.parametrize("cg_flag,M,N,K,ctas,out", [
    (dg.GEMM_FLAG_CTA_GROUP_2, 1024, 1024, 3072, 10, "f32"),
    (dg.GEMM_FLAG_CTA_GROUP_2, 600, 704, 3088, 8, "bf16"),
    (dg.GEMM_FLAG_CTA_GROUP_1, 640, 768, 3200, 7, "f32"),
    (dg.GEMM_FLAG_CTA_GROUP_1, 520, 600, 4112, 4, "f16"),
])
def test_stream_k_integers_bit_exact(cg_flag, M, N, K, ctas, out):
    """Capping the clusters forces a partial last wave: its tiles are split
    along K between two clusters (contributor partial + finisher)."""
    prob = inputs.make("square8192_bf16", M=M, N=N, K=K, dist="ints", seed=17)
    r, info = check_full(prob, out, exact=True, flags=cg_flag, max_ctas=ctas, tile_n=256)
    assert info["stream_k_tiles"] > 0


@pytest.mark.parametrize("cg_flag,M,N,K,ctas,out", [
    (dg.GEMM_FLAG_CTA_GROUP_2, 600, 1000, 3088, 16, "f32"),   # 12 tiles on 8 pairs
    (dg.GEMM_FLAG_CTA_GROUP_1, 520, 600, 4112, 8, "bf16"),    # 15 tiles on 8 CTAs
])
def test_stream_k_only_ragged_bit_exact(cg_flag, M, N, K, ctas, out):
    """Every tile in the stream-K region, so each finisher is its cluster's
    last unit and gathers the partial through the operand ring; ragged M, N
    and K leave some of its chunks (and, past M, whole warps) without work."""
    prob = inputs.make("square8192_bf16", M=M, N=N, K=K, dist="ints", seed=19)
    r, info = check_full(prob, out, exact=True, flags=cg_flag, max_ctas=ctas, tile_n=256)
    assert info["stream_k_tiles"] == info["num_tiles"], info


def test_stream_k_matches_data_parallel():
    prob = inputs.make("square4096_bf16", M=1024, N=768, K=4096, seed=18)
    D1, info1 = run_gpu(prob, "f32", flags=dg.GEMM_FLAG_CTA_GROUP_2, max_ctas=10)
    D2, info2 = run_gpu(prob, "f32", flags=dg.GEMM_FLAG_CTA_GROUP_2 | dg.GEMM_FLAG_NO_STREAM_K, max_ctas=10)
    assert info1["stream_k_tiles"] > 0 and info2["stream_k_tiles"] == 0
    dref, s = oracle_rows(prob)
    for D in (D1, D2):
        assert compare(D.double().cpu().numpy().reshape(dref.shape), dref, s, "f32", TOL_16BIT)["ok"]
    # repeated launches of one plan reuse the partial slots (flags carry a launch counter)
    desc = dg.make_desc(prob.wl.M, prob.wl.N, prob.wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                        flags=dg.GEMM_FLAG_CTA_GROUP_2, max_ctas=10)
    A, B = prob.A.cuda(), prob.B.cuda()
    with dg.Plan(desc) as plan:
        for _ in range(3):
            D = torch.full_like(D1, float("nan"))
            plan.run(A, B, D)
            assert plan.sync_status()[0] == dg.GEMM_OK
            assert torch.equal(D, D1)


def test_persistent_batched_small():
    prob = inputs.make("batched256_f16", batch=7, seed=15)
    check_full(prob, "f16")
    prob = inputs.make("batched256_f16", M=200, N=136, K=72, batch=5, seed=16)
    check_full(prob, "f16", flags=dg.GEMM_FLAG_NO_SINGLE_CTA)


def test_k_zero_writes_zeros_and_empty_is_noop():
    for M, N, K in [(33, 72, 0), (0, 16, 16), (16, 0, 16)]:
        D = torch.full((max(M, 1), max(N, 1)), 7.0, device="cuda")
        A = torch.zeros(max(M, 1), 16, dtype=torch.bfloat16, device="cuda")
        B = torch.zeros(max(N, 1), 16, dtype=torch.bfloat16, device="cuda")
        with dg.Plan(dg.make_desc(M, N, K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, lda=16, ldb=16,
                                  ldd=max(N, 1))) as plan:
            plan.run(A, B, D)
            torch.cuda.synchronize()
        if K == 0 and M and N:
            assert (D == 0).all()
        else:
            assert (D == 7.0).all()


def test_misaligned_pointer_is_rejected():
    A = torch.zeros(256 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    D = torch.zeros(256, 256, dtype=torch.float32, device="cuda")
    with dg.Plan(dg.make_desc(256, 256, 64, dtype_a=dg.GEMM_BF16)) as plan:
        s = dg.gemm_run(plan.handle, A.data_ptr() + 2, B.data_ptr(), D.data_ptr(), None, None,
                        torch.cuda.current_stream().cuda_stream)
        assert s == dg.GEMM_ERR_ALIGNMENT


# ------------------------------------------------------------------ full-size workloads (sampled)

def check_sampled(name, out_dtype, rows_per_tile=None, **desc_kw):
    prob = inputs.make(name)
    D, info = run_gpu(prob, out_dtype, **desc_kw)
    wl = prob.wl
    rows = inputs.sample_rows(wl.M, wl.batch, n_random=48, seed=1, tile_m=info["tile_m"])
    dref, s = oracle_rows(prob, rows)
    got = D.reshape(wl.batch * wl.M, wl.N)[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, out_dtype, TOL_16BIT)
    assert r["ok"], (name, r, info)
    return r, info


@pytest.mark.slow
def test_full_square8192_bf16_f32():
    r, info = check_sampled("square8192_bf16", "f32")
    assert info["cta_group"] == 2 and info["tile_n"] == 512 and info["tmem_stages"] == 1   # 512-wide pair tiles


@pytest.mark.slow
def test_full_square4096_bf16_bf16():
    check_sampled("square4096_bf16", "bf16")


@pytest.mark.slow
def test_full_batched256_f16():
    check_sampled("batched256_f16", "f16")


# ------------------------------------------------------------------ full-size workloads, integer-valued, bit-exact
#
# The same shapes, element types and default plans the benchmark times (pair
# tiles, the whole grid, the raster groups and the serpentine K order), with
# entries in {-3..3}: every partial sum stays below 9 K <= 73,728 < 2^24 in
# magnitude, so any fp32 summation order gives the exact sum and the one
# rounding to D's type must equal the oracle's rounding bit for bit.  A dropped,
# repeated or misplaced K slice changes some element by an integer and fails.

def check_sampled_exact(name, out_dtype, whole=False, expect=None, **desc_kw):
    prob = inputs.make(name, dist="ints")
    wl = prob.wl
    D, info = run_gpu(prob, out_dtype, **desc_kw)
    if expect:
        assert {k: info[k] for k in expect} == expect, info
    if whole:
        dref, s = oracle_rows(prob)
        got = D.double().cpu().numpy().reshape(dref.shape)
    else:
        # seeded random rows plus the first and last row of every 128-row
        # block (each CTA's own rows, not only the pair tile's edges)
        rows = inputs.sample_rows(wl.M, wl.batch, n_random=64, seed=3, tile_m=128)
        dref, s = oracle_rows(prob, rows)
        got = D.reshape(wl.batch * wl.M, wl.N)[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref, s, out_dtype, TOL_16BIT, exact=True)
    if not r["ok"]:
        dump_on_failure("exact_" + name, got=got, dref=dref, sabs=s)
    assert r["ok"], (name, r, info)
    return info


@pytest.mark.slow
def test_full_square8192_bf16_f32_integers_bit_exact():
    check_sampled_exact("square8192_bf16", "f32",
                        expect={"cta_group": 2, "tile_n": 512, "tmem_stages": 1, "grid": 152, "stream_k_tiles": 0})


@pytest.mark.slow
def test_full_square8192_bf16_f32_256x256_pair_tiles_integers_bit_exact():
    """The configuration's literal plan: cta_group::2 with 256 x 256 tiles (two
    accumulators, two-atom stages, stream-K over the partial last wave)."""
    check_sampled_exact("square8192_bf16", "f32", tile_n=256, flags=dg.GEMM_FLAG_CTA_GROUP_2,
                        expect={"cta_group": 2, "tile_n": 256, "tmem_stages": 2})


@pytest.mark.slow
def test_full_square4096_bf16_bf16_integers_bit_exact():
    check_sampled_exact("square4096_bf16", "bf16", expect={"cta_group": 2, "tile_n": 512})


@pytest.mark.slow
def test_full_batched256_f16_integers_bit_exact_whole_output():
    check_sampled_exact("batched256_f16", "f16", whole=True)

