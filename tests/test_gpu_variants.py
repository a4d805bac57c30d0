"""GPU parity of the variant input types against the CPU oracle.

tf32: fp32 storage multiplied at tf32 precision (kind::tf32, K = 8 per
instruction).  Small integers are exact in tf32, so integer runs must match
bit for bit; random inputs must stay within 4e-3 of S = sum |a||b| (the
oracle uses the exact fp32 inputs; see tests/parity.py for the bound).
e5m2: the block-scaled kernel with E5M2 operands, alone and paired with E4M3
(kind::f8f6f4 takes the two formats independently).
"""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import TOL_FP8, TOL_TF32, compare, dump_on_failure

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32, "tf32": dg.GEMM_TF32,
        "e4m3": dg.GEMM_E4M3, "e5m2": dg.GEMM_E5M2}


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def run(prob, out, **kw):
    wl = prob.wl
    db = wl.extra["dtype_b"]
    A, B = prob.A.cuda(), prob.B.cuda()
    sa = prob.scale_a.cuda() if prob.scale_a is not None else None
    sb = prob.scale_b.cuda() if prob.scale_b is not None else None
    D = torch.full((wl.M, wl.N), float("nan"), dtype=TDT[out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=CODE[wl.dtype_in], dtype_b=CODE[db], dtype_d=CODE[out],
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128 if sa is not None else 0, **kw)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D, sa, sb)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
        info = plan.info.as_dict()
    ref_a = "f32" if wl.dtype_in == "tf32" else wl.dtype_in
    ref_b = "f32" if db == "tf32" else db
    kw_o = {}
    if sa is not None:
        kw_o = dict(scale_a=prob.scale_a.numpy(), scale_b=prob.scale_b.numpy())
    dref, s = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a=ref_a, dtype_b=ref_b, **kw_o)
    return D.double().cpu().numpy(), dref[0], s[0], info


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tf32_integers_bit_exact(cg_flag, out):
    prob = inputs.make("square8192_bf16", M=600, N=712, K=1060, dist="ints", seed=71, dtype_in="tf32")
    got, dref, s, info = run(prob, out, flags=cg_flag)
    assert info["tile_k"] in (32, 64)   # one or two 128-byte atoms of 32 tf32 (two if three stages fit)
    r = compare(got, dref, s, out, TOL_TF32, exact=True)
    if not r["ok"]:
        dump_on_failure("tf32_%s_%d" % (out, cg_flag), got=got, dref=dref, sabs=s)
    assert r["ok"], r


def test_tf32_random_and_stream_k():
    prob = inputs.make("square4096_bf16", M=1024, N=1024, K=2048, seed=72, dtype_in="tf32")
    got, dref, s, info = run(prob, "f32", flags=dg.GEMM_FLAG_CTA_GROUP_2, max_ctas=10, tile_n=256)
    assert info["stream_k_tiles"] > 0
    r = compare(got, dref, s, "f32", TOL_TF32)
    assert r["ok"], r


@pytest.mark.parametrize("fa,fb", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_fp8_format_pairings_bit_exact(fa, fb):
    prob = inputs.make("fp8_block8192", M=400, N=520, K=384, dist="ints", seed=73, dtype_in=fa, dtype_b=fb)
    got, dref, s, info = run(prob, "bf16")
    assert info["kernel"] == dg.GEMM_KERNEL_FP8_BLOCK
    r = compare(got, dref, s, "bf16", TOL_FP8, exact=True)
    assert r["ok"], r


def test_e5m2_quantised_normal():
    prob = inputs.make("fp8_block8192", M=300, N=520, K=512, seed=74, dtype_in="e5m2")
    got, dref, s, info = run(prob, "bf16")
    r = compare(got, dref, s, "bf16", TOL_FP8)
    assert r["ok"], r


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("dtype_in,K", [("bf16", 1000), ("bf16", 64), ("f16", 200), ("tf32", 1060), ("tf32", 32)])
def test_two_atom_stages_bit_exact(cg_flag, dtype_in, K):
    """Ring stages two 128-byte K atoms deep: the second atom of the last
    stage is partly (K = 1000, 200, 1060) or wholly (K = 64, 32) past K and
    reads TMA's zero fill."""
    prob = inputs.make("square8192_bf16", M=520, N=600, K=K, dist="ints", seed=73, dtype_in=dtype_in)
    got, dref, s, info = run(prob, "f32", flags=cg_flag | dg.GEMM_FLAG_STAGE_K2 | dg.GEMM_FLAG_NO_SINGLE_CTA)
    assert info["tile_k"] == (128 if dtype_in != "tf32" else 64)
    assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT
    r = compare(got, dref, s, "f32", TOL_TF32, exact=True)
    if not r["ok"]:
        dump_on_failure("k2_%s_%d_cg%d" % (dtype_in, K, info["cta_group"]), got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


def test_two_atom_stages_stream_k_random():
    """Stream-K splits count K blocks of the deeper stage (sampled rows of
    every tile row band against the oracle)."""
    prob = inputs.make("square8192_bf16", M=2048, N=2560, K=4096, seed=74)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.full((wl.M, wl.N), float("nan"), device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                        flags=dg.GEMM_FLAG_CTA_GROUP_2 | dg.GEMM_FLAG_STAGE_K2)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D)
        assert plan.sync_status()[0] == dg.GEMM_OK
        info = plan.info.as_dict()
    assert info["stream_k_tiles"] > 0 and info["tile_k"] == 128
    rows = inputs.sample_rows(wl.M, 1, n_random=48, seed=2, tile_m=info["tile_m"])
    dref, s = oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="bf16", dtype_b="bf16", rows=rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref.reshape(got.shape), s.reshape(got.shape), "f32", 2e-3)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("cg_flag", [dg.GEMM_FLAG_CTA_GROUP_1, dg.GEMM_FLAG_CTA_GROUP_2])
@pytest.mark.parametrize("dtype_in,out,epi", [("bf16", "f32", dg.GEMM_FLAG_EPILOGUE_TMA),
                                             ("bf16", "f32", dg.GEMM_FLAG_EPILOGUE_DIRECT),
                                             ("f16", "bf16", dg.GEMM_FLAG_EPILOGUE_TMA),
                                             ("tf32", "f32", dg.GEMM_FLAG_EPILOGUE_DIRECT)])
def test_wide_tiles_bit_exact(cg_flag, dtype_in, out, epi):
    """512-wide tiles: two N = 256 MMAs per K step into one 512-column
    accumulator.  N = 1104 leaves the third tile column mostly past N."""
    prob = inputs.make("square8192_bf16", M=520, N=1104, K=400, dist="ints", seed=75, dtype_in=dtype_in)
    got, dref, s, info = run(prob, out, flags=cg_flag | epi, tile_n=512)
    assert info["tile_n"] == 512 and info["tmem_stages"] == 1 and info["tmem_cols"] == 512
    r = compare(got, dref, s, out, TOL_TF32, exact=True)
    if not r["ok"]:
        dump_on_failure("wide_%s_%s_cg%d" % (dtype_in, out, info["cta_group"]), got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("cg_flag,max_ctas", [(dg.GEMM_FLAG_CTA_GROUP_1, 5), (dg.GEMM_FLAG_CTA_GROUP_2, 6)])
@pytest.mark.parametrize("K", [1472, 1536, 1560])
def test_wide_tiles_split_schedule_bit_exact(cg_flag, max_ctas, K):
    """A 512-wide whole tile of at least 24 K blocks runs its first six K
    blocks for the left accumulator half alone and repeats them for the right
    half after its last one: K = 1472 is 23 blocks (no split), 1536 is 24 and
    1560 is 25 with a ragged last block.  Four tiles per cluster (max_ctas),
    so every other tile walks K backwards and each tile's split stages follow
    the previous tile's."""
    prob = inputs.make("square8192_bf16", M=520, N=2048, K=K, dist="ints", seed=77)
    got, dref, s, info = run(prob, "f32", flags=cg_flag, tile_n=512, max_ctas=max_ctas)
    assert info["tile_n"] == 512 and info["num_tiles"] == 4 * info["grid"] // info["cta_group"]
    r = compare(got, dref, s, "f32", TOL_TF32, exact=True)
    if not r["ok"]:
        dump_on_failure("wide_split_K%d_cg%d" % (K, info["cta_group"]), got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


def test_wide_tiles_stream_k_and_split_integers_bit_exact():
    """One launch with both kinds of 512-wide units: the stream-K region's
    partial units run every stage on both halves, the data-parallel whole
    tiles after them run the split schedule.  Integer inputs: every partial
    sum, the fp32 fix-up included, is exact."""
    prob = inputs.make("square8192_bf16", M=4096, N=5120, K=4096, dist="ints", seed=78)
    got, dref, s, info = run(prob, "f32", flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=512)
    assert info["tile_n"] == 512 and 0 < info["stream_k_tiles"] < info["num_tiles"], info
    r = compare(got, dref, s, "f32", TOL_TF32, exact=True)
    if not r["ok"]:
        dump_on_failure("wide_sk_split", got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


def test_wide_tiles_batched_split_integers_bit_exact():
    """512-wide split tiles across batch entries (3 x 512 x 1024 x 2048)."""
    prob = inputs.make("square8192_bf16", M=512, N=1024, K=2048, batch=3, dist="ints", seed=79)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.full((wl.batch, wl.M, wl.N), float("nan"), device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                        flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=512)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
        info = plan.info.as_dict()
    assert info["tile_n"] == 512
    dref, sabs = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, batch=wl.batch, dtype_a="bf16", dtype_b="bf16")
    r = compare(D.double().cpu().numpy(), dref, sabs, "f32", TOL_TF32, exact=True)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("epi", [dg.GEMM_FLAG_EPILOGUE_TMA, dg.GEMM_FLAG_EPILOGUE_DIRECT])
def test_wide_tiles_stream_k_random(epi):
    """512-wide pair tiles with stream-K (sampled rows of every tile row band)."""
    prob = inputs.make("square8192_bf16", M=2048, N=5120, K=4096, seed=76)
    wl = prob.wl
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.full((wl.M, wl.N), float("nan"), device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32,
                        flags=dg.GEMM_FLAG_CTA_GROUP_2 | epi, tile_n=512)
    with dg.Plan(desc) as plan:
        plan.run(A, B, D)
        assert plan.sync_status()[0] == dg.GEMM_OK
        info = plan.info.as_dict()
    assert info["stream_k_tiles"] > 0 and info["tile_n"] == 512
    rows = inputs.sample_rows(wl.M, 1, n_random=48, seed=3, tile_m=info["tile_m"])
    dref, s = oracle.gemm_rows(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a="bf16", dtype_b="bf16", rows=rows)
    got = D[torch.tensor(rows, device="cuda")].double().cpu().numpy()
    r = compare(got, dref.reshape(got.shape), s.reshape(got.shape), "f32", 2e-3)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("cg_flag,N", [(dg.GEMM_FLAG_CTA_GROUP_1, 600), (dg.GEMM_FLAG_CTA_GROUP_2, 600),
                                       (dg.GEMM_FLAG_CTA_GROUP_2, 2048)])
@pytest.mark.parametrize("out", ["f16", "f32"])
def test_fp16_accumulation_integers_bit_exact(cg_flag, N, out):
    """fp16 accumulator: integer inputs in [-3, 3] and K = 192 keep every
    partial sum an integer of magnitude <= 1728, exact in fp16, so the result
    is the exact product.  N = 2048 takes 512-wide pair tiles."""
    prob = inputs.make("batched256_f16", M=520, N=N, K=192, batch=1, dist="ints", seed=77)
    got, dref, s, info = run(prob, out, flags=cg_flag | dg.GEMM_FLAG_ACCUM_F16)
    assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT and info["stream_k_tiles"] == 0
    r = compare(got, dref, s, out, 0.0, exact=True)
    if not r["ok"]:
        dump_on_failure("acc16_%s_%d_cg%d" % (out, N, info["cta_group"]), got=got, dref=dref, sabs=s)
    assert r["ok"], (r, info)


def test_fp16_accumulation_random_within_bound_and_differs_from_fp32():
    """Random f16 inputs, K = 512: with the running sum rounded to fp16 at most
    once per 8 products (the tensor core rounds once per K16 instruction or
    less often), |D - exact| <= (K / 8) 2^-11 S.  The fp32-accumulated product
    of the same inputs must differ somewhere, or the flag did not take effect."""
    K = 512
    prob = inputs.make("batched256_f16", M=512, N=1024, K=K, batch=1, seed=78)
    got16, dref, s, info = run(prob, "f32", flags=dg.GEMM_FLAG_ACCUM_F16)
    r = compare(got16, dref, s, "f32", (K / 8) * 2.0 ** -11)
    assert r["ok"], (r, info)
    got32, _, _, _ = run(prob, "f32")
    assert compare(got32, dref, s, "f32", 2e-3)["ok"]
    assert (got16 != got32).any()
    # and fp32 accumulation is the closer of the two
    import numpy as np
    assert np.abs(got32 - dref).max() < np.abs(got16 - dref).max()
