"""GPU: problems with fewer output tiles than SMs (or SM pairs).

The planner then grows the grid past the tile count and splits every tile
along K over several clusters (equal ranges per tile; a CTA cap below that
grid leaves ranges that straddle tiles).  Each cluster but the one holding a tile's
last K blocks leaves an fp32 partial, and that finisher adds them all, the
latest K range first, before writing D.  Ranges need not line up with tiles:
with a grid that is not a multiple of the tile count a cluster can hold the
end of one tile and the start of the next, or a middle piece of one tile.

Integer-valued inputs keep every partial sum exact in fp32, so the result
must equal the oracle's bit for bit whatever the split.  Random inputs check
the fp32 error bound.  Every case runs twice on one plan, because the second
launch reuses the partial slots and flags under a new epoch.
"""
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


def run_twice(M, N, K, out, dist, seed, batch=1, **kw):
    prob = inputs.make("square8192_bf16", M=M, N=N, K=K, batch=batch, dist=dist, seed=seed)
    A, B = prob.A.cuda(), prob.B.cuda()
    shape = (batch, M, N) if batch > 1 else (M, N)
    desc = dg.make_desc(M, N, K, batch=batch, dtype_a=dg.GEMM_BF16, dtype_d=CODE[out], **kw)
    results = []
    with dg.Plan(desc) as plan:
        info = plan.info.as_dict()
        for _ in range(2):
            D = torch.full(shape, float("nan"), dtype=TDT[out], device="cuda")
            plan.run(A, B, D)
            s, rec = plan.sync_status()
            assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role, rec.stage, rec.tile)
            results.append(D.double().cpu().numpy())
    dref, sabs = oracle.gemm(prob.A, prob.B, M=M, N=N, K=K, batch=batch, dtype_a="bf16", dtype_b="bf16")
    return results, dref, sabs, info


def parts_per_tile(M, N, K, info, batch=1, **kw):
    desc = dg.make_desc(M, N, K, batch=batch, dtype_a=dg.GEMM_BF16, **kw)
    plan_info = dg.GemmPlanInfo()
    for name, value in info.items():
        setattr(plan_info, name, value)
    counts = {}
    for c in range(info["grid"] // info["cta_group"]):
        for i in range(64):
            s, u = dg.gemm_plan_work_unit(desc, plan_info, c, i)
            assert s == dg.GEMM_OK
            if u.tile < 0:
                break
            counts[u.tile] = counts.get(u.tile, 0) + 1
    return counts


# (M, N, K, out, batch, plan options): one tile, aligned splits, uneven ranges
# across tile boundaries (a CTA cap below tiles x splits), SM pairs with
# 512-wide tiles, a ragged edge and a batch
CASES = [
    (64, 64, 65536, "f32", 1, {}),
    (256, 256, 16384, "bf16", 1, {}),
    (128, 2048, 4096, "bf16", 1, {}),
    (128, 2048, 4096, "bf16", 1, {"tile_n": 256}),
    (128, 2048, 4096, "f32", 1, {"max_ctas": 13, "tile_n": 256}),
    (200, 1000, 4160, "f16", 1, {"max_ctas": 11, "tile_n": 256}),
    (1024, 2048, 8192, "f32", 1, {"flags": dg.GEMM_FLAG_CTA_GROUP_2, "tile_n": 512}),
    (512, 768, 6144, "bf16", 1, {"flags": dg.GEMM_FLAG_CTA_GROUP_2, "tile_n": 256}),
    (128, 256, 8192, "f32", 3, {}),
    (128, 512, 4096, "f32", 1, {"flags": dg.GEMM_FLAG_EPILOGUE_DIRECT}),
]


@pytest.mark.parametrize("M,N,K,out,batch,kw", CASES)
def test_few_tiles_split_integers_bit_exact(M, N, K, out, batch, kw):
    results, dref, sabs, info = run_twice(M, N, K, out, "ints", 91, batch=batch, **kw)
    assert info["stream_k_tiles"] == info["num_tiles"] < info["grid"] // info["cta_group"], info
    parts = parts_per_tile(M, N, K, info, batch=batch, dtype_d=CODE[out], **kw)
    assert max(parts.values()) >= 2, parts
    shape = (batch, M, N) if batch > 1 else (M, N)
    for n, got in enumerate(results):
        r = compare(got, dref.reshape(shape), sabs.reshape(shape), out, TOL_16BIT, exact=True)
        if not r["ok"]:
            dump_on_failure("few_tiles_%dx%dx%d_run%d" % (M, N, K, n), got=got, dref=dref, sabs=sabs)
        assert r["ok"], (r, info, n)


@pytest.mark.parametrize("M,N,K,out,kw", [
    (64, 64, 65536, "f32", {}),
    (256, 1024, 8192, "bf16", {"max_ctas": 27}),
])
def test_few_tiles_split_random(M, N, K, out, kw):
    results, dref, sabs, info = run_twice(M, N, K, out, "normal", 92, **kw)
    assert info["stream_k_tiles"] == info["num_tiles"] < info["grid"] // info["cta_group"], info
    for got in results:
        r = compare(got, dref, sabs, out, TOL_16BIT)
        assert r["ok"], (r, info)
    # one fixed order of additions: the two launches agree bit for bit
    assert (results[0] == results[1]).all()


def test_few_tiles_opt_out_matches():
    """The same problem without stream-K (one cluster per tile) gives the same
    integers: the split changes the work's placement, not the result."""
    M, N, K = 128, 1024, 8192
    split, dref, sabs, info = run_twice(M, N, K, "f32", "ints", 93)
    whole, _, _, info1 = run_twice(M, N, K, "f32", "ints", 93, flags=dg.GEMM_FLAG_NO_STREAM_K)
    assert info["stream_k_tiles"] > 0 and info1["stream_k_tiles"] == 0
    assert info1["grid"] == info1["num_tiles"] * info1["cta_group"]
    assert (split[0] == whole[0]).all() and (split[0] == oracle.round_to("f32", dref)).all()


def test_few_tiles_split_tf32_integers_bit_exact():
    """fp32 storage at tf32 precision (32-element K atoms): small integers are
    exact, so the split product equals the oracle bit for bit."""
    M, N, K = 128, 1024, 4096
    g = torch.Generator().manual_seed(94)
    A = torch.randint(-3, 4, (M, K), generator=g).float()
    B = torch.randint(-3, 4, (N, K), generator=g).float()
    desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_TF32, dtype_d=dg.GEMM_F32)
    D = torch.full((M, N), float("nan"), device="cuda")
    with dg.Plan(desc) as plan:
        info = plan.info.as_dict()
        plan.run(A.cuda(), B.cuda(), D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    assert info["stream_k_tiles"] == info["num_tiles"] < info["grid"] // info["cta_group"], info
    dref, sabs = oracle.gemm(A, B, M=M, N=N, K=K, dtype_a="f32", dtype_b="f32")
    r = compare(D.double().cpu().numpy(), dref, sabs, "f32", 4e-3, exact=True)
    assert r["ok"], (r, info)


@pytest.mark.parametrize("mn_a,mn_b", [(True, False), (False, True), (True, True)])
def test_few_tiles_split_mn_major_f16_bit_exact(mn_a, mn_b):
    """MN-major operands (stored [k][m] / [k][n]) on split tiles, f16 in and out."""
    M, N, K = 256, 512, 8192
    prob = inputs.make("square8192_bf16", M=M, N=N, K=K, dist="ints", seed=95, dtype_in="f16")
    A, B = prob.A, prob.B
    As = A.t().contiguous() if mn_a else A
    Bs = B.t().contiguous() if mn_b else B
    desc = dg.make_desc(M, N, K, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F16,
                        major_a=dg.GEMM_MN_MAJOR if mn_a else dg.GEMM_K_MAJOR,
                        major_b=dg.GEMM_MN_MAJOR if mn_b else dg.GEMM_K_MAJOR)
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    with dg.Plan(desc) as plan:
        info = plan.info.as_dict()
        plan.run(As.cuda(), Bs.cuda(), D)
        s, rec = plan.sync_status()
        assert s == dg.GEMM_OK, dg.gemm_status_string(s)
    assert info["stream_k_tiles"] == info["num_tiles"] < info["grid"] // info["cta_group"], info
    dref, sabs = oracle.gemm(As, Bs, M=M, N=N, K=K, dtype_a="f16", dtype_b="f16",
                             major_a="mn" if mn_a else "k", major_b="mn" if mn_b else "k")
    r = compare(D.double().cpu().numpy(), dref, sabs, "f16", TOL_16BIT, exact=True)
    assert r["ok"], (r, info)
