"""CUDA-graph capture of gemm_run.

gemm_run only enqueues kernels on the caller's stream (no allocation, no
synchronisation, tensor maps encoded on the host), so a launch can be
captured into a CUDA graph and replayed with new data in the same buffers.
A replay reuses the captured kernel parameters; stream-K plans therefore take
each launch's epoch from a counter in device memory, so a replay never
mistakes a previous replay's published partials for its own."""
import pytest
import torch

import dense_gemm_blackwell_gb300 as dg
from dense_gemm_blackwell_gb300 import inputs
import oracle
from parity import compare

pytestmark = pytest.mark.gpu

TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
CODE = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32}


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()
    torch.cuda.init()


def capture(plan, A, B, D):
    """One warm-up launch outside the graph, then a captured one."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        plan.run(A, B, D)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run(A, B, D)
    return g


def replay_and_check(name, dtype_out, rounds, seed0, expect, flags=0, **kw):
    base = inputs.make(name, dist="ints", seed=seed0, **kw)
    wl = base.wl
    A, B = base.A.cuda(), base.B.cuda()
    D = torch.empty((wl.M, wl.N), dtype=TDT[dtype_out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=CODE[wl.dtype_in], dtype_d=CODE[dtype_out], flags=flags)
    with dg.Plan(desc) as plan:
        info = plan.info.as_dict()
        expect(info)
        g = capture(plan, A, B, D)
        for r in range(rounds):
            prob = inputs.make(name, dist="ints", seed=seed0 + 1 + r, **kw)
            A.copy_(prob.A.cuda())
            B.copy_(prob.B.cuda())
            D.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            s, rec = plan.sync_status()
            assert s == dg.GEMM_OK, (dg.gemm_status_string(s), rec.role)
            dref, sabs = oracle.gemm(prob.A, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in,
                                     dtype_b=wl.dtype_in)
            res = compare(D.double().cpu().numpy(), dref[0], sabs[0], dtype_out, 0.0, exact=True)
            assert res["ok"], (r, res, info)
    return info


def test_single_cta_graph_replays_new_data():
    """The 128x64x64 example (one CTA) captured once and replayed on three new
    integer-valued inputs, each bit-exact against the oracle."""
    def expect(info):
        assert info["kernel"] == dg.GEMM_KERNEL_SINGLE_CTA, info
    replay_and_check("single_cta_ints", "f32", 3, 40, expect)


def test_stream_k_graph_replays_new_data():
    """A persistent plan with stream-K tiles (contributors publish partials with
    the launch's epoch) captured once and replayed five times on new inputs:
    every replay is bit-exact, so no replay consumed a stale partial."""
    def expect(info):
        assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT and info["stream_k_tiles"] > 0, info
    # 80 pair tiles of 256 x 256 on 76 clusters: every tile is split along K
    replay_and_check("square8192_bf16", "f32", 5, 60, expect,
                     flags=dg.GEMM_FLAG_CTA_GROUP_2 | dg.GEMM_FLAG_STAGE_K2, M=2048, N=2560, K=4096)


def test_few_tiles_split_graph_replays_new_data():
    """Fewer tiles than clusters: each finisher adds several clusters' partials,
    each waited for by its flag.  Five replays of one capture on new inputs,
    each bit-exact: no finisher took a previous replay's partial."""
    def expect(info):
        clusters = info["grid"] // info["cta_group"]
        assert info["kernel"] == dg.GEMM_KERNEL_PERSISTENT, info
        assert info["stream_k_tiles"] == info["num_tiles"] and clusters >= 4 * info["num_tiles"], info
    # 512 x 512 x 8192: 8 pair tiles of 256 x 128, each split four ways
    replay_and_check("square8192_bf16", "bf16", 5, 70, expect, M=512, N=512, K=8192)


def test_graph_replay_is_cheaper_than_a_call():
    """Replaying a captured small problem costs the host less than calling
    gemm_run through the binding (the launch-bound case graphs are for):
    host time to enqueue the same number of GEMMs, and device time per GEMM
    (which both paths must keep to a few microseconds)."""
    import time
    prob = inputs.make("single_cta")
    A, B = prob.A.cuda(), prob.B.cuda()
    D = torch.empty((128, 64), dtype=torch.float32, device="cuda")
    per_graph = 20
    with dg.Plan(dg.make_desc(128, 64, 64, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32)) as plan:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            plan.run(A, B, D)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(per_graph):
                plan.run(A, B, D)
        n = 20
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            g.replay()
        h_graph = (time.perf_counter() - t0) / (n * per_graph)
        torch.cuda.synchronize()
        t_graph = (time.perf_counter() - t0) / (n * per_graph)
        t0 = time.perf_counter()
        for _ in range(n * per_graph):
            plan.run(A, B, D)
        h_call = (time.perf_counter() - t0) / (n * per_graph)
        torch.cuda.synchronize()
        t_call = (time.perf_counter() - t0) / (n * per_graph)
        assert plan.sync_status()[0] == dg.GEMM_OK
    # host timings on a shared machine are reported, not asserted: they say
    # nothing about correctness and vary with whatever else the host runs
    print("per GEMM: graph replay %.2f us (host %.2f us), direct call %.2f us (host %.2f us)"
          % (t_graph * 1e6, h_graph * 1e6, t_call * 1e6, h_call * 1e6))
