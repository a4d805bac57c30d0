"""The N > 1 host path on CPU (gloo, world size 2): row and batch shards cover
the product exactly once with no data exchange, and the benchmark's
max-over-ranks timing reduction returns the slowest rank's time."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from dense_gemm_blackwell_gb300 import inputs
        from dense_gemm_blackwell_gb300.sharding import row_shard, batch_shard

        # rows of one product: each rank computes its own slab from the whole of B
        prob = inputs.make("square8192_bf16", M=600, N=96, K=64, dist="ints", seed=51)
        m0, m1 = row_shard(600, world, rank, align=256)
        part, _ = oracle.gemm(prob.A[m0:m1].contiguous(), prob.B, M=m1 - m0, N=96, K=64,
                              dtype_a="bf16", dtype_b="bf16")
        rows = [None] * world
        dist.all_gather_object(rows, (m0, m1, part[0]))          # test-side check only
        # batch entries of a batched product
        bp = inputs.make("batched256_f16", M=16, N=16, K=32, batch=5, dist="ints", seed=52)
        b0, b1 = batch_shard(5, world, rank)
        bpart, _ = oracle.gemm(bp.A[b0:b1].contiguous(), bp.B[b0:b1].contiguous(), M=16, N=16, K=32,
                               batch=b1 - b0, dtype_a="f16", dtype_b="f16")
        batches = [None] * world
        dist.all_gather_object(batches, (b0, b1, bpart))
        # slowest rank's time
        slowest = bench.max_over_ranks(1.5 if rank == 1 else 0.25, dist, "cpu")
        if rank == 0:
            full, _ = oracle.gemm(prob.A, prob.B, M=600, N=96, K=64, dtype_a="bf16", dtype_b="bf16")
            seen = np.zeros(600, int)
            for a, b, d in rows:
                seen[a:b] += 1
                assert np.array_equal(d, full[0][a:b])
            assert (seen == 1).all()
            bfull, _ = oracle.gemm(bp.A, bp.B, M=16, N=16, K=32, batch=5, dtype_a="f16", dtype_b="f16")
            bseen = np.zeros(5, int)
            for a, b, d in batches:
                bseen[a:b] += 1
                assert np.array_equal(d, bfull[a:b])
            assert (bseen == 1).all()
            assert slowest == 1.5
            out.put("ok")
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_and_timing_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert q.get(timeout=5) == "ok"


def test_shard_bounds():
    from dense_gemm_blackwell_gb300.sharding import row_shard, batch_shard
    for M in (1, 255, 256, 8192, 8193):
        for world in (1, 2, 3, 8):
            spans = [row_shard(M, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == M
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert all(s[0] % 256 == 0 for s in spans)
    assert [batch_shard(512, 8, r) for r in range(8)][3] == (192, 256)
    with pytest.raises(ValueError):
        row_shard(10, 2, 2)
