#!/usr/bin/env python3
"""Benchmark: D = A @ B^T, M = N = K = 8192, bf16 inputs (TN), fp32 accumulation,
fp32 output, on one GB300 -- TFLOP/s and fraction of the measured dense bf16 peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one gemm_run of the whole product (host planning of the tensor maps
+ one persistent kernel launch).  Inputs are seeded synthetic matrices (U[-1,1])
resident in HBM; the working set (A 134 MB + B 134 MB + D 268 MB) is larger than
the 129 MB L2, so no flush is inserted between steps.  With N > 1 (torchrun),
every rank runs its own replica of the product on its own GPU (no collective on
the data path); the elapsed time is the maximum over ranks.

--impl reference times the CPU oracle (the plain fp64 triple loop) on this
host's cores on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "square8192_bf16"
METRIC = "GEMM TFLOP/s (bf16 in, fp32 acc, 8192^3) and fraction of GB300 dense peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE = os.path.join(ROOT, "profiles", "persistent_pair_square8192_bf16_f32.md")
KERNEL_SOURCES = ["dense_gemm_blackwell_gb300/csrc/kernels_persistent.cu",
                  "dense_gemm_blackwell_gb300/csrc/ptx.cuh",
                  "dense_gemm_blackwell_gb300/csrc/common.cuh"]


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)) or None, "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, None, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [p for ts, p in rows if t0 <= ts <= t1] or [p for _, p in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in inside:
            for name, val in zip(names, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        pw = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][2]), "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max(pw) if pw else None}


def cpu_oracle_sample(seconds_target: float, prob=None):
    """Time the CPU oracle on a bounded row sample of the workload.  Returns
    (tflops, cores, sample description, seconds)."""
    import oracle
    from dense_gemm_blackwell_gb300 import inputs
    if prob is None:
        prob = inputs.make(WORKLOAD)
    wl = prob.wl
    kw = dict(M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in, dtype_b=wl.dtype_in)
    t = time.perf_counter()
    oracle.gemm_rows(prob.A, prob.B, rows=list(range(2)), **kw)
    per_row = max((time.perf_counter() - t) / 2, 1e-4)
    rows = max(2, min(wl.M, int(seconds_target / per_row)))
    t = time.perf_counter()
    oracle.gemm_rows(prob.A, prob.B, rows=list(range(rows)), **kw)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * wl.N * wl.K
    desc = "%d of %d rows of D (all %d columns, K=%d) of %s, fp64 oracle" % (rows, wl.M, wl.N, wl.K, wl.name)
    return flops / dt / 1e12, oracle.num_threads(), desc, dt


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_gemm_blackwell_gb300 import inputs
    prob = inputs.make(WORKLOAD)
    wl = prob.wl
    kw = dict(M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in, dtype_b=wl.dtype_in)
    t = time.perf_counter()
    oracle.gemm_rows(prob.A, prob.B, rows=[0, 1], **kw)
    per_row = max((time.perf_counter() - t) / 2, 1e-4)
    budget = 150.0  # seconds for warmup + timed steps together
    rows = max(1, int(budget / max(args.steps + args.warmup, 1) / per_row))
    rows = min(rows, wl.M)
    for i in range(args.warmup):
        oracle.gemm_rows(prob.A, prob.B, rows=list(range(rows)), **kw)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm_rows(prob.A, prob.B, rows=list(range(rows)), **kw)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * wl.N * wl.K * args.steps
    value = flops / dt / 1e12
    sample = "each step: %d of %d rows of D (all %d columns, K=%d), fp64 oracle" % (rows, wl.M, wl.N, wl.K)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": wl.M, "N": wl.N, "K": wl.K, "inputs": "bf16 U[-1,1] seed %d" % wl.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import dense_gemm_blackwell_gb300 as dg
    from dense_gemm_blackwell_gb300 import inputs

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    prob = inputs.make(WORKLOAD)
    wl = prob.wl
    dg.build()
    A = prob.A.cuda()
    B = prob.B.cuda()
    D = torch.empty(wl.M, wl.N, dtype=torch.float32, device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    plan = dg.Plan(desc)
    info = plan.info.as_dict()
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    flops = float(wl.flops)

    def step():
        s = dg.gemm_run(plan.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), None, None, sptr)
        if s != dg.GEMM_OK:
            raise dg.GemmError(s, "gemm_run")

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "warm-up device status")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(args.steps):
        events[i][0].record(stream)
        step()
        events[i][1].record(stream)
    g1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t_wall1 = time.time()
    total_ms = g0.elapsed_time(g1)
    launch_ms = [a.elapsed_time(b) for a, b in events]
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "timed-region device status")

    if dist is not None:
        t = torch.tensor([total_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = flops * world * args.steps / (total_ms / 1e3) / 1e12

    # roofline of the dominant (only) kernel
    peak, peak_sustained, peak_kind = peaks()
    mean_launch_ms = sum(launch_ms) / len(launch_ms)
    achieved = flops / (mean_launch_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(),
                "peak_kind": "%s burst bf16 (MEASURED_PEAKS.json)" % peak_kind if peak_kind == "measured"
                else "fallback 1900 TFLOP/s bf16",
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": float(wl.M * wl.K * 2 + wl.N * wl.K * 2 + wl.M * wl.N * 4)}
    if peak_sustained:
        roofline["frac_of_sustained"] = achieved / peak_sustained

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    hA = prob.A.pin_memory()
    hB = prob.B.pin_memory()
    hD = torch.empty(wl.M, wl.N, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        s = dg.gemm_run_host(plan.handle, hA.data_ptr(), hB.data_ptr(), hD.data_ptr(), None, None,
                             A.data_ptr(), B.data_ptr(), D.data_ptr(), None, None, sptr)
        if s != dg.GEMM_OK:
            raise dg.GemmError(s, "gemm_run_host")

    e2e_step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if dist is not None:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = flops * world * e2e_steps / (e2e_ms / 1e3) / 1e12
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "e2e device status")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, secs = cpu_oracle_sample(args.cpu_seconds, prob)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s: D = A*B^T, M=N=K=8192, bf16 TN, fp32 accumulate, fp32 out" % WORKLOAD,
                   "M": wl.M, "N": wl.N, "K": wl.K, "inputs": "U[-1,1] seed %d" % wl.seed,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "no flush: working set 537 MB > 129 MB L2",
                   "plan": {k: info[k] for k in ("kernel", "cta_group", "tile_m", "tile_n", "tile_k", "stages",
                                                  "tmem_stages", "grid", "num_tiles", "smem_bytes")}},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "steps": e2e_steps,
                "h2d_bytes_per_step": int(hA.numel() * hA.element_size() + hB.numel() * hB.element_size()),
                "d2h_bytes_per_step": int(hD.numel() * hD.element_size())},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "launch_ms": {"mean": mean_launch_ms, "min": min(launch_ms), "max": max(launch_ms),
                      "median": statistics.median(launch_ms)},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
