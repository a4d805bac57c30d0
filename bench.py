#!/usr/bin/env python3
"""Benchmark: D = A @ B^T, M = N = K = 8192, bf16 inputs (TN), fp32 accumulation,
fp32 output, on one GB300 -- TFLOP/s and fraction of the measured dense bf16 peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-other-workloads]

One step = one gemm_run of the whole product (host planning of the tensor maps
+ one persistent kernel launch).  Inputs are seeded synthetic matrices (U[-1,1])
resident in HBM; the working set (A 134 MB + B 134 MB + D 268 MB) is larger than
the 129 MB L2, so no flush is inserted between steps.  With N > 1 (torchrun),
every rank runs its own replica of the product on its own GPU (no collective on
the data path); the elapsed time is the maximum over ranks.

After the headline, the same run times every other workload of the suite
(single-CTA example, 4096^3, batched 512 x 256^3, fp32-block-scaled e4m3,
MXFP8, MXFP4, NVFP4) with its own launches, CUDA events, clock samples and
roofline, reported under "other_workloads" on the same JSON line; then
torch.matmul (cuBLAS) on the 16-bit shapes, as context only
("library_context"), off this library's measured path.

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
# tcgen05.mma throughput per SM per cycle, measured on GB300 with a probe that
# issues M128 N256 MMAs back to back on every SM: 128 cycles per instruction
# for kind::f16 (K16), kind::f8f6f4 / mxf8f6f4 (K32) and kind::mxf4 /
# mxf4nvf4 (K64) alike.  (The 4-bit rate is 4x bf16, not the 6x of GB300's
# nominal dense figures; the roofline "peak" keeps the nominal ratio.)
MMA_FLOP_PER_CYCLE_SM = {"bf16": 8192.0, "fp8": 16384.0, "fp4": 32768.0}
# Files that decide what each kernel does: its code, its work schedule, the host
# code that plans and launches it.  A profile's DRAM figures count only while
# these hash to the value the profile records.
_SHARED = ["dense_gemm_blackwell_gb300/csrc/pipeline.cuh", "dense_gemm_blackwell_gb300/csrc/units.cuh",
           "dense_gemm_blackwell_gb300/csrc/ptx.cuh", "dense_gemm_blackwell_gb300/csrc/common.cuh",
           "dense_gemm_blackwell_gb300/csrc/launch.h", "dense_gemm_blackwell_gb300/csrc/gemm_api.cu",
           "include/gemm.h"]
SOURCES = {
    "persistent": ["dense_gemm_blackwell_gb300/csrc/kernels_persistent.cu"] + _SHARED,
    "single": ["dense_gemm_blackwell_gb300/csrc/kernels_single.cu"] + _SHARED,
    "fp8_block": ["dense_gemm_blackwell_gb300/csrc/kernels_fp8.cu"] + _SHARED,
    "mx": ["dense_gemm_blackwell_gb300/csrc/kernels_mx.cu", "dense_gemm_blackwell_gb300/csrc/mx_ptx.cuh"] + _SHARED,
}
KERNEL_SOURCES = SOURCES["persistent"]


def _prof(name):
    return os.path.join(ROOT, "profiles", name)


# Per-workload metric, roofline bound, peak (a multiple of the measured bf16
# peak: the nominal dtype ratio), kernel family and committed ncu summary.
WORKLOAD_INFO = {
    "square8192_bf16": dict(metric=METRIC, unit=UNIT, bound="tensor", peak_ratio=1.0, rate="bf16",
                            kernel="persistent", profile=_prof("persistent_pair_square8192_bf16_f32.md"),
                            text="D = A*B^T, M=N=K=8192, bf16 TN, fp32 accumulate, fp32 out"),
    "square4096_bf16": dict(metric="GEMM TFLOP/s (bf16 in, fp32 acc, bf16 out, 4096^3)", unit=UNIT,
                            bound="tensor", peak_ratio=1.0, rate="bf16", kernel="persistent",
                            profile=_prof("persistent_pair_square4096_bf16.md"),
                            text="D = A*B^T, M=N=K=4096, bf16 TN, fp32 accumulate, bf16 out"),
    "batched256_f16": dict(metric="batched GEMM GB/s (512 x 256^3, f16 in/out, fp32 acc)", unit="GB/s",
                           bound="hbm", peak_ratio=1.0, rate="bf16", kernel="persistent",
                           profile=_prof("persistent_batched256_f16.md"),
                           text="512 independent D = A*B^T of 256^3, f16 TN, fp32 accumulate, f16 out"),
    "fp8_block8192": dict(metric="GEMM TFLOP/s (e4m3 block-scaled in, fp32 acc, bf16 out, 8192^3)", unit=UNIT,
                          bound="tensor", peak_ratio=2.0, rate="fp8", kernel="fp8_block",
                          profile=_prof("fp8_block_square8192_e4m3_bf16.md"),
                          text="D = (qA sA)(qB sB)^T, 8192^3, e4m3 TN, fp32 scales 1x128 / 128x128, bf16 out"),
    "mxfp8_8192": dict(metric="GEMM TFLOP/s (MXFP8: e4m3 in, E8M0 per 32, fp32 acc, bf16 out, 8192^3)", unit=UNIT,
                       bound="tensor", peak_ratio=2.0, rate="fp8", kernel="mx",
                       profile=_prof("mx_pair_mxfp8_8192_bf16.md"),
                       text="D = (qA . sA)(qB . sB)^T, 8192^3, e4m3 TN, E8M0 scale per 32 K elements "
                            "(tcgen05 block scaling), bf16 out"),
    "mxfp4_8192": dict(metric="GEMM TFLOP/s (MXFP4: e2m1 in, E8M0 per 32, fp32 acc, bf16 out, 8192^3)", unit=UNIT,
                       bound="tensor", peak_ratio=6.0, rate="fp4", kernel="mx",
                       profile=_prof("mx_pair_mxfp4_8192_bf16.md"),
                       text="D = (qA . sA)(qB . sB)^T, 8192^3, e2m1 TN (packed), E8M0 scale per 32 K elements "
                            "(tcgen05 block scaling), bf16 out"),
    "nvfp4_8192": dict(metric="GEMM TFLOP/s (NVFP4: e2m1 in, E4M3 per 16 + fp32 per tensor, fp32 acc, bf16 out, "
                              "8192^3)", unit=UNIT, bound="tensor", peak_ratio=6.0, rate="fp4", kernel="mx",
                       profile=_prof("mx_pair_nvfp4_8192_bf16.md"),
                       text="D = tA tB (qA . sA)(qB . sB)^T, 8192^3, e2m1 TN (packed), E4M3 scale per 16 K elements "
                            "(tcgen05 block scaling), bf16 out"),
    "square8192_bf16_tile256": dict(
        metric="GEMM TFLOP/s (bf16 in, fp32 acc, 8192^3, cta_group::2 256x256 tiles)", unit=UNIT, bound="tensor",
        peak_ratio=1.0, rate="bf16", kernel="persistent", data="square8192_bf16",
        desc=dict(tile_n=256, flags=2),        # GEMM_FLAG_CTA_GROUP_2: the pair form with 256-wide tiles
        profile=_prof("persistent_pair_square8192_bf16_f32_tile256.md"),
        text="D = A*B^T, M=N=K=8192, bf16 TN, fp32 accumulate, fp32 out, persistent grid, cta_group::2 256x256 tiles"),
    "single_cta": dict(metric="single-CTA GEMM latency (128x64x64 f16 -> f32)", unit="us/launch",
                       bound="latency", peak_ratio=1.0, rate="bf16", kernel="single",
                       profile=_prof("single_cta_128x64x64_f16.md"),
                       text="Out = A @ B.T, A 128x64, B 64x64 f16, fp32 out, one CTA"),
}
# the other workloads timed after the headline, with launches per timed region
OTHER_WORKLOADS = [("square8192_bf16_tile256", 200), ("single_cta", 2000), ("square4096_bf16", 400), ("batched256_f16", 600),
                   ("fp8_block8192", 100), ("mxfp8_8192", 100), ("mxfp4_8192", 200), ("nvfp4_8192", 200)]


def kernel_source_hash(name: str = WORKLOAD) -> str:
    h = hashlib.sha256()
    for rel in SOURCES[WORKLOAD_INFO[name]["kernel"]]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(name: str = WORKLOAD):
    """DRAM bytes per launch from the workload's committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    try:
        text = open(WORKLOAD_INFO[name]["profile"]).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash(name):
        return None
    return float(m_tr.group(1))


def data_of(name: str) -> str:
    """The input workload (shapes, types, values) a bench entry runs on."""
    return WORKLOAD_INFO[name].get("data", name)


def config_for(name: str, world: int = 1) -> dict:
    """The `config` object of a workload's line (identical in both arms)."""
    from dense_gemm_blackwell_gb300 import inputs
    wl = inputs.WORKLOADS[data_of(name)]
    winfo = WORKLOAD_INFO[name]
    ws = working_set_bytes(name)
    return {"workload": "%s: %s" % (name, winfo["text"]), "M": wl.M, "N": wl.N, "K": wl.K, "batch": wl.batch,
            "inputs": "%s seed %d" % (wl.dist, wl.seed),
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": ("no flush: working set %.0f MB > 129 MB L2" % (ws / 1e6)) if ws > 129e6
            else "no flush: working set %.1f MB fits L2 (L2-warm)" % (ws / 1e6)}


def working_set_bytes(name: str) -> float:
    """Algorithmic bytes of one launch: A, B, D and any scales, once each."""
    from dense_gemm_blackwell_gb300 import inputs
    wl = inputs.WORKLOADS[data_of(name)]
    bits = {"f16": 16, "bf16": 16, "f32": 32, "e4m3": 8, "e5m2": 8, "e2m1": 4}
    total = (wl.M + wl.N) * wl.K * wl.batch * bits[wl.dtype_in] / 8 + wl.M * wl.N * wl.batch * bits[wl.dtype_out] / 8
    mode = wl.extra.get("scale_mode")
    if wl.block_scaled:
        total += 4 * (wl.M * -(-wl.K // 128) + -(-wl.N // 128) * -(-wl.K // 128))
    elif mode in ("mx", "nv"):
        v = 32 if mode == "mx" else 16
        kq = -(-(-(-wl.K // v)) // 4)
        total += 512 * kq * (-(-wl.M // 128) + -(-wl.N // 128)) + (8 if mode == "nv" else 0)
    return float(total)


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's `value` (a job takes as long as its slowest rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured HBM copy (MEASURED_PEAKS.json)"
    except Exception:
        return 6800.0, "fallback 6.8 TB/s"


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


def _oracle_rows(prob, rows, ncols=None):
    """The oracle on selected rows (and optionally the first ncols columns)."""
    import oracle
    wl = prob.wl
    N = wl.N if ncols is None else ncols
    B = prob.B if ncols is None else (prob.B[..., :N, :] if wl.batch == 1 else prob.B[:, :N, :]).contiguous()
    kw = dict(M=wl.M, N=N, K=wl.K, batch=wl.batch, dtype_a=wl.dtype_in, dtype_b=wl.extra.get("dtype_b", wl.dtype_in))
    if wl.extra.get("scale_mode") in ("mx", "nv"):
        # tiled scales: a row's scales sit where its row block puts them, whatever N is
        kw.update(scale_a=prob.scale_a, scale_b=prob.scale_b, scale_mode=wl.extra["scale_mode"],
                  tensor_scales=prob.tensor_scales)
    elif wl.block_scaled:
        sb = prob.scale_b.numpy()[: (N + 127) // 128]
        kw.update(scale_a=prob.scale_a.numpy(), scale_b=sb, ld_sb=prob.scale_b.shape[1])
    oracle.gemm_rows(prob.A, B, rows=rows, **kw)


def cpu_oracle_sample(seconds_target: float, prob=None, unit=UNIT):
    """Time the CPU oracle on a bounded row sample of the workload.  Returns
    (value in `unit`, cores, sample description, seconds)."""
    import oracle
    from dense_gemm_blackwell_gb300 import inputs
    if prob is None:
        prob = inputs.make(WORKLOAD)
    wl = prob.wl
    t = time.perf_counter()
    _oracle_rows(prob, list(range(2)))
    per_row = max((time.perf_counter() - t) / 2, 1e-5)
    rows = max(2, min(wl.M * wl.batch, int(seconds_target / per_row)))
    t = time.perf_counter()
    _oracle_rows(prob, list(range(rows)))
    dt = time.perf_counter() - t
    flops = 2.0 * rows * wl.N * wl.K
    desc = "%d of %d rows of D (all %d columns, K=%d) of %s, fp64 oracle" % (rows, wl.M * wl.batch, wl.N, wl.K, wl.name)
    if unit == "GB/s":
        frac = rows / float(wl.M * wl.batch)
        return working_set_bytes(wl.name) * frac / dt / 1e9, oracle.num_threads(), desc, dt
    if unit == "us/launch":
        return dt * 1e6 * (wl.M * wl.batch) / rows, oracle.num_threads(), desc, dt
    return flops / dt / 1e12, oracle.num_threads(), desc, dt


def run_reference(args):
    """The CPU oracle, as it stands, on this host's cores: each step is a bounded
    sample (rows, and if one row is too long for the budget, leading columns)
    of the workload; rank 0 only."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_gemm_blackwell_gb300 import inputs
    winfo = WORKLOAD_INFO[args.workload]
    prob = inputs.make(data_of(args.workload))
    wl = prob.wl
    t = time.perf_counter()
    _oracle_rows(prob, [0, 1])
    per_row = max((time.perf_counter() - t) / 2, 1e-5)
    budget = 150.0  # seconds for warm-up + timed steps together
    per_step = budget / max(args.steps + args.warmup, 1)
    rows = max(1, min(wl.M * wl.batch, int(per_step / per_row)))
    ncols = wl.N
    if per_row > per_step:
        ncols = max(16, min(wl.N, int(wl.N * per_step / per_row)))
    sample_rows = list(range(rows))
    for _ in range(args.warmup):
        _oracle_rows(prob, sample_rows, ncols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_rows(prob, sample_rows, ncols)
    dt = time.perf_counter() - t0
    frac = rows * ncols / float(wl.M * wl.batch * wl.N)
    work_s = dt / max(args.steps, 1) / frac          # seconds for the whole product at this rate
    if winfo["unit"] == "GB/s":
        value = working_set_bytes(args.workload) / work_s / 1e9
    elif winfo["unit"] == "us/launch":
        value = work_s * 1e6
    else:
        value = wl.flops / work_s / 1e12
    sample = "each step: %d of %d rows x %d of %d columns of D (K=%d), fp64 oracle" % (
        rows, wl.M * wl.batch, ncols, wl.N, wl.K)
    line = {
        "impl": "reference", "metric": winfo["metric"], "value": value, "unit": winfo["unit"],
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(args.steps, 1),
        "higher_is_better": winfo["unit"] != "us/launch", "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_for(args.workload, args.gpus),
        "cpu_baseline": {"value": value, "unit": winfo["unit"], "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": winfo["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def peaks_block(sm_count, sm_mhz):
    """The denominators side by side: measured cuBLAS bf16 burst and sustained
    peaks, the tcgen05 rate times SMs times the sampled and the maximum clock,
    and the datasheet's dense figure."""
    burst, sustained, kind = peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            max_mhz = float(json.load(f).get("sm_max_mhz") or 2070.0)
    except Exception:
        max_mhz = 2070.0
    return {"bf16_burst_measured": burst if kind == "measured" else None,
            "bf16_sustained_measured": sustained,
            "bf16_computed_at_sampled_clock": computed_peak("bf16", sm_count, sm_mhz),
            "bf16_computed_at_max_clock": computed_peak("bf16", sm_count, max_mhz),
            "bf16_datasheet_dense": 2250.0, "unit": "TFLOP/s",
            "computed_from": "%d SMs x %d flop/cycle/SM (kind::f16, measured) x SM clock" % (
                sm_count, MMA_FLOP_PER_CYCLE_SM["bf16"])}


def setup_workload(dg, torch, name):
    """Inputs of a workload on the GPU, its plan and a one-launch step function."""
    from dense_gemm_blackwell_gb300 import inputs
    prob = inputs.make(data_of(name))
    wl = prob.wl
    code = {"f16": dg.GEMM_F16, "bf16": dg.GEMM_BF16, "f32": dg.GEMM_F32, "e4m3": dg.GEMM_E4M3,
            "e5m2": dg.GEMM_E5M2, "e2m1": dg.GEMM_E2M1}
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    mode = wl.extra.get("scale_mode")
    if mode == "mx":
        smode = dg.GEMM_SCALE_MX_E8M0_32
    elif mode == "nv":
        smode = dg.GEMM_SCALE_NV_E4M3_16
    else:
        smode = dg.GEMM_SCALE_BLOCK_1x128_128x128 if wl.block_scaled else dg.GEMM_SCALE_NONE
    t = {"A": prob.A.cuda(), "B": prob.B.cuda(),
         "SA": prob.scale_a.cuda() if prob.scale_a is not None else None,
         "SB": prob.scale_b.cuda() if prob.scale_b is not None else None,
         "TS": torch.tensor(prob.tensor_scales, dtype=torch.float32, device="cuda") if mode == "nv" else None}
    dshape = (wl.batch, wl.M, wl.N) if wl.batch > 1 else (wl.M, wl.N)
    t["D"] = torch.empty(dshape, dtype=tdt[wl.dtype_out], device="cuda")
    desc = dg.make_desc(wl.M, wl.N, wl.K, batch=wl.batch, dtype_a=code[wl.dtype_in],
                        dtype_b=code[wl.extra.get("dtype_b", wl.dtype_in)], dtype_d=code[wl.dtype_out],
                        scale_mode=smode, **WORKLOAD_INFO[name].get("desc", {}))
    plan = dg.Plan(desc)
    sptr = torch.cuda.current_stream().cuda_stream
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    a, b, d, sa, sb, ts = (ptr(t[k]) for k in ("A", "B", "D", "SA", "SB", "TS"))
    handle = plan.handle
    if mode in ("mx", "nv"):
        def step():
            st = dg.gemm_run_mx(handle, a, b, d, sa, sb, ts, sptr)
            if st != dg.GEMM_OK:
                raise dg.GemmError(st, "gemm_run_mx")
    else:
        def step():
            st = dg.gemm_run(handle, a, b, d, sa, sb, sptr)
            if st != dg.GEMM_OK:
                raise dg.GemmError(st, "gemm_run")
    return {"prob": prob, "wl": wl, "t": t, "plan": plan, "info": plan.info.as_dict(), "step": step,
            "flops": float(wl.flops), "bytes": working_set_bytes(name)}


def computed_peak(rate: str, sm_count: int, mhz):
    """SMs x tcgen05 flop per cycle per SM x SM clock (TFLOP/s), or None."""
    if not mhz:
        return None
    return sm_count * MMA_FLOP_PER_CYCLE_SM[rate] * mhz * 1e6 / 1e12


def roofline_for(name, mean_launch_ms, sm_count, sm_mhz):
    winfo = WORKLOAD_INFO[name]
    from dense_gemm_blackwell_gb300 import inputs
    flops = float(inputs.WORKLOADS[data_of(name)].flops)
    nbytes = working_set_bytes(name)
    peak_bf16, peak_bf16_sustained, peak_kind = peaks()
    if winfo["bound"] == "hbm":
        hbm, kind = hbm_peak()
        achieved = nbytes / (mean_launch_ms / 1e3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
             "traffic": profiled_traffic(name), "peak_kind": kind}
    elif winfo["bound"] == "latency":
        r = {"bound": "latency", "achieved": mean_launch_ms * 1e3, "peak": None, "unit": "us/launch", "frac": None,
             "traffic": profiled_traffic(name),
             "note": "launch-latency bound (one CTA, 1 MFLOP): no throughput roofline applies"}
    else:
        peak = peak_bf16 * winfo["peak_ratio"]
        achieved = flops / (mean_launch_ms / 1e3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
             "traffic": profiled_traffic(name),
             "peak_kind": ("%s burst bf16 (MEASURED_PEAKS.json)%s" % (
                 peak_kind, "" if winfo["peak_ratio"] == 1 else " x %g (nominal %s/bf16 dense ratio of GB300)" % (
                     winfo["peak_ratio"], winfo["rate"]))) if peak_kind == "measured" else "fallback 1900 TFLOP/s bf16"}
        if peak_bf16_sustained:
            r["frac_of_sustained"] = achieved / (peak_bf16_sustained * winfo["peak_ratio"])
        comp = computed_peak(winfo["rate"], sm_count, sm_mhz)
        if comp:
            r["computed_peak"] = comp
            r["frac_of_computed"] = achieved / comp
    r["algorithmic_flops_per_launch"] = flops
    r["algorithmic_bytes_per_launch"] = nbytes
    return r


def metric_value(name, elapsed_ms, launches, world=1):
    winfo = WORKLOAD_INFO[name]
    from dense_gemm_blackwell_gb300 import inputs
    if winfo["unit"] == "GB/s":
        return working_set_bytes(name) * world * launches / (elapsed_ms / 1e3) / 1e9
    if winfo["unit"] == "us/launch":
        return elapsed_ms * 1e3 / launches
    return inputs.WORKLOADS[data_of(name)].flops * world * launches / (elapsed_ms / 1e3) / 1e12


def measure_other(dg, torch, name, sampler, sm_count, target_ms=200.0):
    """One other workload: warm-up, a timed region of back-to-back launches
    (about target_ms long), clocks sampled inside it, its roofline."""
    w = setup_workload(dg, torch, name)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        w["step"]()
    torch.cuda.synchronize()
    st, rec = w["plan"].sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "%s warm-up device status" % name)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(10):
        w["step"]()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = int(min(50000, max(20, target_ms / max(e0.elapsed_time(e1) / 10, 1e-3))))
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(launches):
        w["step"]()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    total_ms = e0.elapsed_time(e1)
    st, rec = w["plan"].sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "%s timed-region device status" % name)
    clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)
    info = w["info"]
    entry = {"metric": WORKLOAD_INFO[name]["metric"], "value": metric_value(name, total_ms, launches),
             "unit": WORKLOAD_INFO[name]["unit"], "launches": launches, "ms_per_launch": total_ms / launches,
             "dtype": w["wl"].dtype_in, "config": config_for(name),
             "plan": {k: info[k] for k in ("kernel", "cta_group", "tile_m", "tile_n", "tile_k", "stages",
                                            "tmem_stages", "grid", "num_tiles", "smem_bytes")},
             "roofline": roofline_for(name, total_ms / launches, sm_count, clocks.get("sm_mhz")),
             "clocks": clocks}
    w["plan"].close()
    del w
    torch.cuda.empty_cache()
    return entry


def library_context(torch, target_ms=100.0):
    """torch.matmul (a vendor library) on the 16-bit workloads' shapes, timed
    like the other workloads: context for the numbers above, not this
    library's path.  torch.matmul of bf16 / f16 operands returns bf16 / f16,
    so the 8192^3 entry has a 16-bit output where the headline writes fp32."""
    g = torch.Generator(device="cuda").manual_seed(9)
    out = {}
    for key, (batch, n, dt) in {"square8192_bf16_out_bf16": (1, 8192, torch.bfloat16),
                                "square4096_bf16": (1, 4096, torch.bfloat16),
                                "batched256_f16": (512, 256, torch.float16)}.items():
        shape = (batch, n, n) if batch > 1 else (n, n)
        A = torch.rand(shape, generator=g, device="cuda").to(dt)
        B = torch.rand(shape, generator=g, device="cuda").to(dt)
        step = lambda: torch.matmul(A, B.transpose(-1, -2))  # noqa: E731
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        launches = int(min(5000, max(10, target_ms / max(e0.elapsed_time(e1), 1e-3))))
        e0.record()
        for _ in range(launches):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / launches
        flop = 2.0 * batch * n ** 3
        byts = 3.0 * batch * n * n * A.element_size()
        out[key] = {"ms_per_launch": ms, "TFLOP/s": flop / ms / 1e9, "GB/s": byts / ms / 1e6, "launches": launches}
        del A, B
    torch.cuda.empty_cache()
    out["note"] = "torch.matmul (cuBLAS) on the same shapes; context only, off this library's measured path"
    return out


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

    winfo = WORKLOAD_INFO[args.workload]
    dg.build()
    w = setup_workload(dg, torch, args.workload)
    prob, wl, plan, info, step = w["prob"], w["wl"], w["plan"], w["info"], w["step"]
    A, B, D, SA, SB = (w["t"][k] for k in ("A", "B", "D", "SA", "SB"))
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    dshape = tuple(D.shape)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    flops = w["flops"]
    nbytes = lambda t: 0 if t is None else t.numel() * t.element_size()  # noqa: E731
    alg_bytes = w["bytes"]
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    sm_count = torch.cuda.get_device_properties(0).multi_processor_count

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "warm-up device status")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    # The timed region holds only the K launches (consecutive launches on the
    # stream overlap one kernel's set-up with the previous one's last CTAs,
    # which an event recorded between them would prevent); the kernel's
    # average launch duration is the region's time over K.  Per-launch
    # durations come from a separate, shorter pass afterwards (reported only).
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(args.steps):
        step()
    g1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t_wall1 = time.time()
    total_ms = g0.elapsed_time(g1)
    n_iso = min(args.steps, 50)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iso)]
    for i in range(n_iso):
        events[i][0].record(stream)
        step()
        events[i][1].record(stream)
    torch.cuda.synchronize()
    launch_ms = [a.elapsed_time(b) for a, b in events]
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "timed-region device status")

    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / args.steps

    value = metric_value(args.workload, total_ms, args.steps, world)
    # roofline of the dominant (only) kernel, from its own launch events
    mean_launch_ms = total_ms / args.steps
    roofline = roofline_for(args.workload, mean_launch_ms, sm_count, clocks.get("sm_mhz"))

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    hA = prob.A.pin_memory()
    hB = prob.B.pin_memory()
    hSA = prob.scale_a.pin_memory() if prob.scale_a is not None else None
    hSB = prob.scale_b.pin_memory() if prob.scale_b is not None else None
    hD = torch.empty(dshape, dtype=tdt[wl.dtype_out]).pin_memory()
    # 100 steps: host<->device copies on this platform now and then take
    # 5-20 ms instead of about 2 (plain cudaMemcpyAsync of pinned buffers too),
    # and a longer run keeps one such step from dominating the average
    e2e_steps = max(3, min(args.steps, 100))

    if wl.extra.get("scale_mode") in ("mx", "nv"):
        # gemm_run_host does not take tiled scales: copy in, gemm_run_mx, copy out
        dTS = w["t"]["TS"]

        def e2e_step():
            for dev, host in ((A, hA), (B, hB), (SA, hSA), (SB, hSB)):
                dev.copy_(host, non_blocking=True)
            s = dg.gemm_run_mx(plan.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), SA.data_ptr(), SB.data_ptr(),
                               ptr(dTS), sptr)
            if s != dg.GEMM_OK:
                raise dg.GemmError(s, "gemm_run_mx")
            hD.copy_(D, non_blocking=True)
    else:
        def e2e_step():
            s = dg.gemm_run_host(plan.handle, hA.data_ptr(), hB.data_ptr(), hD.data_ptr(), ptr(hSA), ptr(hSB),
                                 A.data_ptr(), B.data_ptr(), D.data_ptr(), ptr(SA), ptr(SB), sptr)
            if s != dg.GEMM_OK:
                raise dg.GemmError(s, "gemm_run_host")

    # warm-up: the first calls create the host pipeline's streams, events and
    # panel plans and encode their tensor maps
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_marks = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    e0.record(stream)
    e2e_marks[0].record(stream)
    for i in range(e2e_steps):
        e2e_step()
        e2e_marks[i + 1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_step_ms = [e2e_marks[i].elapsed_time(e2e_marks[i + 1]) for i in range(e2e_steps)]
    e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
    e2e_value = metric_value(args.workload, e2e_ms, e2e_steps, world)
    st, rec = plan.sync_status()
    if st != dg.GEMM_OK:
        raise dg.GemmError(st, "e2e device status")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, secs = cpu_oracle_sample(args.cpu_seconds, prob, winfo["unit"])
        cpu = {"value": v, "unit": winfo["unit"], "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}

    line = {
        "metric": winfo["metric"], "value": value, "unit": winfo["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": winfo["unit"] != "us/launch", "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype_in, "data": "synthetic",
        "config": config_for(args.workload, world),
        "plan": {k: info[k] for k in ("kernel", "cta_group", "tile_m", "tile_n", "tile_k", "stages",
                                       "tmem_stages", "grid", "num_tiles", "smem_bytes")},
        "roofline": roofline,
        "peaks": peaks_block(sm_count, clocks.get("sm_mhz")),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": winfo["unit"], "steps": e2e_steps,
                "h2d_bytes_per_step": int(nbytes(hA) + nbytes(hB) + nbytes(hSA) + nbytes(hSB)),
                "d2h_bytes_per_step": int(nbytes(hD)),
                "step_ms": {"min": min(e2e_step_ms), "median": statistics.median(e2e_step_ms),
                            "max": max(e2e_step_ms)}},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "launch_ms": {"mean_in_timed_region": mean_launch_ms,
                      "separate_pass": {"launches": len(launch_ms), "min": min(launch_ms), "max": max(launch_ms),
                                        "median": statistics.median(launch_ms)}},
    }
    if rank == 0 and world == 1 and args.workload == WORKLOAD and not args.no_other_workloads:
        # the rest of the suite, each with its own timed region, clocks and roofline
        plan.close()
        del w, A, B, D, SA, SB, hA, hB, hD, hSA, hSB
        torch.cuda.empty_cache()
        sampler = ClockSampler(local_rank)
        sampler.start()
        time.sleep(0.3)
        others = {}
        for name, _ in OTHER_WORKLOADS:
            others[name] = measure_other(dg, torch, name, sampler, sm_count)
        sampler.stop()
        line["other_workloads"] = others
        line["library_context"] = library_context(torch)
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
    ap.add_argument("--workload", choices=sorted(WORKLOAD_INFO), default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only --workload (profiling runs)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
