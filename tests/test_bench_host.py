"""Host-side pieces of bench.py (no GPU): the reference arm's JSON line, the
clock sampler's summary and the gate that ties the reported DRAM traffic to
the kernel sources it was measured on."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_line():
    """--impl reference times the CPU oracle and prints one JSON line with the
    keys the driver reads (small workload so that the test takes seconds)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "single_cta", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["impl"] == "reference" and j["steps"] == 3 and j["warmup"] == 3 and j["value"] > 0
    assert j["unit"] == "us/launch" and j["higher_is_better"] is False
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"] and j["cpu_baseline"]["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert j["config"]["workload"].startswith("single_cta")


def test_clock_summary():
    """Median SM clock and throttle reasons from nvidia-smi CSV lines taken
    inside the timed window; lines outside it are ignored."""
    cs = bench.ClockSampler(0)
    t = time.time()
    row = "0, {sm}, 2070, {pw}, 0x0, {hw}, Not Active, Not Active, {cap}"
    cs.lines = [
        (t - 10, row.format(sm=600, pw=100.0, hw="Active", cap="Not Active")),     # before the window
        (t + 1, row.format(sm=1650, pw=1380.5, hw="Not Active", cap="Active")),
        (t + 2, row.format(sm=1700, pw=1390.0, hw="Not Active", cap="Active")),
        (t + 3, row.format(sm=1600, pw=1370.0, hw="Not Active", cap="Not Active")),
        (t + 3.5, "garbled"),
    ]
    s = cs.summary(t, t + 5)
    assert s["sm_mhz"] == 1650 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1390.0
    s = cs.summary(t - 20, t + 5)
    assert "hw_slowdown" in s["reasons"]


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    """A committed summary's DRAM bytes count only while its recorded source
    hash matches the current sources of that workload's kernel."""
    name = bench.WORKLOAD
    fake = tmp_path / "profile.md"
    fake.write_text("kernel_source_sha256_16: %s\ndram_bytes_per_launch: 1.5e9\n" % bench.kernel_source_hash(name))
    info = dict(bench.WORKLOAD_INFO[name], profile=str(fake))
    monkeypatch.setitem(bench.WORKLOAD_INFO, name, info)
    assert bench.profiled_traffic(name) == 1.5e9
    fake.write_text("kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_launch: 1.5e9\n")
    assert bench.profiled_traffic(name) is None
    # each kernel family hashes its own sources
    assert bench.kernel_source_hash("mxfp8_8192") != bench.kernel_source_hash("fp8_block8192")
    assert bench.kernel_source_hash("square4096_bf16") == bench.kernel_source_hash(name)


def test_every_workload_has_a_profile_path_and_known_kernel():
    for name, info in bench.WORKLOAD_INFO.items():
        assert info["kernel"] in bench.SOURCES and info["profile"].startswith(os.path.join(ROOT, "profiles"))
        assert info["rate"] in bench.MMA_FLOP_PER_CYCLE_SM
    assert {n for n, _ in bench.OTHER_WORKLOADS} | {bench.WORKLOAD} == set(bench.WORKLOAD_INFO)


def test_algorithmic_bytes():
    MB = 1 << 20
    assert bench.working_set_bytes("square8192_bf16") == 512 * MB            # A, B bf16 + D fp32
    assert bench.working_set_bytes("batched256_f16") == 512 * 3 * 256 * 256 * 2
    # e4m3 A, B + bf16 D + fp32 scales [8192][64] and [64][64]
    assert bench.working_set_bytes("fp8_block8192") == 64 * MB * 2 + 128 * MB + 4 * (8192 * 64 + 64 * 64)
    # MXFP8: + 512-byte scale tiles, 64 row blocks x 64 K groups per operand
    assert bench.working_set_bytes("mxfp8_8192") == 64 * MB * 2 + 128 * MB + 2 * 512 * 64 * 64
    # NVFP4: 4-bit operands, E4M3 scales per 16 (128 K groups), two fp32 tensor scales
    assert bench.working_set_bytes("nvfp4_8192") == 32 * MB * 2 + 128 * MB + 2 * 512 * 64 * 128 + 8


def test_both_arms_share_the_config():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "single_cta", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    j = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][0])
    assert j["config"] == bench.config_for("single_cta", 1)
