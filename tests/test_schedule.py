"""Pipeline schedule model ("Hopper and Blackwell GEMM", section "Maths"):
the oracle's plain restatement pinned to the numbers the page prints, and the
library's C implementation (gemm_schedule_model) checked against it."""
import json
import math
import os
import random

import pytest

import dense_gemm_blackwell_gb300 as dg
from oracle.schedule import model

PAGE = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))["schedule_model"]
T, K, LOAD, MMA = PAGE["T"], PAGE["K"], PAGE["t_load"], PAGE["t_mma"]
# epilogue of the animation's defaults: the page's closed form 12 + 3*6*4 + t_epi = 92 gives t_epi = 8
EPI = PAGE["run_length_A2_A1"][0] - LOAD - T * K * MMA


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_busy_fraction_by_stage_count(stages):
    busy = model(T, K, stages, 2, 0.0, LOAD, MMA, EPI)["busy"]
    assert round(100 * busy) == PAGE["busy_percent_by_stages_A2"][str(stages)]


def test_accumulator_buffers_and_long_epilogue():
    assert [model(T, K, 4, a, 0.0, LOAD, MMA, EPI)["run"] for a in (2, 1)] == PAGE["run_length_A2_A1"]
    assert [model(T, K, 4, a, 0.0, LOAD, MMA, 30.0)["run"] for a in (2, 1)] == PAGE["run_length_epi30_A2_A1"]


def test_issue_time_does_not_change_the_defaults():
    for issue in (0.0, 1.0, 2.0):
        assert model(T, K, 4, 2, issue, LOAD, MMA, EPI)["run"] == 92


def test_closed_form_run_with_two_buffers():
    """A = 2 and t_epi <= K t_mma with enough stages: run = t_load + T K t_mma + t_epi."""
    rng = random.Random(3)
    for _ in range(200):
        t_mma = rng.randint(1, 8)
        k = rng.randint(1, 12)
        load = rng.randint(0, 30)
        s = math.ceil((load + t_mma) / t_mma)
        epi = rng.randint(0, k * t_mma)
        tiles = rng.randint(1, 6)
        assert model(tiles, k, s, 2, 0.0, load, t_mma, epi)["run"] == load + tiles * k * t_mma + epi


def test_steady_state_period():
    """Within a long tile, M_{g+S} - M_g = max(S t_mma, S t_issue, t_load + t_mma)."""
    rng = random.Random(4)
    for _ in range(200):
        s = rng.randint(1, 8)
        t_mma, issue, load = rng.randint(1, 9), rng.randint(0, 9), rng.randint(0, 60)
        r = model(1, 40 * s, s, 2, issue, load, t_mma, 0.0)
        g = 40 * s - 1 - s
        assert r["M"][g + s] - r["M"][g] == max(s * t_mma, s * issue, load + t_mma)


def test_stages_needed():
    assert math.ceil((LOAD + MMA) / MMA) == PAGE["stages_needed"]


def test_library_matches_oracle():
    rng = random.Random(5)
    for _ in range(300):
        args = (rng.randint(1, 5), rng.randint(1, 10), rng.randint(1, 8), rng.randint(1, 3),
                float(rng.randint(0, 3)), float(rng.randint(0, 40)), float(rng.randint(1, 9)),
                float(rng.randint(0, 40)))
        st, r = dg.gemm_schedule_model(*args)
        ref = model(*args)
        assert st == dg.GEMM_OK
        assert r.run_length == ref["run"] and r.tensor_busy == pytest.approx(ref["busy"], rel=1e-15)
    st, r = dg.gemm_schedule_model(T, K, 4, 2, 0.0, LOAD, MMA, EPI)
    assert r.stages_needed == PAGE["stages_needed"]
    st, r = dg.gemm_schedule_model(1, 64, 4, 2, 0.0, LOAD, MMA, 0.0)
    assert r.steady_period == max(4 * MMA, LOAD + MMA)
    assert dg.gemm_schedule_model(0, K, 4, 2, 0.0, LOAD, MMA, EPI)[0] == dg.GEMM_ERR_INVALID_ARG


def test_library_chooses_stages_and_buffers():
    """The page's defaults: two buffers and four stages reach the best run (92)."""
    st, s, a = dg.gemm_schedule_choose(T, K, 0.0, LOAD, MMA, EPI, 8, 2, 0.0)
    assert st == dg.GEMM_OK and (s, a) == (PAGE["stages_needed"], 2)


# ------------------------------------------------------------------ the model applied to this library's plans
#
# Kernel cycles of one 8192^3 bf16 -> bf16 launch measured on GB300 with three
# tile shapes (clock64 totals of an instrumented copy of the persistent
# kernel, recorded in profiles/persistent_pair_square8192_bf16_f32.md, "How
# the tile width was chosen").  The model's unit costs come from other
# measurements (a loads-only copy of the kernel, the MMA rate probe, the
# tcgen05.ld rate), so these are predictions, not fits.
GB300 = dict(sm_count=152, smem_optin_bytes=232448, cc_major=10, cc_minor=3)
MEASURED_8192 = [
    # (desc overrides, measured kernel cycles, planner's (S, A))
    (dict(), 914e3, (4, 1)),                                                      # 256x512, K = 64 stages
    (dict(tile_n=256, flags=dg.GEMM_FLAG_CTA_GROUP_2 | dg.GEMM_FLAG_STAGE_K1), 1111e3, (6, 2)),   # K = 64
    (dict(tile_n=256, flags=dg.GEMM_FLAG_CTA_GROUP_2), 967e3, (3, 2)),           # 256x256, K = 128 stages
]


@pytest.mark.parametrize("over,cycles,planned", MEASURED_8192)
def test_plan_schedule_predicts_measured_kernel_cycles(over, cycles, planned):
    props = dg.GemmDeviceProps(**GB300)
    desc = dg.make_desc(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, **over)
    st, info = dg.gemm_plan_query(desc, props)
    assert st == dg.GEMM_OK and (info.stages, info.tmem_stages) == planned
    st, p, r, s_model, a_model = dg.gemm_plan_schedule(desc, info, props)
    assert st == dg.GEMM_OK
    assert abs(r.run_length / cycles - 1) < 0.08, (r.run_length, cycles)
    # the library's parameters fed to the oracle's restatement give the same run
    ref = model(p.tiles, p.k_slices, p.stages, p.accumulators, p.t_issue, p.t_load, p.t_mma, p.t_epi)
    assert r.run_length == pytest.approx(ref["run"], rel=1e-12)
    # the planner keeps every stage the shared memory holds; the model's pick is
    # never deeper, and never asks for more accumulators than the tile allows
    assert s_model <= info.stages and a_model <= info.tmem_stages


def test_plan_schedule_finds_the_load_bound_shape():
    """Measured: only the 256x256 tile with one-atom (K = 64) stages leaves the
    tensor core waiting for operands (79.5 % of the ideal, against 96.7 and
    91.3 %).  The model puts exactly that shape's copy throughput per stage
    below its MMA time, and gives it the lowest busy fraction."""
    props = dg.GemmDeviceProps(**GB300)
    out = []
    for over, cycles, _ in MEASURED_8192:
        desc = dg.make_desc(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, **over)
        st, info = dg.gemm_plan_query(desc, props)
        st, p, r, _, _ = dg.gemm_plan_schedule(desc, info, props)
        out.append((p.t_issue > p.t_mma, r.tensor_busy))
    assert [o[0] for o in out] == [False, True, False]
    assert min(range(3), key=lambda i: out[i][1]) == 1


def test_plan_schedule_few_tiles_runs_one_share():
    """Fewer tiles than clusters: each cluster runs one K range of one tile,
    so the model runs a single tile of that range's K slices; a stream-K plan
    with ranges of a tile or more still counts whole tiles."""
    props = dg.GemmDeviceProps(**GB300)
    desc = dg.make_desc(512, 512, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16)
    st, info = dg.gemm_plan_query(desc, props)
    assert st == dg.GEMM_OK and 0 < info.stream_k_tiles == info.num_tiles < info.grid // info.cta_group
    st, p, r, _, _ = dg.gemm_plan_schedule(desc, info, props)
    assert st == dg.GEMM_OK
    k_slices = -(-8192 // info.tile_k)
    clusters = info.grid // info.cta_group
    assert p.tiles == 1 and p.k_slices == -(-info.num_tiles * k_slices // clusters) < k_slices
    desc = dg.make_desc(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, tile_n=256)
    st, info = dg.gemm_plan_query(desc, props)
    assert st == dg.GEMM_OK and info.stream_k_tiles >= info.grid // info.cta_group
    st, p, r, _, _ = dg.gemm_plan_schedule(desc, info, props)
    assert p.k_slices == -(-8192 // info.tile_k) and p.tiles == 14   # 1024 tiles over 76 pairs: 13.5 -> 14


def test_plan_schedule_rejects_what_it_does_not_model():
    props = dg.GemmDeviceProps(**GB300)
    desc = dg.make_desc(4096, 4096, 4096, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16,
                        scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    st, info = dg.gemm_plan_query(desc, props)
    assert st == dg.GEMM_OK
    assert dg.gemm_plan_schedule(desc, info, props)[0] == dg.GEMM_ERR_UNSUPPORTED
    bad = dg.gemm_machine_gb300()
    bad.ingest_bytes_per_cycle = 0.0
    desc = dg.make_desc(4096, 4096, 4096, dtype_a=dg.GEMM_BF16)
    st, info = dg.gemm_plan_query(desc, props)
    assert dg.gemm_plan_schedule(desc, info, props, bad)[0] == dg.GEMM_ERR_INVALID_ARG


# Ring-depth sweep of the 8192^3 bf16 -> bf16 plans on GB300 (medians of
# 10-launch groups, CUDA events): time relative to the planner's depth.
STAGE_SWEEP_512 = {4: 1.000, 3: 1.016, 2: 1.388}
STAGE_SWEEP_256_K128 = {3: 1.000, 2: 1.212}


def _run(over, stages):
    props = dg.GemmDeviceProps(**GB300)
    desc = dg.make_desc(8192, 8192, 8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16, stages=stages, **over)
    st, info = dg.gemm_plan_query(desc, props)
    assert st == dg.GEMM_OK
    return dg.gemm_plan_schedule(desc, info, props)[2].run_length


def test_model_reproduces_the_ring_depth_sweep():
    """512-wide tiles: three stages are as good as four (measured +1.6 %), two
    are far slower (measured +39 %); the model agrees on both, within 5 points."""
    base = _run({}, 4)
    for s, measured in STAGE_SWEEP_512.items():
        assert abs(_run({}, s) / base - measured) < 0.05, (s, _run({}, s) / base, measured)
    # 256-wide tiles with 128-deep stages: two stages are too few in both
    over = dict(tile_n=256, flags=dg.GEMM_FLAG_CTA_GROUP_2)
    assert _run(over, 2) / _run(over, 3) > 1 + (STAGE_SWEEP_256_K128[2] - 1) / 2
