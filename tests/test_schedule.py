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
