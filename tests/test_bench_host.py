"""Host logic of bench.py on the CPU: the post-run validation's restated
definitions agree with the oracle and reject a planted error, the metric
arithmetic matches the oracle's closed forms, and the taxonomy, strict T_comm,
dispersion and workload lookup behave as documented."""
import math
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from concurrent_communication_overlap_gb300 import inputs as I  # noqa: E402


@pytest.mark.parametrize("name", ["tiny_ag", "tiny_a2a", "tiny_ar"])
def test_expected_collective_is_the_oracles(name):
    w = I.WORKLOADS[name]
    pay = I.coll_payload(w)
    got = bench.expected_collective(np, w, pay)
    if w.coll == "allgather":
        ref = oracle.allgather(pay)
    elif w.coll == "alltoall":
        ref = oracle.alltoall(pay, w.nranks)
    else:
        ref = oracle.allreduce(pay)[0].reshape(-1).view(np.uint8)
    assert np.array_equal(got, ref)


def test_gemm_rows_check_accepts_exact_rows_and_rejects_an_error():
    w = I.WORKLOADS["tiny_ag"]
    A, B = I.gemm_operands(w)
    rows = np.array([0, 1, 255, 511])
    C, S = oracle.gemm(A[rows], B)
    ref = bench.gemm_rows_reference(np, A, B, rows)
    assert bench.gemm_rows_ok(np, A, B, rows, C.astype(np.float32), ref)
    bad = C.astype(np.float32).copy()
    bad[2, 7] += 1e-2 * S[2, 7]              # one entry off by 100x the tolerance
    assert not bench.gemm_rows_ok(np, A, B, rows, bad, ref)
    nan = C.astype(np.float32).copy()
    nan[0, 0] = np.nan                        # an unwritten output
    assert not bench.gemm_rows_ok(np, A, B, rows, nan, ref)


@pytest.mark.parametrize("tg,tc,tconc", [(100.0, 42.0, 130.0), (2.0, 2.0, 2.0), (50.0, 80.0, 90.0),
                                         (7.0, 3.0, 10.0)])
def test_metric_arithmetic_matches_the_oracle(tg, tc, tconc):
    m = bench.pct_gain(tg, tc, tconc)
    o = oracle.c3_metrics(tg, tc, tconc)
    assert math.isclose(m["s_ideal"], o["s_ideal"], rel_tol=1e-12)
    assert math.isclose(m["s_real"], o["s_real"], rel_tol=1e-12)
    assert math.isclose(m["pct_ideal_gain"], 100.0 * o["pct_ideal_gain"], rel_tol=1e-12, abs_tol=1e-12)
    assert math.isclose(m["pct_ideal_ratio"], 100.0 * o["pct_ideal_ratio"], rel_tol=1e-12)
    assert bench.c3_class(tg, tc) == o["class"]


def test_taxonomy_thresholds():
    assert bench.c3_class(115.0, 100.0) == "G-long"
    assert bench.c3_class(114.9, 100.0) == "GC-equal"
    assert bench.c3_class(100.0, 115.0) == "C-long"
    assert bench.c3_class(100.0, 100.0) == "GC-equal"


def test_strict_comm_time_is_the_faster_engines_mean():
    modes = [("baseline", 1, 0, 0), ("ce", 2, 0, 0), ("ce_rp_8", 2, 8, 0)]
    per_mode = {"baseline": [{"t_comm_iso": t} for t in (5.0, 6.0, 10.0)],
                "ce": [{"t_comm_iso": t} for t in (6.5, 6.5)],
                "ce_rp_8": [{"t_comm_iso": t} for t in (6.5,)]}
    # SM engine: mean 7.0 (median 6.0); memcpy engine: mean 6.5 over both memcpy modes
    assert bench.strict_comm_time(per_mode, modes) == 6.5


def test_step_mean_resolves_below_the_clock_step():
    # times that snap to a 2.048 us clock: the mean recovers the true centre,
    # a median can only return a clock step
    tick = 2.048
    samples = [tick * 60] * 3 + [tick * 61] * 2
    assert bench.step_mean(samples) == pytest.approx(tick * 60.4)
    assert bench.step_mean(samples) not in samples


def test_spread_ignores_missing_values():
    s = bench.spread([3.0, None, float("nan"), 1.0, 2.0])
    assert s == {"mean": 2.0, "median": 2.0, "min": 1.0, "max": 3.0, "stdev": pytest.approx(math.sqrt(2.0 / 3.0)),
                 "n": 3}
    assert bench.spread([None]) is None


def test_workload_lookup():
    assert bench.find_workload(I, "mem_ag") is I.WORKLOADS["mem_ag"]
    w = bench.find_workload(I, "sweep_alltoall_4194304k")
    assert (w.M, w.N, w.K, w.coll, w.coll_bytes) == (8192, 8192, 8192, "alltoall", 4 << 30)
    with pytest.raises(SystemExit):
        bench.find_workload(I, "no_such_workload")


def _recs(tg, tconc):
    return [{"t_gemm_iso": a, "t_conc": b} for a, b in zip(tg, tconc)]


def test_share_ci_of_constant_steps_is_the_point_estimate():
    recs = _recs([100.0] * 10, [120.0] * 10)
    point = bench.pct_gain(100.0, 40.0, 120.0)["pct_ideal_gain"]
    lo, hi = bench.share_ci95(recs, 40.0)
    assert lo == pytest.approx(point) and hi == pytest.approx(point)
    assert bench.share_ci95(recs[:2], 40.0) is None


def test_share_ci_covers_the_estimate_and_narrows_with_more_steps():
    rng = np.random.default_rng(7)

    def draw(n):
        return _recs(100.0 + rng.normal(0, 1.0, n), 125.0 + rng.normal(0, 1.0, n))
    few, many = draw(20), draw(320)
    for recs in (few, many):
        tg = bench.step_mean([r["t_gemm_iso"] for r in recs])
        tconc = bench.step_mean([r["t_conc"] for r in recs])
        point = bench.pct_gain(tg, 42.0, tconc)["pct_ideal_gain"]
        lo, hi = bench.share_ci95(recs, 42.0)
        assert lo < point < hi
    w_few = bench.share_ci95(few, 42.0)
    w_many = bench.share_ci95(many, 42.0)
    assert (w_many[1] - w_many[0]) < 0.5 * (w_few[1] - w_few[0])      # ~1/sqrt(16) in theory
