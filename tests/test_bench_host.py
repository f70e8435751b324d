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


def _synthetic_detail(n_modes=12, long_strings=False):
    """A detail record shaped like the bench's, with every optional part."""
    pad = "x" * (4000 if long_strings else 10)
    modes = {f"mode_{i:02d}_{pad[:20]}": {"pct_ideal_gain": 12.3456789 + i, "other": list(range(50))}
             for i in range(n_modes)}
    return {
        "detail": "c3", "metric": bench.METRIC, "value": 19.87654321, "unit": bench.UNIT, "n_gpus": 1,
        "steps": 20, "warmup": 5, "ms_per_step": 312.123456789, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "l405_a2a", "description": pad, "M": 8192, "N": 53248, "K": 16384,
                   "collective": "alltoall 8 ranks x 8388608 B", "l2": pad, "parallelism": "single GPU",
                   "coll_l2": "normal", "ce_variant": "graph", "coll_src": "device", "modes": list(modes)},
        "best_mode": "baseline", "value_ci95": [10.123456, 29.987654], "class": "G-long",
        "gemm_bound": "compute", "coll_bound": "bandwidth",
        "gemm_tflops_overlap": 1650.123456, "copy_gbs_overlap": 3100.98765,
        "roofline": {"bound": "tensor", "achieved": 1650.1, "peak": 1706.7, "unit": "TFLOP/s", "frac": 0.96681,
                     "frac_of_burst": 0.9, "traffic": 1.2345678e10, "algorithmic_per_launch": 1.4293e13,
                     "kernel": "gemm_bf16_kernel (tcgen05)", "peak_source": "measured bf16, sustained " + pad[:40]},
        "roofline_copy": {"bound": "hbm", "achieved": 5900.0, "peak": 6781.4, "unit": "GB/s", "frac": 0.87,
                          "kernel": "copy_vec_kernel (default budget)", "regime": pad},
        "gpu_launches": 123456,
        "validation": {"collective_bit_exact": True, "gemm_rows_in_tolerance": True,
                       "per_mode": {k: {"collective_bit_exact": True} for k in modes}, "gemm_rows": [0, 1, 2, 3]},
        "modes": modes, "device": {"name": "NVIDIA GB300", "sm_count": 152},
        "clocks": {"sm_mhz": 1455.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 300},
        "aux": {"gemm": {f"s{i}": {"us": 1.0 * i} for i in range(100)}},
        "e2e": {"value": 55.5, "unit": bench.UNIT, "h2d_bytes_per_step": 826277888, "d2h_bytes_per_step": 146800640,
                "engine": "memcpy", "mode": "baseline", "variants": {f"v{i}": pad for i in range(8)}},
        "cpu_baseline": {"value": 3.25, "unit": bench.UNIT, "cores": 16, "kind": "oracle",
                         "sample": "28 of 8192 rows of A against all 53248x16384 of B " + pad[:200]},
    }


@pytest.mark.parametrize("n_modes,long_strings", [(8, False), (12, False), (40, True)])
def test_headline_line_is_compact_and_parses(n_modes, long_strings):
    import json
    line = bench.headline_line(_synthetic_detail(n_modes, long_strings))
    text = json.dumps(line)
    assert len(text) <= bench.HEADLINE_MAX_BYTES
    back = json.loads(text)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "dtype", "config", "best_mode", "value_ci95", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                "validation"):
        assert key in back, key
    assert back["config"]["workload"] == "l405_a2a"
    assert back["roofline"]["frac"] == pytest.approx(0.96681)
    assert back["e2e"]["h2d_bytes_per_step"] == 826277888
    assert set(back["validation"]) == {"collective_bit_exact", "gemm_rows_in_tolerance"}
    assert "modes" not in back and "aux" not in back and "detail" not in back


def test_headline_line_keeps_every_mode_share_when_it_fits():
    import json
    d = _synthetic_detail(8)
    line = bench.headline_line(d)
    assert set(line["modes_pct"]) == set(d["modes"])
    assert len(json.dumps(line)) <= bench.HEADLINE_MAX_BYTES
    assert line["value"] == pytest.approx(19.877, rel=1e-4)       # 5 significant digits


def test_headline_of_the_default_run_keeps_every_mode_share():
    """The default run's own shape: the 405B-shaped pair's nine modes, the full
    clock record, the real peak-source and CPU-sample wordings; every mode's
    share stays in the line, under the cap."""
    import json
    d = _synthetic_detail(0)
    names = [m[0] for m in bench.select_modes("l405_a2a")]
    d["modes"] = {n: {"pct_ideal_gain": -123.456789 + i} for i, n in enumerate(names)}
    d["config"] = {"workload": "l405_a2a", "M": 8192, "N": 53248, "K": 16384,
                   "collective": "alltoall 8 ranks x 8388608 B", "coll_src": "device",
                   "l2": "flushed before every timed phase (2 x L2 zero-fill)", "parallelism": "single GPU"}
    d["settle_us"] = 18828
    d["roofline"]["peak_source"] = "measured bf16 burst (phases start after 18828 us idle)"
    d["clocks"] = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 315, "sm_mhz_p10": 2070.0,
                   "sm_mhz_min": 2070.0, "power_w_max": 556.97,
                   "basis": "nvidia-smi every 200 ms over the timed region (settle periods included)"}
    d["cpu_baseline"]["sample"] = ("8/8192 rows of A x all of B (fp64, 15 threads); 0.0010 of the collective "
                                   "(1 thread); isolated, then concurrent")
    line = bench.headline_line(d)
    assert set(line["modes_pct"]) == set(names) and len(names) == 9
    assert "basis" not in line["clocks"] and line["clocks"]["power_w_max"] == pytest.approx(556.97)
    assert len(json.dumps(line)) <= bench.HEADLINE_MAX_BYTES


def test_default_modes_of_the_405b_pair_and_explicit_subsets():
    names = [m[0] for m in bench.select_modes("l405_a2a")]
    for n in ("baseline", "prioritised", "partitioned_8", "partitioned_16", "partitioned_32", "ce", "ce_rp_8",
              "ce_staged"):
        assert n in names
    assert [m[0] for m in bench.select_modes("mem_ag")] == [m[0] for m in bench.MODES]
    assert [m[0] for m in bench.select_modes("l405_a2a", "ce,baseline")] == ["baseline", "ce"]
    with pytest.raises(SystemExit):
        bench.select_modes("mem_ag", "no_such_mode")


def test_gemm_rows_reference_in_chunks_equals_one_pass():
    w = I.WORKLOADS["tiny_ag"]
    A, B = I.gemm_operands(w)
    rows = np.array([3, 100, 511])
    ref1, b1 = bench.gemm_rows_reference(np, A, B, rows, chunk=1 << 20)
    ref2, b2 = bench.gemm_rows_reference(np, A, B, rows, chunk=97)      # ragged last chunk
    # the same fp64 dot products; a BLAS may block K differently per shape, so allow its last bits
    assert np.allclose(ref1, ref2, rtol=1e-12, atol=1e-12) and np.allclose(b1, b2, rtol=1e-12, atol=0)


def test_settle_period_follows_the_gemm_time_within_its_clamp():
    assert bench.auto_settle_us(7.4e-3) == 18500           # 2.5 x 7.4 ms
    assert bench.auto_settle_us(1.0) == 20000              # clamped to 20 ms
    assert bench.auto_settle_us(10e-6) == 200              # clamped to 0.2 ms
    assert bench.auto_settle_us(7.4e-3, settle_ms=0) == 0  # explicit values win
    assert bench.auto_settle_us(7.4e-3, settle_ms=3.5) == 3500


def test_pooled_gemm_time_is_the_per_step_mean_over_modes():
    per_mode = {"a": [{"t_gemm_iso": 1.0}, {"t_gemm_iso": 3.0}],
                "b": [{"t_gemm_iso": 2.0}, {"t_gemm_iso": 5.0}, {"t_gemm_iso": 9.0}]}
    assert bench.pooled_gemm_times(per_mode) == [1.5, 4.0]   # steps both modes completed


def test_share_ci_uses_the_pooled_gemm_times_when_given():
    recs = _recs([100.0] * 10, [120.0] * 10)
    lo, hi = bench.share_ci95(recs, 40.0, tg_steps=[110.0] * 10)
    point = bench.pct_gain(110.0, 40.0, 120.0)["pct_ideal_gain"]
    assert lo == pytest.approx(point) and hi == pytest.approx(point)


def test_collective_bound_of_the_strict_engine():
    modes = [("baseline", 1, 0, 0), ("ce", 2, 0, 0)]
    per_mode = {"baseline": [{"t_comm_iso": 2.0}], "ce": [{"t_comm_iso": 4.0}]}
    # SM engine is faster (2 s for 1 byte = 0.5 B/s); against its plateau of 1 B/s that is exactly half
    assert bench.coll_bound_strict(per_mode, modes, {"sm": 1.0, "ce": 100.0}, 1) == "bandwidth"
    assert bench.coll_bound_strict(per_mode, modes, {"sm": 1.01, "ce": 0.1}, 1) == "latency"
    assert bench.coll_bound_strict(per_mode, modes, {}, 1) == "unknown"
    assert bench.most_common(["a", "b", "b"]) == "b" and bench.most_common([]) is None


def test_default_step_count_fits_about_a_minute_of_timed_work():
    # the 8192x53248x16384 pair with its settle periods: ~0.8 s a step
    assert bench.auto_steps(0.8) == 75
    assert bench.auto_steps(0.8) * 0.8 <= bench.STEP_BUDGET_S
    # short steps: capped, long steps: never below the floor
    assert bench.auto_steps(0.01) == bench.AUTO_STEPS_MAX
    assert bench.auto_steps(30.0) == bench.AUTO_STEPS_MIN
    assert bench.auto_steps(0.0) == bench.AUTO_STEPS_MAX
    assert bench.parse_args([]).steps is None
    assert bench.parse_args(["--steps", "7"]).steps == 7


def test_host_staged_mode_is_an_engine_of_its_own():
    assert bench.mode_engine("ce_staged", 2) == "ce_staged"
    assert bench.mode_engine("ce", 2) == "ce" and bench.mode_engine("ce_rp_8", 2) == "ce"
    assert bench.mode_engine("baseline", 1) == "sm" and bench.mode_engine("reclaim_16", 4) == "sm"
    # the strict T_comm is the fastest engine's mean: the staged DMA path's slow isolated time
    # neither sets it nor blends into the driver memcpy's mean
    modes = [("baseline", 1, 0, 0), ("ce", 2, 0, 0), ("ce_staged", 2, 0, 0)]
    per_mode = {"baseline": [{"t_comm_iso": 2e-4}, {"t_comm_iso": 2e-4}],
                "ce": [{"t_comm_iso": 3e-4}],
                "ce_staged": [{"t_comm_iso": 3.8e-3}]}
    assert bench.strict_comm_time(per_mode, modes) == pytest.approx(2e-4)
    per_mode["baseline"] = [{"t_comm_iso": 5e-4}]
    assert bench.strict_comm_time(per_mode, modes) == pytest.approx(3e-4)
    assert bench.coll_bound_strict(per_mode, modes, {"ce": 1e12}, 1e8) == "latency"
