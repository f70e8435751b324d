"""The pages' runtime heuristics (Section V-C) as host logic of libc3, checked
against hand-worked cases: schedule the lower-CTA-count kernel first; choose
the SM split minimising max(T_gemm * slowdown_gemm, T_comm * slowdown_comm)
with isolated times from a roofline at 70% efficiency."""
import pytest


@pytest.fixture(scope="module")
def c3():
    from concurrent_communication_overlap_gb300 import build
    build.build()
    from concurrent_communication_overlap_gb300 import c3 as mod
    return mod


def test_sp_rule(c3):
    assert c3.c3_sp_predict(152, 32) == 1     # collective has fewer CTAs: it goes first
    assert c3.c3_sp_predict(16, 152) == 0     # small GEMM goes first
    assert c3.c3_sp_predict(64, 64) == 0      # tie: the GEMM (baseline order)
    with pytest.raises(c3.C3Error):
        c3.c3_sp_predict(-1, 3)


def test_rp_memory_bound_worked_example(c3):
    # peak 1e15 flop/s, 1e12 B/s -> ridge 1000 flop/B.  GEMM 7e11 flop on 1e9 B:
    # 700 flop/B, memory-bound.  T_g = 1e9 / 0.7e12 = 1.428571e-3 s.
    # Collective 3.5e8 B: T_c = 2 * 3.5e8 / 0.7e12 = 1e-3 s.
    # k=8:  max(1.428571e-3 * 1.1, 1e-3 * 3.0) = 3.0e-3
    # k=32: max(1.428571e-3 * 1.4, 1e-3 * 1.2) = 2.0e-3   <- best
    table = [(8, 1.05, 1.1, 3.0), (32, 1.3, 1.4, 1.2)]
    best, t, each = c3.c3_rp_predict(table, 7e11, 1e9, 3.5e8, 1e15, 1e12)
    assert best == 32
    assert t == pytest.approx(2.0e-3, rel=1e-12)
    assert each == pytest.approx([3.0e-3, 2.0e-3], rel=1e-12)


def test_rp_compute_bound_uses_the_compute_column(c3):
    # 2e12 flop on 1e9 B: 2000 flop/B >= ridge 1000, compute-bound.
    # T_g = 2e12 / 0.7e15 = 2.857143e-3; T_c = 2 * 7e7 / 0.7e12 = 2e-4.
    # k=8:  max(2.857143e-3 * 1.05, 2e-4 * 3.0) = 3.0e-3     <- best
    # k=32: max(2.857143e-3 * 1.30, 2e-4 * 1.2) = 3.714286e-3
    # (with the memory column, 1.1 vs 1.4, the answer would be the same k but
    # other times: the times below pin which column was used)
    table = [(8, 1.05, 1.1, 3.0), (32, 1.3, 1.4, 1.2)]
    best, t, each = c3.c3_rp_predict(table, 2e12, 1e9, 7e7, 1e15, 1e12)
    assert best == 8
    assert each == pytest.approx([2e12 / 0.7e15 * 1.05, 2e12 / 0.7e15 * 1.3], rel=1e-12)


def test_rp_elastic_model_counts_the_widening_after_the_gemm(c3):
    # memory-bound GEMM as above: T_g = 1e9 / 0.7e12 = 1.428571e-3 s; T_c = 1e-3 s.
    # k=8:  a = T_g * 1.2 = 1.714286e-3, b = T_c * 4.0 = 4e-3.  Static: max = 4e-3.
    #       Elastic: by a the collective has moved a / b of its bytes, the rest at the
    #       every-SM rate: T_c + a * (1 - 1/4) = 1e-3 + 1.285714e-3 = 2.285714e-3   <- best
    # k=32: a = T_g * 2.0 = 2.857143e-3 >= b = T_c * 1.0: the GEMM's time in both models.
    table = [(8, 1.0, 1.2, 4.0), (32, 1.0, 2.0, 1.0)]
    best_s, _, each_s = c3.c3_rp_predict(table, 7e11, 1e9, 3.5e8, 1e15, 1e12)
    best_e, t_e, each_e = c3.c3_rp_predict(table, 7e11, 1e9, 3.5e8, 1e15, 1e12, elastic=True)
    t_g = 1e9 / 0.7e12
    assert best_s == 32 and each_s == pytest.approx([4e-3, 2.0 * t_g], rel=1e-12)
    assert best_e == 8 and t_e == pytest.approx(1e-3 + 1.2 * t_g * 0.75, rel=1e-12)
    assert each_e == pytest.approx([1e-3 + 1.2 * t_g * 0.75, 2.0 * t_g], rel=1e-12)
    with pytest.raises(c3.C3Error):
        c3.c3_rp_predict([(8, 1.0, 1.0, 0.0)], 1e12, 1e9, 1e8, 1e15, 1e12, elastic=True)


def test_rp_rejects_bad_tables(c3):
    with pytest.raises(c3.C3Error):
        c3.c3_rp_predict([], 1, 1, 1, 1, 1)
    with pytest.raises(c3.C3Error):
        c3.c3_rp_predict([(8, 0.0, 1.0, 1.0)], 1e12, 1e9, 1e8, 1e15, 1e12)
    with pytest.raises(c3.C3Error):
        c3.c3_rp_predict([(8, 1.0, 1.0, 1.0)], 1e12, 0.0, 1e8, 1e15, 1e12)


def _record():
    """The GB300 validation record committed with the profiles: slowdown table,
    peaks and, per scenario, the measured T_conc of each split and the split
    the heuristic predicted."""
    import json
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles", "heuristics_rp.md")
    text = open(path).read()
    return json.loads(re.search(r"```json\n(.*?)\n```", text, re.S).group(1))


def test_recorded_predictions_are_reproduced_from_the_committed_table(c3):
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from concurrent_communication_overlap_gb300 import inputs as I
    rec = _record()
    table = [(e["sms"], e["gemm_compute"], e["gemm_memory"], e["coll"]) for e in rec["table"]]
    pf, pb = rec["peaks"]["bf16_tflops"] * 1e12, rec["peaks"]["hbm_gbs"] * 1e9
    assert len(rec["rows"]) == rec["scenarios"] == 29
    hits = 0
    for row in rec["rows"]:
        w = bench.find_workload(I, row["scenario"])
        best_pred, _, _ = c3.c3_rp_predict(table, w.gemm_flops, w.gemm_bytes, w.coll_bytes, pf, pb)
        assert best_pred == row["predicted_sms"], row["scenario"]
        # recount the verdict from the measured times: the swept best, the loss, the 1.5% rule
        t = {int(k): v for k, v in row["t_conc_us"].items()}
        best = min(t, key=t.get)
        assert best == row["best_sms"], row["scenario"]
        loss = t[best_pred] / t[best] - 1.0
        assert loss == pytest.approx(row["loss_pct"] / 100.0, abs=1e-4)
        hit = best_pred == best or loss <= 0.015
        assert hit == row["hit"], row["scenario"]
        hits += hit
    assert hits == rec["hits"] == 23   # the pages' own bar: 24 of 30 (Section V-C)


def test_elastic_model_reproduces_the_recorded_predictions(c3):
    """The elastic model (partitions that dissolve when the GEMM ends) on the
    committed GB300 record: every recorded prediction is reproduced, and the
    verdicts recounted from the measured T_conc of each split give 25 of 29
    within 1.5% of the swept best, against 23 for the static model.  The misses
    are where the two kernels share HBM while both run (the 1-2 GiB crossovers
    and the memory-bound pair), which neither model captures."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from concurrent_communication_overlap_gb300 import inputs as I
    rec = _record()
    table = [(e["sms"], e["gemm_compute"], e["gemm_memory"], e["coll"]) for e in rec["table"]]
    pf, pb = rec["peaks"]["bf16_tflops"] * 1e12, rec["peaks"]["hbm_gbs"] * 1e9
    misses = []
    for row in rec["rows"]:
        w = bench.find_workload(I, row["scenario"])
        k, _, _ = c3.c3_rp_predict(table, w.gemm_flops, w.gemm_bytes, w.coll_bytes, pf, pb, elastic=True)
        assert k == row["predicted_sms_elastic"], row["scenario"]
        t = {int(a): v for a, v in row["t_conc_us"].items()}
        best = min(t, key=t.get)
        hit = k == best or t[k] / t[best] - 1.0 <= 0.015
        assert hit == row["hit_elastic"], row["scenario"]
        if not hit:
            misses.append(row["scenario"])
    assert len(rec["rows"]) - len(misses) == rec["hits_elastic"] == 25
    assert sorted(misses) == ["mem_ag", "sweep_allgather_1048576k", "sweep_allgather_2097152k",
                              "sweep_alltoall_2097152k"]
