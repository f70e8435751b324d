"""Failure detection without a GPU fault.

A bounded device wait that nothing satisfies must give up after its limit and
come back as C3_ETIMEOUT, leaving the CUDA context usable (a GEMM right after
is still correct).  Failures injected on the host (c3_inject_fault: a GEMM
launch, an SM collective launch, a memcpy transfer, the device
initialisation) must come back as C3_ECUDA, alone or inside a concurrent run,
and the next call must work and be exact."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    from concurrent_communication_overlap_gb300 import c3
    assert c3.c3_selftest_wait(1_000_000, 1) == c3.C3_OK          # satisfied wait
    t0 = time.perf_counter()
    assert c3.c3_selftest_wait(1_000_000, 0) == c3.C3_ETIMEOUT    # 1 ms, never satisfied
    assert time.perf_counter() - t0 < 5.0
    assert "site" in c3.c3_last_error()
    assert c3.c3_selftest_wait(200_000_000, 0) == c3.C3_ETIMEOUT  # 200 ms
    # the context is intact and the status block clean: a GEMM runs and checks out
    M, N, K = 256, 192, 128
    A = I.bf16_uniform(1, (M, K))
    B = I.bf16_uniform(2, (N, K))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    c3.c3_gemm(dA, dB, dC, M, N, K)
    assert c3.c3_status_check() == c3.C3_OK
    C_ref, S_ref = oracle.gemm(A, B)
    assert (np.abs(dC.cpu().numpy() - C_ref) <= 1e-4 * S_ref).all()


# ---------------------------------------------------------------- host-injected failures

def _gemm_case(c3):
    M, N, K = 300, 200, 136
    A = I.bf16_uniform(11, (M, K))
    B = I.bf16_uniform(12, (N, K))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    C_ref, S_ref = oracle.gemm(A, B)

    def ok():
        return bool((np.abs(dC.cpu().numpy().astype(np.float64) - C_ref) <= 1e-4 * S_ref).all())
    return (M, N, K), dA, dB, dC, ok


def _ag_case(c3):
    sb = 64 * 1024 + 16
    shards = [I.random_bytes(1002 + r, sb) for r in range(8)]
    ds = [torch.from_numpy(x).cuda() for x in shards]
    out = torch.zeros(8 * sb, dtype=torch.uint8, device="cuda")
    ref = oracle.allgather(shards)
    return sb, ds, out, lambda: np.array_equal(out.cpu().numpy(), ref)


def test_injected_gemm_launch_failure_is_reported_and_recovers():
    from concurrent_communication_overlap_gb300 import c3
    (M, N, K), dA, dB, dC, ok = _gemm_case(c3)
    c3.c3_inject_fault(c3.C3_FAULT_GEMM_LAUNCH)
    assert c3.c3_gemm(dA, dB, dC, M, N, K, check=False) == c3.C3_ECUDA
    assert "injected" in c3.c3_last_error()
    assert torch.isnan(dC).all()                                 # nothing was launched
    c3.c3_gemm(dA, dB, dC, M, N, K)                              # the next call works
    assert c3.c3_status_check() == c3.C3_OK and ok()


@pytest.mark.parametrize("engine,site", [(0, 2), (1, 3)])
def test_injected_collective_failure_is_reported_and_recovers(engine, site):
    from concurrent_communication_overlap_gb300 import c3
    sb, ds, out, ok = _ag_case(c3)
    c3.c3_inject_fault(site)
    assert c3.c3_allgather(ds, out, sb, 8, engine=engine, check=False) == c3.C3_ECUDA
    assert "injected" in c3.c3_last_error()
    c3.c3_allgather(ds, out, sb, 8, engine=engine)
    assert c3.c3_status_check() == c3.C3_OK and ok()


@pytest.mark.parametrize("mode,site,priority", [(1, 2, 0), (1, 1, 0), (2, 3, 0), (4, 2, 0), (1, 1, 1), (4, 1, 0)])
def test_injected_failure_inside_a_concurrent_run(mode, site, priority):
    # one half of the pair fails after (or before) the other was launched: the
    # run reports C3_ECUDA, and the next run of the same problem is exact
    import ctypes
    from concurrent_communication_overlap_gb300 import c3
    (M, N, K), dA, dB, dC, gemm_ok = _gemm_case(c3)
    sb, ds, out, coll_ok = _ag_case(c3)
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLGATHER, out, sb, 8, shards=ds)
    split = 16 if mode == 4 else 0
    c3.c3_inject_fault(site)
    t = c3.C3Timing()
    assert c3.lib().c3_run(ctypes.byref(p.rec), mode, split, priority, ctypes.byref(t)) == c3.C3_ECUDA
    assert "injected" in c3.c3_last_error()
    if site == c3.C3_FAULT_GEMM_LAUNCH and (priority or mode == 4):
        # the collective went out before the GEMM's launch failed: it completes,
        # ordered before the caller's own stream
        torch.cuda.current_stream().synchronize()
        assert coll_ok() and torch.isnan(dC).all()
    torch.cuda.synchronize()
    dC.fill_(float("nan"))
    out.zero_()
    r = c3.c3_run(p, mode, split, 0)
    assert r["status"] == 0 and gemm_ok() and coll_ok()
    # every collective work counter is clean: a run whose second launch part
    # never went out had its counter cleared, so the slots (64, round robin)
    # serve later launches correctly
    for i in range(70):
        out.zero_()
        c3.c3_allgather(ds, out, sb, 8, engine=c3.C3_ENGINE_SM, sm_budget=1 + i % 5)
        assert coll_ok(), i


def test_injected_device_init_failure_and_reinit():
    import ctypes
    from concurrent_communication_overlap_gb300 import c3
    torch.cuda.synchronize()
    c3.c3_shutdown()
    c3.c3_inject_fault(c3.C3_FAULT_DEVICE_INIT)
    info = c3.C3DeviceInfo()
    assert c3.lib().c3_get_device_info(ctypes.byref(info)) == c3.C3_ECUDA
    assert "injected" in c3.c3_last_error()
    assert c3.c3_get_device_info()["sm_count"] > 0             # initialises on the next call
    (M, N, K), dA, dB, dC, ok = _gemm_case(c3)
    c3.c3_gemm(dA, dB, dC, M, N, K)
    assert c3.c3_status_check() == c3.C3_OK and ok()
