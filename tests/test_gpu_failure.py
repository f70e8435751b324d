"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies must give up after its limit and come back as C3_ETIMEOUT, leaving
the CUDA context usable (a GEMM right after is still correct)."""
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
