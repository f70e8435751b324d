"""c3_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(code running under a host framework that owns a fixed memory pool, a plugin
invoked while its caller holds the whole device, real-time code that may not
enter the allocator).  Its scratch lives in a static device array inside
libc3.so, so it must give the same C as c3_gemm, call after call, without the
library's per-device state.  This file is collected last on purpose: if it
fails, a run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 1e-4  # the GEMM tolerance of every other test: |err| <= 1e-4 * sum_k |a*b|


def test_noalloc_gemm_matches_c3_gemm_two_calls_in_a_row():
    from concurrent_communication_overlap_gb300 import c3
    shapes = [(512, 768, 512, 0), (300, 200, 264, 5)]   # second call: ragged edges, capped grid
    for call, (M, N, K, budget) in enumerate(shapes):
        A = I.bf16_uniform(2000 + call, (M, K), -1.0, 1.0)
        B = I.bf16_uniform(3000 + call, (N, K), -1.0, 1.0)
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B.view(np.int16)).cuda()
        c_noalloc = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        c_ref = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        # the allocation-free entry point first: in a fresh process this is its first call
        assert c3.c3_gemm_noalloc(dA, dB, c_noalloc, M, N, K, budget, sync_check=True, check=False) == c3.C3_OK, \
            c3.c3_last_error()
        c3.c3_gemm(dA, dB, c_ref, M, N, K, budget)
        c3.c3_status_check()
        got = c_noalloc.cpu().numpy().astype(np.float64)
        ref = c_ref.cpu().numpy().astype(np.float64)
        _, S = oracle.gemm(A, B)
        assert not np.isnan(got).any()
        assert (np.abs(got - ref) <= TOL * S).all(), call


def test_noalloc_rejects_bad_arguments_without_launching():
    from concurrent_communication_overlap_gb300 import c3
    before = c3.c3_kernel_launches()
    assert c3.c3_gemm_noalloc(0x1000, 0x1000, 0x1000, -1, 4, 8, check=False) == c3.C3_EINVAL
    assert c3.c3_gemm_noalloc(0x1000, 0x1000, 0x1000, 4, 4, 12, check=False) == c3.C3_EALIGN
    assert c3.c3_gemm_noalloc(0x1000, 0x1000, 0x1004, 4, 4, 16, check=False) == c3.C3_EALIGN
    assert c3.c3_kernel_launches() == before
