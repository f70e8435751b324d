"""GPU parity of collectives whose sources sit in page-locked host memory,
alone, in every c3_run mode, and as asynchronous calls beside the GEMM.

The remote ranks' buffers are placed across the CPU-GPU link (pinned host
memory) while the output stays in device memory.  The SM copy kernel reads
them with plain loads over the link; the memcpy path reaches them with
host-to-device DMA.  Either way the result is the oracle's byte for byte.
Pageable host memory and host destinations are argument errors, and the
cp.async.bulk kernel (device sources only) refuses host sources."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c3():
    from concurrent_communication_overlap_gb300 import c3 as mod
    return mod


def pinned_bytes(a):
    t = torch.empty(a.size, dtype=torch.uint8, pin_memory=True)
    t.numpy()[:] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    return t


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("shard_bytes", [1 << 20, 16, 3 * 65536 + 4096 + 48])
@pytest.mark.parametrize("engine,budget", [(0, 0), (0, 4), (1, 0)])
def test_allgather_from_host(c3, shard_bytes, engine, budget):
    shards = [I.random_bytes(1002 + r, shard_bytes) for r in range(8)]
    hs = [pinned_bytes(s) for s in shards]
    out = torch.full((8 * shard_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    c3.c3_allgather(hs, out, shard_bytes, 8, engine=engine, sm_budget=budget)
    c3.c3_status_check()
    assert np.array_equal(out.cpu().numpy(), oracle.allgather(shards))


def test_allgather_mixed_host_and_device(c3):
    # rank 0's shard is local (device), the other seven across the link
    sb = 64 * 1024 + 16
    shards = [I.random_bytes(1002 + r, sb) for r in range(8)]
    srcs = [torch.from_numpy(shards[0]).cuda()] + [pinned_bytes(s) for s in shards[1:]]
    ref = oracle.allgather(shards)
    for engine in (0, 1):
        out = torch.zeros(8 * sb, dtype=torch.uint8, device="cuda")
        c3.c3_allgather(srcs, out, sb, 8, engine=engine)
        c3.c3_status_check()
        assert np.array_equal(out.cpu().numpy(), ref), engine


@pytest.mark.parametrize("block", [128 * 1024, 16, 4096 + 32])
@pytest.mark.parametrize("engine", [0, 1])
def test_alltoall_from_host(c3, block, engine):
    send = I.random_bytes(1002, 64 * block)
    hin = pinned_bytes(send)
    out = torch.full((64 * block,), 0x5A, dtype=torch.uint8, device="cuda")
    c3.c3_alltoall(hin, out, block, 8, engine=engine)
    c3.c3_status_check()
    assert np.array_equal(out.cpu().numpy(), oracle.alltoall(send, 8))


@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("coll", ["allgather", "alltoall"])
def test_memcpy_variants_from_host(c3, variant, coll):
    unit = 64 * 1024 + 16
    if coll == "allgather":
        payload = [I.random_bytes(1002 + r, unit) for r in range(8)]
        ref = oracle.allgather(payload)
        shards, send, cid = [pinned_bytes(x) for x in payload], None, c3.C3_COLL_ALLGATHER
    else:
        payload = I.random_bytes(1002, 64 * unit)
        ref = oracle.alltoall(payload, 8)
        shards, send, cid = None, pinned_bytes(payload), c3.C3_COLL_ALLTOALL
    out = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    p = c3.Problem(None, None, None, 0, 0, 0, cid, out, unit, 8, shards=shards, send=send, ce_variant=variant)
    for _ in range(2):
        out.fill_(0x33)
        c3.c3_run(p, c3.C3_MODE_SERIAL_CE, 0, 0)
        assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("mode,split,prio", [(1, 0, 0), (1, 0, 1), (1, 16, 0), (4, 16, 0), (2, 0, 0), (2, 8, 0),
                                             (0, 0, 0), (3, 0, 0)])
def test_every_mode_with_host_sources(c3, mode, split, prio):
    w = I.WORKLOADS["tiny_ag"]
    A, B = I.gemm_operands(w)
    shards = I.coll_payload(w)
    ref = oracle.allgather(shards)
    C_ref, S_ref = oracle.gemm(A, B)
    dA, dB = dev_u16(A), dev_u16(B)
    hs = [pinned_bytes(s) for s in shards]
    dC = torch.full((w.M, w.N), float("nan"), device="cuda")
    out = torch.zeros(w.coll_bytes, dtype=torch.uint8, device="cuda")
    p = c3.Problem(dA, dB, dC, w.M, w.N, w.K, c3.C3_COLL_ALLGATHER, out, w.unit_bytes, 8, shards=hs)
    t = c3.c3_run(p, mode, split, prio)
    assert t["status"] == 0
    assert np.array_equal(out.cpu().numpy(), ref)
    C = dC.cpu().numpy().astype(np.float64)
    assert not np.isnan(C).any()
    assert (np.abs(C - C_ref) <= 1e-4 * S_ref).all()
    if mode in (1, 4) and split:
        assert t["smid_overlap"] == 0


def test_host_source_argument_errors(c3):
    sb = 4096
    shards = [I.random_bytes(1002 + r, sb) for r in range(8)]
    pageable = [torch.from_numpy(s) for s in shards]          # not page-locked
    out = torch.zeros(8 * sb, dtype=torch.uint8, device="cuda")
    assert c3.c3_allgather(pageable, out, sb, 8, check=False) == c3.C3_EINVAL
    hs = [pinned_bytes(s) for s in shards]
    host_out = torch.zeros(8 * sb, dtype=torch.uint8, pin_memory=True)
    ds = [torch.from_numpy(s).cuda() for s in shards]
    assert c3.c3_allgather(ds, host_out, sb, 8, check=False) == c3.C3_EINVAL   # destination on the host
    p = c3.Problem(None, None, None, 0, 0, 0, c3.C3_COLL_ALLGATHER, out, sb, 8, shards=hs,
                   sm_kernel=c3.C3_SMK_BULK)
    t = c3.C3Timing()
    assert c3.lib().c3_run(ctypes.byref(p.rec), c3.C3_MODE_SERIAL_SM, 0, 0, ctypes.byref(t)) == c3.C3_EUNSUP
    # nothing was left in a failed state: a valid call still works
    c3.c3_allgather(hs, out, sb, 8)
    c3.c3_status_check()
    assert np.array_equal(out.cpu().numpy(), oracle.allgather(shards))


@pytest.mark.parametrize("engine", [0, 1])
@pytest.mark.parametrize("coll", ["allgather", "alltoall"])
def test_async_calls_on_two_streams(c3, engine, coll):
    # What a caller with host-resident inputs does: the GEMM chain on one
    # stream (copy A in, c3_gemm, read C back) and the collective reading its
    # pinned host sources on another, both in flight at once.
    w = I.WORKLOADS["tiny_ag"]
    A, B = I.gemm_operands(w)
    C_ref, S_ref = oracle.gemm(A, B)
    hA = torch.from_numpy(np.ascontiguousarray(A).view(np.int16)).pin_memory()
    dA = torch.empty(hA.shape, dtype=torch.int16, device="cuda")
    dB = dev_u16(B)
    dC = torch.full((w.M, w.N), float("nan"), device="cuda")
    hC = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
    unit = 1 << 20 if coll == "allgather" else 128 * 1024
    if coll == "allgather":
        payload = [I.random_bytes(1002 + r, unit) for r in range(8)]
        ref = oracle.allgather(payload)
        srcs = [pinned_bytes(x) for x in payload]
    else:
        payload = I.random_bytes(1002, 64 * unit)
        ref = oracle.alltoall(payload, 8)
        srcs = pinned_bytes(payload)
    out = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        dC.fill_(float("nan"))
        out.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s1):
            dA.copy_(hA, non_blocking=True)
            c3.c3_gemm(dA, dB, dC, w.M, w.N, w.K, 0, s1)
            hC.copy_(dC, non_blocking=True)
        if coll == "allgather":
            c3.c3_allgather(srcs, out, unit, 8, engine=engine, stream=s2)
        else:
            c3.c3_alltoall(srcs, out, unit, 8, engine=engine, stream=s2)
        torch.cuda.synchronize()
        c3.c3_status_check()
        assert np.array_equal(out.cpu().numpy(), ref)
        C = hC.numpy().astype(np.float64)
        assert not np.isnan(C).any()
        assert (np.abs(C - C_ref) <= 1e-4 * S_ref).all()


@pytest.mark.parametrize("mode,split", [(1, 8), (4, 8), (4, 32)])
def test_partitioned_link_collective_overlaps_the_gemm(c3, mode, split):
    """A 128 MiB all-gather from host memory (link-bound, ~0.6 ms) beside an
    8192^3 GEMM (~0.6 ms), partitioned or with reclaim: the collective's
    second launch part must not take the SMs the GEMM is waiting for, so the
    pair overlaps -- T_conc well under the serial sum -- and stays exact."""
    M = N = K = 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    dA = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    dB = (0.02 * torch.randn((N, K), device="cuda", generator=g)).to(torch.bfloat16)
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    sb = 16 << 20
    shards = [I.random_bytes(1002 + r, sb) for r in range(8)]
    hs = [pinned_bytes(s) for s in shards]
    out = torch.zeros(8 * sb, dtype=torch.uint8, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLGATHER, out, sb, 8, shards=hs)
    for r in c3.c3_time(p, mode, split, 0, warmup=1, reps=3):
        assert r["status"] == 0
        assert r["t_conc"] < 0.8 * (r["t_gemm_iso"] + r["t_comm_iso"]), r
    assert np.array_equal(out.cpu().numpy(), oracle.allgather(shards))


@pytest.mark.parametrize("mode,split", [(4, 8), (4, 32)])
def test_reclaim_link_collective_overlaps_the_compute_bound_ffn_gemm(c3, mode, split):
    """The Llama-70B-FFN-shaped GEMM (2 ms) beside a 448 MiB all-gather from
    host memory (link-bound, ~2.2 ms) with reclaim: the collective's first
    part must hold its SMs from the start, beside the GEMM, not after it."""
    M, N, K = 8192, 28672, 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    dA = torch.randn((M, K), device="cuda", generator=g).to(torch.bfloat16)
    dB = (0.02 * torch.randn((N, K), device="cuda", generator=g)).to(torch.bfloat16)
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    sb = 56 << 20
    hs = [torch.randint(0, 256, (sb,), dtype=torch.uint8).pin_memory() for _ in range(8)]
    out = torch.zeros(8 * sb, dtype=torch.uint8, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLGATHER, out, sb, 8, shards=hs, settle_us=5000)
    for r in c3.c3_time(p, mode, split, 0, warmup=1, reps=3):
        assert r["status"] == 0
        assert r["t_conc"] < 0.8 * (r["t_gemm_iso"] + r["t_comm_iso"]), r
    assert torch.equal(out.cpu(), torch.cat(hs))
