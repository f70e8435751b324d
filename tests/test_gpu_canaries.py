"""Guard words around every output buffer: no kernel of the library writes
outside the bytes its result owns.

Each output (the GEMM's C, a collective's output) is carved out of a larger
device buffer whose 4 KiB on either side hold a fixed bit pattern.  After the
call the pattern must be intact, bit for bit, and the output must still match
the oracle.  The shapes are ragged in M and N, so the TMA-store epilogue's
clipping at the tensor edges and the direct-store path (N % 4 != 0) are both
covered, as are the SM copy kernels, the memcpy path and every concurrent mode."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

pytestmark = pytest.mark.gpu
PAD = 4096            # bytes of guard on each side
PATTERN = 0x5AC3E17B  # guard word


@pytest.fixture(scope="module")
def c3():
    from concurrent_communication_overlap_gb300 import c3 as mod
    return mod


class Guarded:
    """A device buffer of `nbytes` (a view into a larger, guarded allocation)."""

    def __init__(self, nbytes, dtype):
        words = (2 * PAD + nbytes + 3) // 4
        fill = PATTERN if PATTERN < (1 << 31) else PATTERN - (1 << 32)  # the same 32 bits as an int32
        self.raw = torch.full((words,), fill, dtype=torch.int32, device="cuda")
        self.nbytes = nbytes
        self.view = self.raw.view(torch.uint8)[PAD:PAD + nbytes].view(dtype)

    def guards_intact(self):
        b = self.raw.view(torch.uint8).cpu().numpy()
        ref = np.full(PAD // 4, PATTERN, dtype=np.uint32).view(np.uint8)
        tail = b[PAD + self.nbytes:]
        tail_ref = np.frombuffer(np.full((tail.size + 3) // 4 + 1, PATTERN, dtype=np.uint32).tobytes(), np.uint8)
        # the tail starts at PAD + nbytes, which may not be word-aligned: compare with the
        # pattern at the same byte offsets
        off = (PAD + self.nbytes) % 4
        return np.array_equal(b[:PAD], ref) and np.array_equal(tail, tail_ref[off:off + tail.size])


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("M,N,K,budget", [
    (300, 500, 200, 0), (300, 500, 200, 2), (400, 1100, 520, 4), (129, 33, 8, 0),
    (256, 203, 136, 0), (400, 700, 520, 2), (512, 512, 512, 0), (1000, 1000, 512, 7),
])
def test_gemm_writes_only_c(c3, M, N, K, budget):
    A = I.bf16_uniform(1000, (M, K), -1.0, 1.0)
    B = I.bf16_uniform(1001, (N, K), -1.0, 1.0)
    g = Guarded(M * N * 4, torch.float32)
    C = g.view.view(M, N)
    c3.c3_gemm(dev_u16(A), dev_u16(B), C, M, N, K, budget)
    c3.c3_status_check()
    assert g.guards_intact()
    C_ref, S_ref = oracle.gemm(A, B)
    Cg = C.cpu().numpy().astype(np.float64)
    assert (np.abs(Cg - C_ref) <= 1e-4 * S_ref).all()


@pytest.mark.parametrize("engine", [0, 1])
@pytest.mark.parametrize("unit", [16, 4096 + 48, 1 << 20])
def test_collectives_write_only_their_output(c3, engine, unit):
    shards = [I.random_bytes(1002 + r, unit) for r in range(8)]
    g = Guarded(8 * unit, torch.uint8)
    c3.c3_allgather([torch.from_numpy(s).cuda() for s in shards], g.view, unit, 8, engine=engine)
    c3.c3_status_check()
    assert g.guards_intact()
    assert np.array_equal(g.view.cpu().numpy(), oracle.allgather(shards))
    send = I.random_bytes(7, 64 * unit)
    g2 = Guarded(64 * unit, torch.uint8)
    c3.c3_alltoall(torch.from_numpy(send).cuda(), g2.view, unit, 8, engine=engine)
    c3.c3_status_check()
    assert g2.guards_intact()
    assert np.array_equal(g2.view.cpu().numpy(), oracle.alltoall(send, 8))


@pytest.mark.parametrize("engine", [0, 1])
def test_allreduce_writes_only_its_output(c3, engine):
    count = 32 * 37
    bufs = [I.normal(1002 + q, count).astype(np.float32) for q in range(8)]
    g = Guarded(8 * count * 4, torch.float32)
    c3.c3_allreduce([torch.from_numpy(b).cuda() for b in bufs], g.view, count, 8, engine=engine)
    c3.c3_status_check()
    assert g.guards_intact()
    out, _ = oracle.allreduce(bufs)
    assert np.array_equal(g.view.cpu().numpy().view(np.uint32), out.reshape(-1).view(np.uint32))


@pytest.mark.parametrize("mode,split,prio", [(1, 0, 0), (1, 0, 1), (1, 16, 0), (4, 16, 0), (2, 0, 0), (2, 8, 0),
                                             (0, 0, 0), (3, 0, 0)])
def test_every_mode_writes_only_its_outputs(c3, mode, split, prio):
    M, N, K = 300, 500, 200
    A = I.bf16_uniform(1000, (M, K), -1.0, 1.0)
    B = I.bf16_uniform(1001, (N, K), -1.0, 1.0)
    unit = 64 * 1024 + 16
    shards = [I.random_bytes(1002 + r, unit) for r in range(8)]
    gc = Guarded(M * N * 4, torch.float32)
    go = Guarded(8 * unit, torch.uint8)
    p = c3.Problem(dev_u16(A), dev_u16(B), gc.view.view(M, N), M, N, K, c3.C3_COLL_ALLGATHER, go.view, unit, 8,
                   shards=[torch.from_numpy(s).cuda() for s in shards])
    t = c3.c3_run(p, mode, split, prio)
    assert t["status"] == 0
    assert gc.guards_intact() and go.guards_intact()
    assert np.array_equal(go.view.cpu().numpy(), oracle.allgather(shards))
    C_ref, S_ref = oracle.gemm(A, B)
    assert (np.abs(gc.view.view(M, N).cpu().numpy().astype(np.float64) - C_ref) <= 1e-4 * S_ref).all()
