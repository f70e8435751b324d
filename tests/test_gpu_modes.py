"""Every C3 mode, run through c3_run / c3_time, followed by the check the
pages' reviewers ask for: after each timed run, every output of the
collective is compared byte for byte with the oracle and the GEMM with the
oracle's tolerance (pith.science verdict, skeptic critique "concrete_test").
Also: the partitioned modes really run on disjoint SMs (%smid maps), and the
timer's derived fields obey their definitions."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

pytestmark = pytest.mark.gpu
TOL = 1e-4

MODES = [  # (name, mode, sm_split, priority)
    ("serial_sm", 0, 0, 0),
    ("baseline", 1, 0, 0),
    ("prioritised", 1, 0, 1),
    ("partitioned16", 1, 16, 0),
    ("partitioned32_prio", 1, 32, 1),
    ("ce", 2, 0, 0),
    ("ce_rp8", 2, 8, 0),
    ("serial_ce", 3, 0, 0),
    ("reclaim16", 4, 16, 0),
    ("reclaim32_prio", 4, 32, 1),
]


@pytest.fixture(scope="module")
def c3():
    from concurrent_communication_overlap_gb300 import c3 as mod
    return mod


class Setup:
    def __init__(self, c3, wname):
        w = I.WORKLOADS[wname]
        self.w = w
        A, B = I.gemm_operands(w)
        self.C_ref, self.S_ref = oracle.gemm(A, B)
        self.dA = torch.from_numpy(A.view(np.int16)).cuda()
        self.dB = torch.from_numpy(B.view(np.int16)).cuda()
        self.dC = torch.empty((w.M, w.N), dtype=torch.float32, device="cuda")
        payload = I.coll_payload(w)
        if w.coll == "allgather":
            self.ref = oracle.allgather(payload)
            self.dshards = [torch.from_numpy(s).cuda() for s in payload]
            self.dsend = None
            coll = c3.C3_COLL_ALLGATHER
        else:
            self.ref = oracle.alltoall(payload, w.nranks)
            self.dshards = None
            self.dsend = torch.from_numpy(payload).cuda()
            coll = c3.C3_COLL_ALLTOALL
        self.out = torch.empty(w.coll_bytes, dtype=torch.uint8, device="cuda")
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.p = c3.Problem(self.dA, self.dB, self.dC, w.M, w.N, w.K, coll, self.out, w.unit_bytes, w.nranks,
                            shards=self.dshards, send=self.dsend, flush=self.flush)

    def poison(self):
        self.dC.fill_(float("nan"))
        self.out.fill_(0xEE)
        torch.cuda.synchronize()

    def verify(self):
        assert np.array_equal(self.out.cpu().numpy(), self.ref), "collective output differs from the oracle"
        C = self.dC.cpu().numpy().astype(np.float64)
        err = np.abs(C - self.C_ref)
        assert not np.isnan(C).any()
        assert (err <= TOL * self.S_ref).all(), float(np.max(err - TOL * self.S_ref))


@pytest.fixture(scope="module", params=["tiny_ag", "tiny_a2a"])
def setup(c3, request):
    return Setup(c3, request.param)


@pytest.mark.parametrize("name,mode,split,prio", MODES, ids=[m[0] for m in MODES])
def test_mode_runs_and_outputs_are_exact(c3, setup, name, mode, split, prio):
    setup.poison()
    t = c3.c3_run(setup.p, mode, split, prio)
    assert t["status"] == 0 and t["t_conc"] > 0
    # T_conc runs from the start event to the later of the two completion events
    assert t["t_gemm_ev"] > 0 and t["t_comm_ev"] > 0
    assert t["t_conc"] == max(t["t_gemm_ev"], t["t_comm_ev"])
    assert t["gemm_ctas"] >= 1
    if mode in (2, 3):  # memcpy path: no collective kernel of this library ran
        assert t["comm_ctas"] == 0 and t["comm_sms"] == 0
    else:
        assert t["comm_ctas"] >= 1 and t["comm_sms"] >= 1
    setup.verify()


@pytest.mark.parametrize("split", [8, 16, 32])
def test_partitioned_runs_on_disjoint_sms(c3, setup, split):
    info = c3.c3_get_device_info()
    setup.poison()
    t = c3.c3_run(setup.p, 1, split, 0)
    # no SM ever held a GEMM CTA and a collective CTA at the same time
    assert t["smid_overlap"] == 0, t
    assert t["gemm_ctas"] <= info["sm_count"] - split
    # one launch group of SM-count CTAs: split now, the rest on SMs the GEMM leaves
    assert t["comm_ctas"] == info["sm_count"]
    setup.verify()


@pytest.mark.parametrize("split", [8, 32])
def test_reclaim_never_shares_an_sm_at_once(c3, setup, split):
    # the GEMM may reuse the collective's SMs after it leaves, never during
    setup.poison()
    info = c3.c3_get_device_info()
    t = c3.c3_run(setup.p, 4, split, 0)
    assert t["smid_overlap"] == 0, t
    assert t["comm_ctas"] == info["sm_count"]
    setup.verify()


@pytest.mark.parametrize("mode,prio", [(1, 0), (1, 1), (4, 0)])
@pytest.mark.parametrize("flavour", [0, 1])   # auto (bulk when exclusive), vec with a reservation
def test_partitioned_collective_widens_onto_the_sms_the_gemm_leaves(c3, mode, prio, flavour):
    """A one-tile GEMM beside a 256 MiB all-gather partitioned onto 8 SMs: the
    GEMM leaves ~140 SMs idle, so the collective's second launch part takes
    them and claims most of the work; the output stays bit-exact and no SM
    ever holds both kernels at once."""
    info = c3.c3_get_device_info()
    M, N, K = 128, 128, 64
    A = I.bf16_uniform(21, (M, K))
    B = I.bf16_uniform(22, (N, K))
    C_ref, S_ref = oracle.gemm(A, B)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    unit = 32 << 20
    shards = [torch.randint(0, 256, (unit,), dtype=torch.uint8, device="cuda") for _ in range(8)]
    out = torch.zeros(8 * unit, dtype=torch.uint8, device="cuda")
    ref = torch.cat(shards)
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLGATHER, out, unit, 8, shards=shards, sm_kernel=flavour)
    t = c3.c3_run(p, mode, 8, prio)
    assert t["status"] == 0
    assert torch.equal(out, ref)
    assert (np.abs(dC.cpu().numpy().astype(np.float64) - C_ref) <= TOL * S_ref).all()
    assert t["smid_overlap"] == 0, t
    assert t["comm_ctas"] == info["sm_count"]
    # 8 SMs alone would need ~3 ms for 512 MiB of traffic; the idle SMs join at once
    assert t["comm_sms"] > 64, t


@pytest.mark.parametrize("mode,prio", [(1, 0), (1, 1), (4, 0)])
def test_partitioned_allreduce_widens_onto_the_sms_the_gemm_leaves(c3, mode, prio):
    """The same one-tile GEMM beside an all-reduce of eight 8 M-element fp32
    vectors partitioned onto 8 SMs: the all-reduce's one-pass kernel is one
    launch group, so its second part takes the SMs the GEMM leaves; the output
    is the oracle's rank-order sum bit for bit and no SM holds both kernels at
    once."""
    info = c3.c3_get_device_info()
    M, N, K = 128, 128, 64
    A = I.bf16_uniform(23, (M, K))
    B = I.bf16_uniform(24, (N, K))
    C_ref, S_ref = oracle.gemm(A, B)
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    R, count = 8, 8 << 20
    bufs = [I.normal(1100 + r, count).astype(np.float32) for r in range(R)]
    dins = [torch.from_numpy(b).cuda() for b in bufs]
    out = torch.full((R * count,), float("nan"), dtype=torch.float32, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLREDUCE, out, count * 4, R, shards=dins)
    t = c3.c3_run(p, mode, 8, prio)
    assert t["status"] == 0
    ref, _ = oracle.allreduce(bufs)
    assert np.array_equal(out.cpu().numpy().reshape(ref.shape).view(np.uint32), ref.view(np.uint32))
    assert (np.abs(dC.cpu().numpy().astype(np.float64) - C_ref) <= TOL * S_ref).all()
    assert t["smid_overlap"] == 0, t
    assert t["comm_ctas"] == info["sm_count"]
    # 8 SMs alone would need ~0.7 ms for its ~0.5 GB of traffic; the idle SMs join at once
    assert t["comm_sms"] > 64, t


def _tiny_gemm(seed):
    M, N, K = 128, 128, 64
    A = I.bf16_uniform(seed, (M, K))
    B = I.bf16_uniform(seed + 1, (N, K))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    return (M, N, K), (A, B), (dA, dB, dC)


def test_partitioned_allreduce_work_counters_recycle_over_many_launches(c3):
    """More partitioned all-reduce runs than work slots (64), with first parts
    of 1..7 SMs (most slices claimed from the counter) and of 12..32 SMs (every
    slice a fixed unit), and a poisoned output each time: a claim counter left
    non-zero would skip slices and leave the poison in place."""
    (M, N, K), _, (dA, dB, dC) = _tiny_gemm(31)
    R, count = 8, 8 * 3000 + 32          # 3004 elements a chunk: ragged slices and pieces
    bufs = [I.normal(1200 + r, count).astype(np.float32) for r in range(R)]
    dins = [torch.from_numpy(b).cuda() for b in bufs]
    ref, _ = oracle.allreduce(bufs)
    ref_t = torch.from_numpy(ref.reshape(-1).copy()).cuda()
    out = torch.empty(R * count, dtype=torch.float32, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLREDUCE, out, count * 4, R, shards=dins)
    splits = [1, 2, 3, 4, 5, 6, 7, 12, 16, 32]
    for i in range(150):
        out.fill_(float("nan"))
        t = c3.c3_run(p, 4 if i % 5 == 4 else 1, splits[i % len(splits)], i % 2)
        assert t["status"] == 0
        assert torch.equal(out.view(torch.int32), ref_t.view(torch.int32)), i
    c3.c3_status_check()


@pytest.mark.parametrize("nranks,count", [(8, 1 << 16), (8, 32 * 37), (5, 20 * 9), (2, 8), (1, 4), (1, 4096 + 4)])
@pytest.mark.parametrize("split", [8, 64])
@pytest.mark.parametrize("l2", [0, 1])   # normal, evict-first loads and stores
def test_partitioned_allreduce_bit_exact(c3, nranks, count, split, l2):
    """The all-reduce's one-pass kernel in partitioned runs at rank counts 1..8
    and ragged sizes, with either L2 policy, against the oracle's rank-order
    fp32 sum."""
    (M, N, K), (A, B), (dA, dB, dC) = _tiny_gemm(41)
    bufs = [I.normal(1300 + r, count).astype(np.float32) for r in range(nranks)]
    bufs[0][:3] = [-0.0, np.inf, 1e38]
    if nranks > 1:
        bufs[1][2] = 1e38
    dins = [torch.from_numpy(b).cuda() for b in bufs]
    out = torch.full((nranks * count,), float("nan"), dtype=torch.float32, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLREDUCE, out, count * 4, nranks, shards=dins, coll_l2=l2)
    t = c3.c3_run(p, 1, split, 0)
    assert t["status"] == 0
    ref, _ = oracle.allreduce(bufs)
    assert np.array_equal(out.cpu().numpy().reshape(ref.shape).view(np.uint32), ref.view(np.uint32))
    C_ref, S_ref = oracle.gemm(A, B)
    assert (np.abs(dC.cpu().numpy().astype(np.float64) - C_ref) <= TOL * S_ref).all()


@pytest.mark.parametrize("M,N,K", [(256, 28672, 1024), (2048, 4096, 512)])
def test_reclaim_plans_the_gemm_for_the_sms_it_starts_on(c3, M, N, K):
    """Reclaim plans the GEMM's tiles for the SM count - sm_split SMs it starts
    on, as a partition does, and launches up to every SM: min(tiles, SM count)
    CTAs.  The memory-bound shape then fits one wave on the free SMs; a shape of
    many waves keeps every SM.  The output stays within the tolerance."""
    info = c3.c3_get_device_info()
    split = 16
    bn, msub, _ = c3.c3_gemm_plan(M, N, K, info["sm_count"] - split)
    tiles = -(-M // (128 * msub)) * -(-N // bn)
    A = I.bf16_uniform(51, (M, K))
    B = I.bf16_uniform(52, (N, K))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    unit = 1 << 20
    shards = [torch.randint(0, 256, (unit,), dtype=torch.uint8, device="cuda") for _ in range(8)]
    out = torch.zeros(8 * unit, dtype=torch.uint8, device="cuda")
    p = c3.Problem(dA, dB, dC, M, N, K, c3.C3_COLL_ALLGATHER, out, unit, 8, shards=shards)
    t = c3.c3_run(p, 4, split, 0)
    assert t["status"] == 0
    assert t["gemm_ctas"] == min(tiles, info["sm_count"]), (t["gemm_ctas"], tiles)
    assert t["smid_overlap"] == 0, t
    assert torch.equal(out, torch.cat(shards))
    rows = np.array([0, M // 2, M - 1])
    C_ref, S_ref = oracle.gemm(A[rows], B)
    got = dC[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert (np.abs(got - C_ref) <= TOL * S_ref).all()


def test_copy_work_counters_recycle_over_many_launches(c3):
    """More collective launches than work-counter slots (64), with launch
    groups of 1..7 CTAs: a counter left non-zero would make a later launch
    skip work, so every output is compared with the expected bytes."""
    unit = (1 << 20) + 48
    shards = [torch.randint(0, 256, (unit,), dtype=torch.uint8, device="cuda") for _ in range(8)]
    ref = torch.cat(shards)
    out = torch.empty(8 * unit, dtype=torch.uint8, device="cuda")
    for i in range(150):
        out.fill_(0xA5)
        c3.c3_allgather(shards, out, unit, 8, engine=c3.C3_ENGINE_SM, sm_budget=1 + i % 7)
        assert torch.equal(out, ref), i
    c3.c3_status_check()


def test_scheduler_slots_recycle_over_many_launches(c3):
    # more launches than scheduler slots (64): every slot must come back to zero
    M, N, K = 640, 1000, 128          # 5 x 8 = 40 tiles of 128 x 128
    A = I.bf16_uniform(5, (M, K))
    B = I.bf16_uniform(6, (N, K))
    dA = torch.from_numpy(A.view(np.int16)).cuda()
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    C_ref, S_ref = oracle.gemm(A, B)
    for i in range(150):
        dC.fill_(float("nan"))
        c3.c3_gemm(dA, dB, dC, M, N, K, 1 + i % 7)
    c3.c3_status_check()
    assert (np.abs(dC.cpu().numpy() - C_ref) <= TOL * S_ref).all()


def test_ce_with_gemm_cap_leaves_sms_free(c3, setup):
    info = c3.c3_get_device_info()
    t = c3.c3_run(setup.p, 2, 16, 0)
    assert t["gemm_sms"] <= info["sm_count"] - 16
    setup.verify()


def test_timer_fields_follow_their_definitions(c3, setup):
    reps = c3.c3_time(setup.p, 1, 0, 1, warmup=1, reps=3)
    for r in reps:
        assert r["t_gemm_iso"] > 0 and r["t_comm_iso"] > 0 and r["t_conc"] > 0
        m = oracle.c3_metrics(r["t_gemm_iso"], r["t_comm_iso"], r["t_conc"])
        assert r["t_serial"] == pytest.approx(m["t_serial"], rel=1e-12)
        assert r["t_ideal"] == pytest.approx(m["t_ideal"], rel=1e-12)
        assert r["s_ideal"] == pytest.approx(m["s_ideal"], rel=1e-12)
        assert r["s_real"] == pytest.approx(m["s_real"], rel=1e-12)
        assert r["pct_ideal_gain"] == pytest.approx(m["pct_ideal_gain"], rel=1e-9, abs=1e-12)
        assert r["pct_ideal_ratio"] == pytest.approx(m["pct_ideal_ratio"], rel=1e-12)
        assert r["class"] == m["class"]
    setup.verify()


def test_every_mode_under_c3_time_stays_exact(c3, setup):
    for name, mode, split, prio in MODES:
        setup.poison()
        c3.c3_time(setup.p, mode, split, prio, warmup=0, reps=2)
        setup.verify()


@pytest.mark.parametrize("plateau_scale", [0.25, 4.0])
def test_timer_bounds_and_settle_follow_their_definitions(c3, setup, plateau_scale):
    """c3_time's gemm_bound / coll_bound equal the oracle's classification of
    the same times and rates, on both sides of the collective's threshold,
    and a settle period leaves the outputs exact and the timer's fields
    consistent."""
    w = setup.w
    first = c3.c3_time(setup.p, 1, 0, 0, warmup=0, reps=1)[0]
    # a plateau that puts this collective clearly on one side of half-plateau
    rate = w.coll_bytes / first["t_comm_iso"]
    plateau = rate * plateau_scale
    peak_flops, peak_bw = 1.9e15, 6.8e12
    p = c3.Problem(setup.dA, setup.dB, setup.dC, w.M, w.N, w.K, setup.p.rec.coll, setup.out, w.unit_bytes,
                   w.nranks, shards=setup.dshards, send=setup.dsend, flush=setup.flush, settle_us=300,
                   peak_flops=peak_flops, peak_bytes_per_s=peak_bw, coll_plateau_sm=plateau, coll_plateau_ce=plateau)
    setup.poison()
    for mode in (1, 2):
        for r in c3.c3_time(p, mode, 0, 0, warmup=0, reps=3):
            g, c = oracle.c3_bounds(w.gemm_flops, w.gemm_bytes, peak_flops, peak_bw, w.coll_bytes,
                                    r["t_comm_iso"], plateau)
            assert r["gemm_bound_name"] == g and r["coll_bound_name"] == c
            m = oracle.c3_metrics(r["t_gemm_iso"], r["t_comm_iso"], r["t_conc"])
            assert r["s_ideal"] == pytest.approx(m["s_ideal"], rel=1e-12)
    setup.verify()
    # no peaks, no plateau: both axes unknown
    r = c3.c3_time(setup.p, 1, 0, 0, warmup=0, reps=1)[0]
    assert r["gemm_bound"] == c3.C3_BOUND_UNKNOWN and r["coll_bound"] == c3.C3_BOUND_UNKNOWN


def test_cta_windows_describe_the_last_run(c3, setup):
    """After a serial run, the GEMM's per-CTA windows: one per launched CTA,
    each on its own SM, ordered start <= end, starting from zero; the
    collective's windows belong to CTAs that moved data."""
    t = c3.c3_run(setup.p, 0, 0, 0)
    g = c3.c3_cta_windows(0)
    assert len(g) == t["gemm_ctas"]
    assert len({sm for _, sm, _, _ in g}) == len(g)
    assert min(t0 for _, _, t0, _ in g) == 0.0
    assert all(0.0 <= t0 <= t1 for _, _, t0, t1 in g)
    assert max(t1 for _, _, _, t1 in g) <= t["t_gemm_ev"]
    cw = c3.c3_cta_windows(1)
    assert 1 <= len(cw) <= t["comm_ctas"]
    assert all(t0 <= t1 for _, _, t0, t1 in cw)


@pytest.mark.parametrize("wname", ["tiny_ag", "tiny_a2a"])
@pytest.mark.parametrize("mode,split", [(2, 0), (2, 8), (3, 0)])
def test_host_staged_copy_engine_is_exact(c3, wname, mode, split):
    """The copy-engine collective bounced through page-locked host memory
    (C3_CE_HOST_STAGED: device -> host -> device in pieces of at most 16 MiB,
    two DMA chains) delivers the oracle's bytes, concurrently with the GEMM
    and serially, and runs no collective kernel of this library."""
    s = Setup(c3, wname)
    w = s.w
    stage = torch.empty(w.coll_bytes, dtype=torch.uint8).pin_memory()
    stage.fill_(0x5A)
    p = c3.Problem(s.dA, s.dB, s.dC, w.M, w.N, w.K, s.p.rec.coll, s.out, w.unit_bytes, w.nranks,
                   shards=s.dshards, send=s.dsend, flush=s.flush, ce_variant=c3.C3_CE_HOST_STAGED, ce_stage=stage)
    for _ in range(2):  # the second run replays the cached graph
        s.poison()
        t = c3.c3_run(p, mode, split, 0)
        assert t["status"] == 0 and t["comm_ctas"] == 0
        s.verify()
    # the bounce buffer holds the collective's pieces in source order: segment i at i * seg_bytes
    if w.coll == "allgather":
        assert np.array_equal(stage.numpy(), s.ref)


def test_host_staged_copy_engine_rejects_a_wrong_bounce_buffer(c3):
    """A bounce buffer in device memory, one too small, or sources that are
    already page-locked host memory are argument errors, with nothing run."""
    s = Setup(c3, "tiny_ag")
    w = s.w

    def run(stage, shards):
        p = c3.Problem(s.dA, s.dB, s.dC, w.M, w.N, w.K, c3.C3_COLL_ALLGATHER, s.out, w.unit_bytes, w.nranks,
                       shards=shards, ce_variant=c3.C3_CE_HOST_STAGED, ce_stage=stage)
        t = c3.C3Timing()
        return c3.lib().c3_run(ctypes.byref(p.rec), 2, 0, 0, ctypes.byref(t))

    dev_stage = torch.empty(w.coll_bytes, dtype=torch.uint8, device="cuda")
    assert run(dev_stage, s.dshards) == c3.C3_EINVAL
    small = torch.empty(w.coll_bytes - 16, dtype=torch.uint8).pin_memory()
    assert run(small, s.dshards) == c3.C3_EINVAL
    pageable = torch.empty(w.coll_bytes, dtype=torch.uint8)
    assert run(pageable, s.dshards) == c3.C3_EINVAL
    host_shards = [torch.from_numpy(x).pin_memory() for x in I.coll_payload(w)]
    ok_stage = torch.empty(w.coll_bytes, dtype=torch.uint8).pin_memory()
    assert run(ok_stage, host_shards) == c3.C3_EUNSUP


def test_host_staged_copy_engine_cuts_segments_into_pieces(c3):
    """Shards of 40 MiB + 16 bytes go through the bounce buffer in pieces of
    16, 16 and 8 MiB + 16 bytes (ragged last piece), byte-exact."""
    nranks, shard = 8, (40 << 20) + 16
    payload = [I.random_bytes(3000 + r, shard) for r in range(nranks)]
    ref = oracle.allgather(payload)
    dsh = [torch.from_numpy(x).cuda() for x in payload]
    out = torch.full((nranks * shard,), 0xEE, dtype=torch.uint8, device="cuda")
    A = torch.zeros((128, 128), dtype=torch.int16, device="cuda")
    C = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    stage = torch.empty(nranks * shard, dtype=torch.uint8).pin_memory()
    p = c3.Problem(A, A, C, 128, 128, 128, c3.C3_COLL_ALLGATHER, out, shard, nranks, shards=dsh,
                   ce_variant=c3.C3_CE_HOST_STAGED, ce_stage=stage)
    t = c3.c3_run(p, 2, 0, 0)
    assert t["status"] == 0
    assert np.array_equal(out.cpu().numpy(), ref)
    assert float(C.abs().max()) == 0.0
