"""Python binding of libc3.so (include/c3_api.h): argument marshalling only.

Every function has the C entry point's name and meaning; tensors are passed
as pointers (``tensor.data_ptr()``: device memory, or page-locked host memory
for a collective's sources), streams as ``cudaStream_t`` handles
(``torch.cuda.Stream.cuda_stream``).  All work runs in the library's CUDA
kernels or in driver memcpy transfers; nothing here computes.  Importing this
module raises ImportError when libc3.so has not been built: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libc3.so")

C3_OK, C3_EINVAL, C3_EALIGN, C3_ECUDA, C3_ETIMEOUT, C3_EUNSUP = 0, -1, -2, -3, -4, -5
C3_ENGINE_SM, C3_ENGINE_CE = 0, 1
C3_COLL_ALLGATHER, C3_COLL_ALLTOALL, C3_COLL_ALLREDUCE = 0, 1, 2
C3_MODE_SERIAL_SM, C3_MODE_CONCURRENT_SM, C3_MODE_CONCURRENT_CE, C3_MODE_SERIAL_CE = 0, 1, 2, 3
C3_MODE_CONCURRENT_SM_RECLAIM = 4
C3_SMK_AUTO, C3_SMK_VEC, C3_SMK_BULK = 0, 1, 2
C3_L2_NORMAL, C3_L2_EVICT_FIRST = 0, 1
C3_CE_PER_SEGMENT, C3_CE_STRIDED, C3_CE_GRAPH, C3_CE_GRAPH_PARALLEL, C3_CE_HOST_STAGED = 0, 1, 2, 3, 4
C3_FAULT_NONE, C3_FAULT_GEMM_LAUNCH, C3_FAULT_SM_COLL_LAUNCH, C3_FAULT_MEMCPY, C3_FAULT_DEVICE_INIT = 0, 1, 2, 3, 4
CLASS_NAMES = {0: "G-long", 1: "GC-equal", 2: "C-long"}

_i64, _int, _vp, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t


class C3DeviceInfo(ctypes.Structure):
    _fields_ = [("device", _int), ("sm_count", _int), ("l2_bytes", _int), ("smem_per_sm", _int),
                ("smem_per_block", _int), ("cc_major", _int), ("cc_minor", _int),
                ("gemm_smem_bytes", _int), ("comm_default_sms", _int)]


class C3Problem(ctypes.Structure):
    _fields_ = [("A", _vp), ("B", _vp), ("C", _vp), ("M", _i64), ("N", _i64), ("K", _i64),
                ("coll", _int), ("shards", ctypes.POINTER(_vp)), ("send", _vp), ("recv", _vp),
                ("unit_bytes", _sz), ("nranks", _int), ("comm_sms", _int), ("sm_kernel", _int), ("coll_l2", _int),
                ("ce_variant", _int),
                ("flush_buf", _vp), ("flush_bytes", _sz), ("stream", _vp),
                ("settle_us", _int), ("peak_flops", ctypes.c_double), ("peak_bytes_per_s", ctypes.c_double),
                ("coll_plateau_sm", ctypes.c_double), ("coll_plateau_ce", ctypes.c_double),
                ("ce_stage", _vp), ("ce_stage_bytes", _sz)]


_TIMING_DOUBLES = ["t_gemm_iso", "t_comm_iso", "t_serial", "t_serial_meas", "t_conc", "t_ideal", "s_ideal",
                   "s_real", "pct_ideal_gain", "pct_ideal_ratio", "t_gemm_dev", "t_comm_dev", "t_gemm_ev",
                   "t_comm_ev"]
_TIMING_INTS = ["cls", "mode", "sm_split", "priority", "gemm_ctas", "comm_ctas", "gemm_sms", "comm_sms",
                "smid_overlap", "sms_shared_any", "status", "gemm_bound", "coll_bound"]
C3_BOUND_UNKNOWN, C3_GEMM_COMPUTE, C3_GEMM_MEMORY = -1, 0, 1
C3_COLL_LATENCY, C3_COLL_BANDWIDTH = 0, 1
GEMM_BOUND_NAMES = {-1: "unknown", 0: "compute", 1: "memory"}
COLL_BOUND_NAMES = {-1: "unknown", 0: "latency", 1: "bandwidth"}


class C3Timing(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in _TIMING_DOUBLES] + [(n, _int) for n in _TIMING_INTS]

    def as_dict(self):
        d = {n: getattr(self, n) for n in _TIMING_DOUBLES + _TIMING_INTS}
        d["class"] = CLASS_NAMES.get(self.cls, "?")
        d["gemm_bound_name"] = GEMM_BOUND_NAMES.get(self.gemm_bound, "?")
        d["coll_bound_name"] = COLL_BOUND_NAMES.get(self.coll_bound, "?")
        return d


class C3CtaWindow(ctypes.Structure):
    _fields_ = [("cta", _int), ("smid", _int), ("t_start", ctypes.c_double), ("t_end", ctypes.c_double)]


C3_RP_MAX = 16


class C3RpTable(ctypes.Structure):
    _fields_ = [("n", _int), ("sms", _int * C3_RP_MAX), ("gemm_compute", ctypes.c_double * C3_RP_MAX),
                ("gemm_memory", ctypes.c_double * C3_RP_MAX), ("coll", ctypes.c_double * C3_RP_MAX)]


class C3Error(RuntimeError):
    def __init__(self, status, where, detail):
        super().__init__(f"{where}: {status} ({c3_strerror(status)}): {detail}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libc3.so is not built ({LIB_PATH}); run "
                          "python -m concurrent_communication_overlap_gb300.build")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "c3_get_device_info": [ctypes.POINTER(C3DeviceInfo)],
        "c3_strerror": [_int],
        "c3_last_error": [],
        "c3_status_check": [_vp],
        "c3_shutdown": [],
        "c3_gemm": [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp],
        "c3_allgather": [ctypes.POINTER(_vp), _vp, _sz, _int, _int, _int, _vp],
        "c3_alltoall": [_vp, _vp, _sz, _int, _int, _int, _vp],
        "c3_allreduce": [ctypes.POINTER(_vp), _vp, _sz, _int, _int, _int, _vp],
        "c3_run": [ctypes.POINTER(C3Problem), _int, _int, _int, ctypes.POINTER(C3Timing)],
        "c3_time": [ctypes.POINTER(C3Problem), _int, _int, _int, _int, _int, ctypes.POINTER(C3Timing)],
        "c3_l2_flush": [_vp, _sz, _vp],
        "c3_gemm_noalloc": [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _int],
        "c3_selftest_wait": [ctypes.c_uint64, _int, _vp],
        "c3_inject_fault": [_int],
        "c3_sp_predict": [_int, _int],
        "c3_rp_predict": [ctypes.POINTER(C3RpTable), ctypes.c_double, ctypes.c_double, ctypes.c_double,
                          ctypes.c_double, ctypes.c_double, ctypes.POINTER(_int), ctypes.POINTER(ctypes.c_double),
                          ctypes.POINTER(ctypes.c_double)],
        "c3_rp_predict_elastic": [ctypes.POINTER(C3RpTable), ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                  ctypes.c_double, ctypes.c_double, ctypes.POINTER(_int),
                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)],
        "c3_gemm_plan": [_i64, _i64, _i64, _int, ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)],
        "c3_cta_windows": [_int, ctypes.POINTER(C3CtaWindow), _int, ctypes.POINTER(_int)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = _int
    lib.c3_kernel_launches.argtypes = []
    lib.c3_kernel_launches.restype = ctypes.c_uint64
    lib.c3_strerror.restype = ctypes.c_char_p
    lib.c3_last_error.restype = ctypes.c_char_p
    return lib


_lib = _load()
EXPORTED = ("c3_get_device_info", "c3_strerror", "c3_last_error", "c3_status_check", "c3_shutdown",
            "c3_gemm", "c3_allgather", "c3_alltoall", "c3_allreduce", "c3_run", "c3_time", "c3_l2_flush", "c3_kernel_launches",
            "c3_gemm_noalloc", "c3_gemm_plan", "c3_selftest_wait", "c3_inject_fault", "c3_sp_predict",
            "c3_rp_predict", "c3_rp_predict_elastic", "c3_cta_windows")


def lib():
    return _lib


def _ptr(x):
    """Address of a tensor (``data_ptr``), an int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check(rc, where):
    if rc != C3_OK:
        raise C3Error(rc, where, _lib.c3_last_error().decode(errors="replace"))
    return rc


def c3_strerror(status: int) -> str:
    return _lib.c3_strerror(int(status)).decode()


def c3_last_error() -> str:
    return _lib.c3_last_error().decode(errors="replace")


def c3_get_device_info() -> dict:
    info = C3DeviceInfo()
    _check(_lib.c3_get_device_info(ctypes.byref(info)), "c3_get_device_info")
    return {n: getattr(info, n) for n, _ in C3DeviceInfo._fields_}


def c3_status_check(stream=None):
    return _check(_lib.c3_status_check(_stream(stream)), "c3_status_check")


def c3_kernel_launches() -> int:
    return int(_lib.c3_kernel_launches())


def c3_shutdown():
    return _check(_lib.c3_shutdown(), "c3_shutdown")


def c3_gemm(A, B, C, M, N, K, sm_budget=0, stream=None, check=True):
    rc = _lib.c3_gemm(_ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), int(sm_budget), _stream(stream))
    return _check(rc, "c3_gemm") if check else rc


def c3_allgather(shards, out, shard_bytes, nranks, engine=C3_ENGINE_SM, sm_budget=0, stream=None, check=True):
    arr = None
    if shards is not None:
        arr = (_vp * max(1, len(shards)))(*[_ptr(s) for s in shards])
    rc = _lib.c3_allgather(arr, _ptr(out), int(shard_bytes), int(nranks), int(engine), int(sm_budget),
                           _stream(stream))
    return _check(rc, "c3_allgather") if check else rc


def c3_alltoall(inp, out, block_bytes, nranks, engine=C3_ENGINE_SM, sm_budget=0, stream=None, check=True):
    rc = _lib.c3_alltoall(_ptr(inp), _ptr(out), int(block_bytes), int(nranks), int(engine), int(sm_budget),
                          _stream(stream))
    return _check(rc, "c3_alltoall") if check else rc


def c3_gemm_noalloc(A, B, C, M, N, K, sm_budget=0, stream=None, sync_check=True, check=True):
    """c3_gemm for callers that cannot allocate: scratch in a static device array."""
    rc = _lib.c3_gemm_noalloc(_ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), int(sm_budget),
                              _stream(stream), 1 if sync_check else 0)
    return _check(rc, "c3_gemm_noalloc") if check else rc


def c3_gemm_plan(M, N, K, sm_budget=0):
    """(BN, 128-row sub-tiles per CTA, CTAs) that c3_gemm would launch."""
    bn, ms, ctas = _int(), _int(), _int()
    _check(_lib.c3_gemm_plan(int(M), int(N), int(K), int(sm_budget), ctypes.byref(bn), ctypes.byref(ms),
                             ctypes.byref(ctas)), "c3_gemm_plan")
    return bn.value, ms.value, ctas.value


def c3_cta_windows(kernel):
    """[(cta, smid, t_start_s, t_end_s)] of the last run's GEMM (0) or SM collective (1) CTAs."""
    arr = (C3CtaWindow * 256)()
    n = _int()
    _check(_lib.c3_cta_windows(int(kernel), arr, 256, ctypes.byref(n)), "c3_cta_windows")
    return [(arr[i].cta, arr[i].smid, arr[i].t_start, arr[i].t_end) for i in range(n.value)]


def c3_selftest_wait(limit_ns, arrive, stream=None):
    """Status of a bounded device wait that succeeds (arrive=1) or runs out (arrive=0)."""
    return int(_lib.c3_selftest_wait(int(limit_ns), int(arrive), _stream(stream)))


def c3_inject_fault(site):
    """Arm a one-shot host-side failure at `site` (C3_FAULT_*; NONE disarms)."""
    _check(_lib.c3_inject_fault(int(site)), "c3_inject_fault")


def c3_sp_predict(gemm_ctas, coll_ctas):
    """1 if the collective should be launched first (fewer CTAs), else 0."""
    rc = _lib.c3_sp_predict(int(gemm_ctas), int(coll_ctas))
    if rc < 0:
        _check(rc, "c3_sp_predict")
    return rc


def c3_rp_predict(table, gemm_flops, gemm_bytes, coll_bytes, peak_flops, peak_bytes_per_s, elastic=False):
    """table: list of (sms, gemm_compute_slowdown, gemm_memory_slowdown, coll_slowdown).
    Returns (best_sms, predicted_seconds, [prediction per entry]).  elastic: the
    model of partitions that dissolve when the GEMM ends (c3_rp_predict_elastic)."""
    fn = _lib.c3_rp_predict_elastic if elastic else _lib.c3_rp_predict
    t = C3RpTable()
    t.n = len(table)
    for i, (k, gc, gm, co) in enumerate(table):
        t.sms[i], t.gemm_compute[i], t.gemm_memory[i], t.coll[i] = int(k), float(gc), float(gm), float(co)
    best, tp = _int(), ctypes.c_double()
    each = (ctypes.c_double * C3_RP_MAX)()
    _check(fn(ctypes.byref(t), float(gemm_flops), float(gemm_bytes), float(coll_bytes), float(peak_flops),
              float(peak_bytes_per_s), ctypes.byref(best), ctypes.byref(tp), each),
           "c3_rp_predict_elastic" if elastic else "c3_rp_predict")
    return best.value, tp.value, [each[i] for i in range(t.n)]


def c3_allreduce(inputs, out, count, nranks, engine=C3_ENGINE_SM, sm_budget=0, stream=None, check=True):
    arr = None
    if inputs is not None:
        arr = (_vp * max(1, len(inputs)))(*[_ptr(x) for x in inputs])
    rc = _lib.c3_allreduce(arr, _ptr(out), int(count), int(nranks), int(engine), int(sm_budget), _stream(stream))
    return _check(rc, "c3_allreduce") if check else rc


def c3_l2_flush(buf, nbytes, stream=None):
    return _check(_lib.c3_l2_flush(_ptr(buf), int(nbytes), _stream(stream)), "c3_l2_flush")


class Problem:
    """Owns the ctypes problem record and keeps the host shard-pointer array alive."""

    def __init__(self, A, B, C, M, N, K, coll, recv, unit_bytes, nranks=8, shards=None, send=None,
                 comm_sms=0, sm_kernel=C3_SMK_AUTO, flush=None, stream=None, coll_l2=C3_L2_NORMAL,
                 ce_variant=C3_CE_PER_SEGMENT, settle_us=0, peak_flops=0.0, peak_bytes_per_s=0.0,
                 coll_plateau_sm=0.0, coll_plateau_ce=0.0, ce_stage=None):
        self._shard_arr = None
        if shards is not None:
            self._shard_arr = (_vp * len(shards))(*[_ptr(s) for s in shards])
        fb, fn = (None, 0) if flush is None else (_ptr(flush), flush.numel() * flush.element_size())
        # the host-staged copy-engine variant's bounce buffer: a page-locked tensor or (address, bytes)
        if ce_stage is None:
            sb, sn = None, 0
        elif isinstance(ce_stage, tuple):
            sb, sn = ce_stage
        else:
            sb, sn = _ptr(ce_stage), ce_stage.numel() * ce_stage.element_size()
        self.rec = C3Problem(_ptr(A), _ptr(B), _ptr(C), int(M), int(N), int(K), int(coll),
                             self._shard_arr, _ptr(send), _ptr(recv), int(unit_bytes), int(nranks),
                             int(comm_sms), int(sm_kernel), int(coll_l2), int(ce_variant), fb, fn,
                             _stream(stream), int(settle_us), float(peak_flops), float(peak_bytes_per_s),
                             float(coll_plateau_sm), float(coll_plateau_ce), sb, int(sn))


def c3_run(problem: Problem, mode, sm_split=0, priority=0, check=True):
    t = C3Timing()
    rc = _lib.c3_run(ctypes.byref(problem.rec), int(mode), int(sm_split), int(priority), ctypes.byref(t))
    if check:
        _check(rc, "c3_run")
    return t.as_dict()


def c3_time(problem: Problem, mode, sm_split=0, priority=0, warmup=3, reps=9, check=True):
    arr = (C3Timing * max(1, reps))()
    rc = _lib.c3_time(ctypes.byref(problem.rec), int(mode), int(sm_split), int(priority), int(warmup),
                      int(reps), arr)
    if check:
        _check(rc, "c3_time")
    return [arr[i].as_dict() for i in range(reps)]
