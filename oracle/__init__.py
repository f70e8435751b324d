"""CPU oracle for C3 (GEMM overlapped with an all-gather / all-to-all).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this package.  It shares no code with the CUDA library
and imports nothing from it.

The arithmetic lives in ``c3_oracle.c`` (plain C, fp64, plain loops); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Each wrapper states the definition it follows; the C file cites the passages
of "Optimizing ML Concurrent Computation and Communication with GPU DMA
Engines" (pith.science review pages) that define them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "c3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_c3.so")
_lib = None
_lock = threading.Lock()

G_LONG, GC_EQUAL, C_LONG = 0, 1, 2
CLASS_NAMES = {G_LONG: "G-long", GC_EQUAL: "GC-equal", C_LONG: "C-long"}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc.  ``-ffp-contract=off`` keeps every product
    and sum a separately rounded fp64 operation on x86 and Arm alike."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, vp, ip = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [vp, vp, i64, i64, i64, vp, vp, ip]
            lib.oracle_gemm_entries.argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, vp, vp, ip]
            lib.oracle_allgather.argtypes = [vp, ip, i64, vp]
            lib.oracle_alltoall.argtypes = [vp, ip, i64, vp]
            lib.oracle_allreduce_f32.argtypes = [vp, ip, i64, vp, vp]
            lib.oracle_reduce_scatter_f32.argtypes = [vp, ip, i64, vp]
            lib.oracle_allreduce_f32.restype = ctypes.c_int
            lib.oracle_reduce_scatter_f32.restype = ctypes.c_int
            lib.oracle_c3_metrics.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double, dp,
                                              ctypes.POINTER(ctypes.c_int)]
            lib.oracle_c3_bounds.argtypes = [ctypes.c_double] * 7 + [ctypes.POINTER(ctypes.c_int)] * 2
            lib.oracle_c3_bounds.restype = ctypes.c_int
            for f in (lib.oracle_gemm, lib.oracle_gemm_entries, lib.oracle_allgather,
                      lib.oracle_alltoall, lib.oracle_c3_metrics):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _threads(nthreads):
    if nthreads:
        return int(nthreads)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as their uint16 bit patterns")
    return a


def gemm(A_bits, B_bits, nthreads=None):
    """C[m,n] = sum_k A[m,k] B[n,k] and S[m,n] = sum_k |A[m,k] B[n,k]| in fp64.

    ``A_bits`` is M x K, ``B_bits`` is N x K, both bf16 bit patterns (uint16).
    Returns (C, S) as float64 M x N arrays."""
    A, B = _u16(A_bits), _u16(B_bits)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A is M x K and B is N x K")
    C = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    rc = _load().oracle_gemm(A.ctypes.data, B.ctypes.data, M, N, K, C.ctypes.data, S.ctypes.data,
                             _threads(nthreads))
    if rc:
        raise ValueError(f"oracle_gemm rc={rc}")
    return C, S


def gemm_entries(A_bits, B_bits, mi, ni, nthreads=None):
    """The same two sums for the listed entries (mi[e], ni[e]) only."""
    A, B = _u16(A_bits), _u16(B_bits)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("A is M x K and B is N x K")
    mi = np.ascontiguousarray(mi, np.int64)
    ni = np.ascontiguousarray(ni, np.int64)
    if mi.shape != ni.shape:
        raise ValueError("index lists differ in length")
    C = np.empty(mi.shape, np.float64)
    S = np.empty(mi.shape, np.float64)
    rc = _load().oracle_gemm_entries(A.ctypes.data, B.ctypes.data, M, N, K, mi.ctypes.data,
                                     ni.ctypes.data, mi.size, C.ctypes.data, S.ctypes.data,
                                     _threads(nthreads))
    if rc:
        raise ValueError(f"oracle_gemm_entries rc={rc}")
    return C, S


def allgather(shards):
    """Rank-order concatenation of equal-size byte shards (list of uint8 arrays)."""
    shards = [np.ascontiguousarray(s).view(np.uint8).reshape(-1) for s in shards]
    n = len(shards)
    size = shards[0].size if n else 0
    if any(s.size != size for s in shards):
        raise ValueError("shards differ in size")
    out = np.empty(n * size, np.uint8)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[s.ctypes.data for s in shards])
    rc = _load().oracle_allgather(ptrs, n, size, out.ctypes.data)
    if rc:
        raise ValueError(f"oracle_allgather rc={rc}")
    return out


def alltoall(buf, nranks):
    """Block transpose of an nranks x nranks grid of equal blocks (bytes)."""
    b = np.ascontiguousarray(buf).view(np.uint8).reshape(-1)
    if b.size % (nranks * nranks):
        raise ValueError("buffer is not nranks^2 equal blocks")
    out = np.empty_like(b)
    rc = _load().oracle_alltoall(b.ctypes.data, nranks, b.size // (nranks * nranks), out.ctypes.data)
    if rc:
        raise ValueError(f"oracle_alltoall rc={rc}")
    return out


def _f32_list(bufs):
    bufs = [np.ascontiguousarray(b, np.float32).reshape(-1) for b in bufs]
    n = bufs[0].size if bufs else 0
    if any(b.size != n for b in bufs):
        raise ValueError("rank buffers differ in length")
    return bufs, n, (ctypes.c_void_p * max(1, len(bufs)))(*[b.ctypes.data for b in bufs])


def allreduce(bufs):
    """All-reduce of R fp32 vectors: returns (out, exact64) where out is
    R x count, every row the fp32 sum in rank order, and exact64 the fp64 sum."""
    bufs, n, ptrs = _f32_list(bufs)
    out = np.empty((len(bufs), n), np.float32)
    ex = np.empty(n, np.float64)
    rc = _load().oracle_allreduce_f32(ptrs, len(bufs), n, out.ctypes.data, ex.ctypes.data)
    if rc:
        raise ValueError(f"oracle_allreduce_f32 rc={rc}")
    return out, ex


def reduce_scatter(bufs, out=None):
    """Reduce-scatter of R fp32 vectors into an R x count array: row r gets
    chunk r of the rank-order fp32 sum; other positions keep `out`'s values."""
    bufs, n, ptrs = _f32_list(bufs)
    if out is None:
        out = np.zeros((len(bufs), n), np.float32)
    out = np.ascontiguousarray(out, np.float32)
    rc = _load().oracle_reduce_scatter_f32(ptrs, len(bufs), n, out.ctypes.data)
    if rc:
        raise ValueError(f"oracle_reduce_scatter_f32 rc={rc}")
    return out


def c3_metrics(t_gemm, t_comm, t_conc):
    """Ideal / realized speedup, share of the ideal gain, ratio and class."""
    out = (ctypes.c_double * 6)()
    cls = ctypes.c_int()
    rc = _load().oracle_c3_metrics(float(t_gemm), float(t_comm), float(t_conc), out, ctypes.byref(cls))
    if rc:
        raise ValueError(f"oracle_c3_metrics rc={rc}")
    return {"s_ideal": out[0], "s_real": out[1], "pct_ideal_gain": out[2], "pct_ideal_ratio": out[3],
            "t_serial": out[4], "t_ideal": out[5], "class": CLASS_NAMES[cls.value]}


GEMM_BOUND_NAMES = {-1: "unknown", 0: "compute", 1: "memory"}
COLL_BOUND_NAMES = {-1: "unknown", 0: "latency", 1: "bandwidth"}


def c3_bounds(gemm_flops, gemm_bytes, peak_flops, peak_bytes_per_s, coll_bytes, t_comm, plateau_bytes_per_s):
    """The taxonomy's other two axes: ("compute" | "memory" | "unknown",
    "latency" | "bandwidth" | "unknown").  Memory-bound GEMM when
    flops / bytes < peak_flops / peak_bytes_per_s; bandwidth-bound collective
    when coll_bytes / t_comm >= plateau / 2.  A peak or plateau <= 0 gives
    "unknown" on its axis."""
    g, c = ctypes.c_int(), ctypes.c_int()
    rc = _load().oracle_c3_bounds(float(gemm_flops), float(gemm_bytes), float(peak_flops), float(peak_bytes_per_s),
                                  float(coll_bytes), float(t_comm), float(plateau_bytes_per_s), ctypes.byref(g),
                                  ctypes.byref(c))
    if rc:
        raise ValueError(f"oracle_c3_bounds rc={rc}")
    return GEMM_BOUND_NAMES[g.value], COLL_BOUND_NAMES[c.value]
