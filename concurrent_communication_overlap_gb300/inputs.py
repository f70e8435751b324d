"""Seeded synthetic inputs and the C3 workload table.

This module is shared by the CUDA-path tests, the oracle tests and the
benchmark.  It holds only input generation and workload shapes: none of the
arithmetic of the method (no GEMM, no collective, no speedup formula).

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) in counter form: word i of stream ``seed`` is
output i+1 of splitmix64 started from state seed * 2^32, i.e. the mix function
applied to seed * 2^32 + (i + 1) * 0x9E3779B97F4A7C15.  Uniform doubles take
the top 53 bits; normals use the Box-Muller transform on consecutive pairs.  Floating-point samples
are drawn in fp64, rounded to fp32 by numpy and then to bf16 with
round-to-nearest-even; the bf16 bit patterns (uint16) are what both the GPU
path and the oracle read.  Buffer ``b`` of a workload uses seed ``1000 + b``.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function; uint64 arithmetic wraps."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _words(seed: int, start: int, count: int) -> np.ndarray:
    base = np.uint64((int(seed) << 32) & 0xFFFFFFFFFFFFFFFF)
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + ctr * _GOLDEN)


def _chunked(n: int, fn, out: np.ndarray, threads: int = 0):
    """Fill ``out[a:b] = fn(a, b)`` chunk by chunk on a thread pool (numpy
    releases the GIL inside its ufuncs)."""
    spans = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for a, b in spans:
            out[a:b] = fn(a, b)
        return out

    def work(span):
        a, b = span
        out[a:b] = fn(a, b)

    import os
    workers = threads or min(16, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 4)
    with ThreadPoolExecutor(max_workers=max(1, workers)) as ex:
        list(ex.map(work, spans))
    return out


def _uniform64(seed, a, b, lo, hi):
    """Samples a..b-1 of the uniform stream, fp64 on [lo, hi) from the top 53 bits."""
    u = (_words(seed, a, b - a) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))
    return lo + (hi - lo) * u


def _normal64(seed, a, b, mean, std):
    """Samples a..b-1 of the normal stream: Box-Muller on word pairs (2i, 2i+1)."""
    w = _words(seed, 2 * a, 2 * (b - a)).reshape(-1, 2)
    u1 = ((w[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / (1 << 53))  # (0, 1]
    u2 = (w[:, 1] >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))          # [0, 1)
    return mean + std * (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2))


def uniform(seed: int, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    """n fp64 samples, uniform on [lo, hi)."""
    return _chunked(n, lambda a, b: _uniform64(seed, a, b, lo, hi), np.empty(n, np.float64))


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n fp64 samples, N(mean, std^2)."""
    return _chunked(n, lambda a, b: _normal64(seed, a, b, mean, std), np.empty(n, np.float64))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.
    NaN stays a quiet NaN."""
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    bits = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return bits


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_uniform(seed: int, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    _chunked(n, lambda a, b: f32_to_bf16_bits(_uniform64(seed, a, b, lo, hi).astype(np.float32)), out)
    return out.reshape(shape)


def bf16_normal(seed: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    _chunked(n, lambda a, b: f32_to_bf16_bits(_normal64(seed, a, b, mean, std).astype(np.float32)), out)
    return out.reshape(shape)


def random_u16(seed: int, n: int) -> np.ndarray:
    """n raw 16-bit patterns (every bf16 encoding, NaN and Inf included)."""
    out = np.empty(n, np.uint16)
    _chunked(n, lambda a, b: (_words(seed, a, b - a) >> np.uint64(48)).astype(np.uint16), out)
    return out


def random_bytes(seed: int, nbytes: int) -> np.ndarray:
    """Random payload of nbytes (uint8), drawn as 16-bit words."""
    words = random_u16(seed, (nbytes + 1) // 2)
    return words.view(np.uint8)[:nbytes].copy() if nbytes % 2 else words.view(np.uint8)


# ---------------------------------------------------------------------------
# Workloads.  The GEMM is C = A B^T with A (M x K) activations and B (N x K)
# weights; the collective runs over 8 virtual ranks inside one device.
# ---------------------------------------------------------------------------

MiB = 1 << 20


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    a_dist: tuple      # ("uniform", lo, hi) or ("normal", mean, std)
    b_dist: tuple
    coll: str          # "allgather", "alltoall" or "allreduce"
    nranks: int
    unit_bytes: int    # shard bytes (all-gather), block bytes (all-to-all), fp32 vector bytes (all-reduce)
    payload: str       # "u16" (random 16-bit patterns) or a bf16 distribution tag
    description: str

    @property
    def coll_bytes(self) -> int:
        """Bytes of the collective's output (= bytes of its input)."""
        if self.coll in ("allgather", "allreduce"):
            return self.nranks * self.unit_bytes
        return self.nranks * self.nranks * self.unit_bytes

    @property
    def coll_traffic_bytes(self) -> int:
        """Bytes the collective must read and write at least: 2x its size for
        the copies; for the all-reduce, every rank's vector read once and every
        rank's row written once (the SM engine's one pass moves exactly that;
        the copy-engine form, a reduce-scatter and then copies of its chunks,
        moves (3R - 1) rows)."""
        if self.coll == "allreduce":
            return 2 * self.nranks * self.unit_bytes
        return 2 * self.coll_bytes

    @property
    def gemm_flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def gemm_bytes(self) -> int:
        return 2 * self.M * self.K + 2 * self.N * self.K + 4 * self.M * self.N


WORKLOADS = {
    "tiny_ag": Workload("tiny_ag", 512, 512, 512, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0),
                        "allgather", 8, 1 * MiB, "u16",
                        "bf16 GEMM 512^3 (U[-1,1]) with an 8-rank all-gather of 8 x 1 MiB"),
    "tiny_a2a": Workload("tiny_a2a", 512, 512, 512, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0),
                         "alltoall", 8, 128 * 1024, "u16",
                         "bf16 GEMM 512^3 (U[-1,1]) with an 8x8 all-to-all of 128 KiB blocks"),
    "mem_ag": Workload("mem_ag", 256, 28672, 8192, ("normal", 0.0, 1.0), ("normal", 0.0, 0.02),
                       "allgather", 8, 16 * MiB, "normal0.02",
                       "memory-bound bf16 GEMM 256x28672x8192 with an 8-rank all-gather of an "
                       "8192x8192 bf16 weight (8 x 16 MiB)"),
    "ffn70_ag": Workload("ffn70_ag", 8192, 28672, 8192, ("normal", 0.0, 1.0), ("normal", 0.0, 0.02),
                         "allgather", 8, 56 * MiB, "normal0.02",
                         "Llama-70B-FFN-shaped bf16 GEMM 8192x28672x8192 with an 8-rank all-gather "
                         "of an 8192x28672 bf16 weight (8 x 56 MiB)"),
    "tiny_ar": Workload("tiny_ar", 512, 512, 512, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0),
                        "allreduce", 8, 1 * MiB, "f32normal",
                        "bf16 GEMM 512^3 (U[-1,1]) with an 8-rank all-reduce of 8 x 1 MiB fp32 vectors"),
    "mem_ar": Workload("mem_ar", 256, 28672, 8192, ("normal", 0.0, 1.0), ("normal", 0.0, 0.02),
                       "allreduce", 8, 16 * MiB, "f32normal",
                       "memory-bound bf16 GEMM 256x28672x8192 with an 8-rank all-reduce of 8 x 16 MiB fp32 "
                       "gradients (one pass on SMs; on the copy engine a reduce-scatter on SMs, then memcpy)"),
    "l405_a2a": Workload("l405_a2a", 8192, 53248, 16384, ("normal", 0.0, 1.0), ("normal", 0.0, 0.02),
                         "alltoall", 8, 8 * MiB, "u16",
                         "Llama-405B-shaped bf16 GEMM 8192x53248x16384 with an 8x8 all-to-all of "
                         "8 MiB blocks"),
}


def sweep_workloads(coll: str, lo_bytes: int = MiB, hi_bytes: int = 1 << 30):
    """8192^3 GEMM with a collective whose total size doubles from lo to hi."""
    out = []
    total = lo_bytes
    while total <= hi_bytes:
        unit = total // 8 if coll == "allgather" else total // 64
        out.append(Workload(f"sweep_{coll}_{total // 1024}k", 8192, 8192, 8192, ("normal", 0.0, 1.0),
                            ("normal", 0.0, 0.02), coll, 8, unit, "u16",
                            f"bf16 GEMM 8192^3 with a {total / MiB:g} MiB {coll}"))
        total *= 2
    return out


def gemm_operands(w: Workload, M=None, N=None, K=None):
    """bf16 bit patterns of A (M x K, seed 1000) and B (N x K, seed 1001)."""
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K

    def draw(seed, shape, dist):
        if dist[0] == "uniform":
            return bf16_uniform(seed, shape, dist[1], dist[2])
        return bf16_normal(seed, shape, dist[1], dist[2])

    return draw(1000, (M, K), w.a_dist), draw(1001, (N, K), w.b_dist)


def coll_payload(w: Workload):
    """The collective's input: a list of nranks shard byte arrays (all-gather,
    seeds 1002 + r), one send buffer of nranks^2 blocks (all-to-all, seed
    1002), or nranks fp32 N(0,1) vectors (all-reduce, seeds 1002 + r)."""
    if w.coll == "allreduce":
        return [normal(1002 + r, w.unit_bytes // 4).astype(np.float32) for r in range(w.nranks)]
    if w.coll == "allgather":
        shards = []
        for r in range(w.nranks):
            if w.payload == "u16":
                s = random_bytes(1002 + r, w.unit_bytes)
            else:
                s = bf16_normal(1002 + r, (w.unit_bytes // 2,), 0.0, 0.02).view(np.uint8)
            shards.append(s)
        return shards
    return random_bytes(1002, w.coll_bytes)
