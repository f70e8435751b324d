"""Pins for the CPU oracle, each against something other than the oracle itself:
hand-listed integer products (brute force in exact rational arithmetic), closed
forms (identity, rank one), involutions, tag patterns with a closed-form
location, and the golden fixtures under tests/golden/.  Each test is chosen so
that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong bf16 decode) fails it."""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from concurrent_communication_overlap_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_exact(x: float) -> int:
    """bf16 bits of a value that is exactly representable in bf16 (checked)."""
    u = struct.unpack("<I", struct.pack("<f", x))[0]
    assert u & 0xFFFF == 0, f"{x} is not exact in bf16"
    return u >> 16


def to_bits(rows):
    return np.array([[bf16_bits_exact(v) for v in r] for r in rows], np.uint16)


# ---------------------------------------------------------------- GEMM pins

A_SMALL = [[1, -2, 3, 0.5],
           [4, 0, -1.5, 2],
           [-3, 5, 2, -0.25]]                 # M=3, K=4
B_SMALL = [[2, 1, 0, -1],
           [-1, 3, 2, 4],
           [0.5, -0.5, 1, 1],
           [7, 0, -2, 1.5],
           [1, 1, 1, 1]]                      # N=5, K=4 (weight layout N x K)


def brute(A, B):
    """Exact C[m][n] = sum_k A[m][k] B[n][k] and S = sum |.| with Fractions."""
    C = [[sum(Fraction(a) * Fraction(b) for a, b in zip(ar, br)) for br in B] for ar in A]
    S = [[sum(abs(Fraction(a) * Fraction(b)) for a, b in zip(ar, br)) for br in B] for ar in A]
    return C, S


def test_gemm_brute_force_nonsquare():
    C, S = oracle.gemm(to_bits(A_SMALL), to_bits(B_SMALL), nthreads=2)
    Ce, Se = brute(A_SMALL, B_SMALL)
    assert C.shape == (3, 5)
    for m in range(3):
        for n in range(5):
            assert C[m, n] == float(Ce[m][n]), (m, n)
            assert S[m, n] == float(Se[m][n]), (m, n)


def test_gemm_hand_value():
    # Row 0 of A times row 1 of B, worked by hand:
    # 1*(-1) + (-2)*3 + 3*2 + 0.5*4 = -1 - 6 + 6 + 2 = 1 ; |.| sum = 1 + 6 + 6 + 2 = 15
    C, S = oracle.gemm(to_bits(A_SMALL), to_bits(B_SMALL))
    assert C[0, 1] == 1.0 and S[0, 1] == 15.0
    # Row 2 of A times row 3 of B: -21 + 0 - 4 - 0.375 = -25.375 ; |.| = 21 + 4 + 0.375
    assert C[2, 3] == -25.375 and S[2, 3] == 25.375


def test_gemm_4x4_integers():
    A = [[1, 2, 3, 4], [5, 6, 7, 8], [-1, -2, -3, -4], [0, 1, 0, -1]]
    B = [[1, 0, 0, 0], [0, 2, 0, 0], [1, 1, 1, 1], [4, -3, 2, -1]]
    C, S = oracle.gemm(to_bits(A), to_bits(B))
    Ce, Se = brute(A, B)
    assert np.array_equal(C, np.array(Ce, dtype=np.float64))
    assert np.array_equal(S, np.array(Se, dtype=np.float64))


def test_gemm_identity():
    # A . I^T = A exactly, for random bf16 A (values far from over/underflow).
    K = 48
    A = I.bf16_uniform(7, (37, K), -3.0, 3.0)
    Ident = np.zeros((K, K), np.uint16)
    Ident[np.arange(K), np.arange(K)] = 0x3F80
    C, S = oracle.gemm(A, Ident)
    Af = I.bf16_bits_to_f32(A).astype(np.float64)
    assert np.array_equal(C, Af)
    assert np.array_equal(S, np.abs(Af))


def test_gemm_rank_one_closed_form():
    # A = u 1^T, B = v 1^T  =>  C = K u v^T and S = K |u| |v|, exact for small integers.
    M, N, K = 6, 9, 1000
    u = np.arange(M) - 2.0
    v = 2.0 * np.arange(N) - 7.0
    A = np.repeat(to_bits([[x] for x in u]), K, axis=1)
    B = np.repeat(to_bits([[x] for x in v]), K, axis=1)
    C, S = oracle.gemm(A, B)
    assert np.array_equal(C, K * np.outer(u, v))
    assert np.array_equal(S, K * np.outer(np.abs(u), np.abs(v)))


def test_gemm_operand_order_matters():
    # C = A B^T, not A^T B nor B A^T: the transposed product of these operands
    # differs, so a swapped or transposed operand would be caught.
    C, _ = oracle.gemm(to_bits(A_SMALL), to_bits(B_SMALL))
    Ct, _ = oracle.gemm(to_bits(B_SMALL), to_bits(A_SMALL))
    assert np.array_equal(Ct, C.T)  # (B A^T) = (A B^T)^T, by the definition
    assert not np.array_equal(C[:3, :3], C[:3, :3].T)


def test_gemm_bf16_decode_special_values():
    # Smallest bf16 subnormal 0x0001 = 2^-133, negative zero, largest finite 0x7F7F.
    A = np.array([[0x0001, 0x8000, 0x7F7F]], np.uint16)
    B = np.array([[0x4000, 0x3F80, 0x0000]], np.uint16)      # 2, 1, 0
    C, S = oracle.gemm(A, B)
    assert C[0, 0] == 2.0 ** -132
    assert S[0, 0] == 2.0 ** -132


def test_gemm_long_sum_is_exact_for_integers():
    # K = 4096 terms of +-1 * small ints: the fp64 sum is exact; closed form below.
    K = 4096
    k = np.arange(K)
    a = np.where(k % 2 == 0, 1.0, -1.0)
    b = (k % 7).astype(np.float64)
    C, S = oracle.gemm(to_bits([a]), to_bits([b]))
    assert C[0, 0] == float(np.sum(a * b)) and S[0, 0] == float(np.sum(b))
    # closed form independent of numpy: pairs (2j, 2j+1) contribute (2j%7 - (2j+1)%7)
    expect = sum((2 * j) % 7 - (2 * j + 1) % 7 for j in range(K // 2))
    assert C[0, 0] == expect


def test_gemm_empty_k_and_entries():
    A = np.zeros((3, 0), np.uint16)
    B = np.zeros((2, 0), np.uint16)
    C, S = oracle.gemm(A, B)
    assert np.array_equal(C, np.zeros((3, 2))) and np.array_equal(S, np.zeros((3, 2)))
    # entries: brute force on listed positions
    Ce, Se = brute(A_SMALL, B_SMALL)
    mi, ni = np.array([2, 0, 1, 2]), np.array([4, 0, 3, 1])
    c, s = oracle.gemm_entries(to_bits(A_SMALL), to_bits(B_SMALL), mi, ni)
    for e in range(4):
        assert c[e] == float(Ce[mi[e]][ni[e]]) and s[e] == float(Se[mi[e]][ni[e]])
    with pytest.raises(ValueError):
        oracle.gemm_entries(to_bits(A_SMALL), to_bits(B_SMALL), np.array([3]), np.array([0]))


def test_gemm_thread_count_does_not_change_result():
    A = I.bf16_normal(11, (33, 64))
    B = I.bf16_normal(12, (17, 64))
    C1, S1 = oracle.gemm(A, B, nthreads=1)
    C7, S7 = oracle.gemm(A, B, nthreads=7)
    assert np.array_equal(C1, C7) and np.array_equal(S1, S7)


# ---------------------------------------------------------------- collective pins

def tag_shard(r, nbytes):
    """byte i of rank r: a closed form that differs between ranks and offsets."""
    i = np.arange(nbytes, dtype=np.int64)
    return ((r * 37 + i * 11 + (i >> 8) * 3) & 0xFF).astype(np.uint8)


@pytest.mark.parametrize("nranks,nbytes", [(8, 4096), (2, 48), (1, 16), (8, 0), (3, 1000)])
def test_allgather_rank_order_concatenation(nranks, nbytes):
    shards = [tag_shard(r, nbytes) for r in range(nranks)]
    out = oracle.allgather(shards)
    assert out.size == nranks * nbytes
    for r in range(nranks):
        # closed form at the location rank r must occupy
        assert np.array_equal(out[r * nbytes:(r + 1) * nbytes], tag_shard(r, nbytes)), r


def test_allgather_random_payload_matches_concatenation():
    shards = [I.random_bytes(1002 + r, 1 << 12) for r in range(8)]
    out = oracle.allgather(shards)
    assert np.array_equal(out, np.concatenate(shards))


def block_tag(i, j, nbytes):
    k = np.arange(nbytes, dtype=np.int64)
    return ((i * 16 + j + k * 7) & 0xFF).astype(np.uint8)


@pytest.mark.parametrize("nranks,block", [(8, 256), (2, 16), (4, 3), (1, 64)])
def test_alltoall_block_tags(nranks, block):
    send = np.concatenate([block_tag(i, j, block) for i in range(nranks) for j in range(nranks)])
    out = oracle.alltoall(send, nranks)
    for j in range(nranks):          # receiving rank
        for i in range(nranks):      # its slot i holds what rank i sent to j
            got = out[(j * nranks + i) * block:(j * nranks + i + 1) * block]
            assert np.array_equal(got, block_tag(i, j, block)), (i, j)


def test_alltoall_twice_is_identity():
    x = I.random_bytes(1002, 64 * 1000)
    y = oracle.alltoall(x, 8)
    assert not np.array_equal(x, y)
    assert np.array_equal(oracle.alltoall(y, 8), x)


def test_alltoall_single_rank_and_diagonal():
    x = I.random_bytes(5, 8 * 8 * 32)
    assert np.array_equal(oracle.alltoall(x[:32], 1), x[:32])
    y = oracle.alltoall(x, 8)
    for i in range(8):  # diagonal blocks stay in place
        s = slice((i * 8 + i) * 32, (i * 8 + i + 1) * 32)
        assert np.array_equal(y[s], x[s])


# ---------------------------------------------------------------- C3 metric pins

def load_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_c3_speedup_closed_forms():
    for r in load_rows("c3_speedup_closed_forms.txt"):
        tg, tc, tconc, s_ideal, s_real, gain, ratio = map(float, r)
        m = oracle.c3_metrics(tg, tc, tconc)
        assert m["s_ideal"] == pytest.approx(s_ideal, rel=1e-14)
        assert m["s_real"] == pytest.approx(s_real, rel=1e-14)
        assert m["pct_ideal_gain"] == pytest.approx(gain, rel=1e-12, abs=1e-15)
        assert m["pct_ideal_ratio"] == pytest.approx(ratio, rel=1e-14)
        assert m["t_serial"] == tg + tc and m["t_ideal"] == max(tg, tc)


def test_c3_taxonomy_thresholds():
    for tg, tc, cls in load_rows("taxonomy_thresholds.txt"):
        assert oracle.c3_metrics(float(tg), float(tc), 1.0)["class"] == cls, (tg, tc)


def test_c3_metrics_reject_nonpositive_times():
    for bad in [(0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 1, 1), (float("nan"), 1, 1)]:
        with pytest.raises(ValueError):
            oracle.c3_metrics(*bad)


def test_c3_gain_fraction_reading_fits_the_pages_numbers():
    # The pages report an average of 21% of ideal at baseline and all-to-all
    # speedups of 1.05x over serial (abstract; "If this is right" list).  With
    # S_ideal <= 2, the plain ratio S_real / S_ideal of a 1.05x scenario is at
    # least 52.5%, so a 21% figure only fits the gain fraction.  This checks
    # the arithmetic behind that reading for the extreme ideal of 2.
    m = oracle.c3_metrics(1.0, 1.0, 2.0 / 1.05)
    assert m["s_real"] == pytest.approx(1.05)
    assert m["pct_ideal_ratio"] >= 0.525 - 1e-12
    assert m["pct_ideal_gain"] == pytest.approx(0.05, rel=1e-9)


# ---------------------------------------------------------------- generator pins

def test_splitmix64_known_answers():
    # Published first outputs of splitmix64 from state 0.
    w = I._words(0, 0, 3)
    assert [int(x) for x in w] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generators_are_reproducible_and_chunk_independent():
    a = I.normal(9, (1 << 22) + 5)
    b = I.normal(9, 5)
    assert np.array_equal(a[:5], b)
    assert np.array_equal(I.random_u16(3, 100), I.random_u16(3, 100))
    assert not np.array_equal(I.random_u16(3, 100), I.random_u16(4, 100))


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1+3*2^-8 ties -> 1+2^-6
    assert list(I.f32_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F80]


def test_distributions_have_the_stated_moments():
    u = I.bf16_bits_to_f32(I.bf16_uniform(1000, (1 << 16,), -1.0, 1.0))
    assert -1.0 <= u.min() and u.max() <= 1.0 and abs(u.mean()) < 0.01
    z = I.bf16_bits_to_f32(I.bf16_normal(1001, (1 << 16,), 0.0, 0.02))
    assert abs(z.std() - 0.02) < 0.001 and abs(z.mean()) < 0.001


# ---------------------------------------------------------------- all-reduce pins

def test_allreduce_integer_sums_exact_and_replicated():
    R, n = 8, 40
    bufs = [np.arange(n, dtype=np.float32) * (q + 1) - q for q in range(R)]
    out, ex = oracle.allreduce(bufs)
    # closed form: sum_q (i*(q+1) - q) = i*R(R+1)/2 - R(R-1)/2
    expect = np.arange(n) * (R * (R + 1) // 2) - R * (R - 1) // 2
    assert out.shape == (R, n)
    for r in range(R):
        assert np.array_equal(out[r], expect.astype(np.float32))
    assert np.array_equal(ex, expect.astype(np.float64))


def test_allreduce_rank_order_is_the_fp32_order():
    # 1e8 + 1 + 1 - 1e8 ... : order matters in fp32; the rank order fixes it
    bufs = [np.array([1e8], np.float32), np.array([1.0], np.float32), np.array([1.0], np.float32),
            np.array([-1e8], np.float32)]
    out, ex = oracle.allreduce(bufs)
    f = np.float32(0)
    for b in bufs:
        f = np.float32(f + b[0])
    assert out[0, 0] == f == np.float32(0.0)       # 1e8+1 rounds to 1e8 in fp32, twice
    assert ex[0] == 2.0


def test_allreduce_one_rank_is_identity_and_one_hot():
    x = I.normal(3, 17).astype(np.float32)
    out, _ = oracle.allreduce([x])
    assert np.array_equal(out[0], x)
    R, n = 4, 8
    bufs = [np.zeros(n, np.float32) for _ in range(R)]
    for q in range(R):
        bufs[q][2 * q] = q + 1.5
    out, _ = oracle.allreduce(bufs)
    assert np.array_equal(out[1], np.array([1.5, 0, 2.5, 0, 3.5, 0, 4.5, 0], np.float32))


def test_reduce_scatter_keeps_only_own_chunk():
    R, n = 4, 12
    bufs = [np.full(n, q + 1, np.float32) for q in range(R)]
    out = oracle.reduce_scatter(bufs, np.full((R, n), -7.0, np.float32))
    for r in range(R):
        own = slice(r * 3, (r + 1) * 3)
        assert np.array_equal(out[r, own], np.full(3, 10.0, np.float32))   # 1+2+3+4
        mask = np.ones(n, bool)
        mask[own] = False
        assert np.all(out[r, mask] == -7.0)


def test_c3_taxonomy_bounds_golden_rows():
    for row in load_rows("taxonomy_bounds.txt"):
        if row[0] == "gemm":
            flops, nbytes, pf, pw = map(float, row[1:5])
            g, _ = oracle.c3_bounds(flops, nbytes, pf, pw, 1.0, 1.0, 1.0)
            assert g == row[5], row
        else:
            cb, t, plat = map(float, row[1:4])
            _, c = oracle.c3_bounds(1.0, 1.0, 1.0, 1.0, cb, t, plat)
            assert c == row[4], row


def test_c3_taxonomy_bounds_follow_the_stated_ratios():
    # the GEMM axis moves with the arithmetic intensity, not with flops or bytes alone
    assert oracle.c3_bounds(1e12, 1e10, 1e15, 1e13, 1, 1, 1)[0] == "compute"     # I = 100 = ridge
    assert oracle.c3_bounds(1e12, 2e10, 1e15, 1e13, 1, 1, 1)[0] == "memory"      # I = 50 < 100
    assert oracle.c3_bounds(2e12, 2e10, 1e15, 1e13, 1, 1, 1)[0] == "compute"     # I = 100 again
    # the collective axis: halving the time at fixed size crosses into bandwidth-bound
    assert oracle.c3_bounds(1, 1, 1, 1, 1e6, 4e-6, 1e12)[1] == "latency"          # 0.25 of plateau
    assert oracle.c3_bounds(1, 1, 1, 1, 1e6, 1e-6, 1e12)[1] == "bandwidth"        # 1.0 of plateau
    for bad in [(0, 1, 1, 1, 1, 1, 1), (1, 0, 1, 1, 1, 1, 1), (1, 1, 1, 1, 0, 1, 1), (1, 1, 1, 1, 1, 0, 1)]:
        with pytest.raises(ValueError):
            oracle.c3_bounds(*bad)
