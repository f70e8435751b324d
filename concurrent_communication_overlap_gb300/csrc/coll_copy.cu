// coll_copy.cu -- SM kernels that carry the emulated collectives.
//
// Both collectives are lists of equal-size byte segments (src -> dst):
//   all-gather: segment r = shard r -> out + r * shard_bytes           (r < nranks)
//   all-to-all: segment (i, j) = in + (i*R + j) * B -> out + (j*R + i) * B
// (the all-gather / all-to-all pair of "Optimizing ML Concurrent Computation
// and Communication with GPU DMA Engines", whose CU-based library kernels
// these stand in for; the skeptic's "concrete_test" fixes the all-gather as
// rank-order concatenation of every rank's initial buffer).
//
// Two flavours:
//   vec  -- every thread moves UNROLL 16-byte vectors per round trip (all loads
//           issued before the stores).  No shared memory, 512 threads, <= 64
//           registers, so two CTAs or one GEMM CTA can share an SM with it.
//           A launch may reserve dynamic shared memory it never touches, which
//           keeps other CTAs off its SM (SM partitioning).
//   bulk -- one elected thread streams 32 KiB chunks global -> shared -> global
//           with cp.async.bulk through a 6-deep shared-memory ring (192 KiB in
//           flight per SM, no register staging).  One CTA per SM by its
//           shared-memory footprint.
// Each flavour has a streaming variant whose loads and stores carry an L2
// evict-first policy (and skip L1), the software counterpart of the pages'
// observation that DMA transfers bypass the caches.
#include "c3_device.cuh"
#include "c3_internal.h"

namespace c3 {

constexpr int kVecThreads = 512;
constexpr int kVecUnroll = 8;
constexpr uint32_t kBulkChunk = 32 * 1024;
constexpr int kBulkBufs = 6;
constexpr int kBulkThreads = 32;
constexpr int kBulkSmem = kBulkBufs * kBulkChunk + 1024;

__device__ __forceinline__ uint4 ld_vec(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_vec(uint8_t* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
// Streaming forms: no L1 allocation, L2 lines marked evict-first, so the
// collective's bytes (touched once) do not push a concurrent GEMM's operands
// out of L2.
__device__ __forceinline__ uint4 ld_vec_stream(const uint8_t* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_vec_stream(uint8_t* p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// The gate of a collective launch part that must start only on SMs a GEMM has
// left: the hardware may dispatch that launch's CTAs before the GEMM's own
// (both wait for the same free SMs), and such a CTA, holding its SM while the
// GEMM still has CTAs waiting, would turn the run serial.  Every GEMM CTA adds
// itself to st->gemm_started as it starts; a gated CTA that finds fewer than
// gate_need started leaves at once, without work (one read, no waiting; a
// stale read only makes it leave when it could have stayed).  The whole CTA
// takes the same decision (one value, broadcast through a barrier reduction).
__device__ __forceinline__ bool gate_closed(const DevStatus* st, unsigned gate_need) {
    if (gate_need == 0 || st == nullptr) return false;
    int closed = 0;
    if (threadIdx.x == 0) closed = *reinterpret_cast<const volatile unsigned*>(&st->gemm_started) < gate_need;
    return __syncthreads_or(closed) != 0;
}

// The last CTA of a launch group to finish puts the group's work counter back
// to zero, so the slot is clean for its next user.
__device__ __forceinline__ void group_done(unsigned int* work, int total_ctas) {
    __threadfence();
    if (atomicAdd(&work[1], 1u) == (unsigned)total_ctas - 1u) {
        atomicExch(&work[0], 0u);
        atomicExch(&work[1], 0u);
    }
}

// Work of the vec kernel, in 4 KiB pieces of one segment (kVecUnroll 16-byte
// vectors per lane of a warp: every lane issues its kVecUnroll loads, each 512
// contiguous bytes across the warp, before its stores).  The group's first
// launch part (F CTAs of 16 warps) starts on fixed pieces, in up to four rounds
// of 16 F: in round j, warp w of CTA b moves piece j * 16F + w * F + b --
// interleaved across CTAs, so even a small collective spreads over every SM of
// the part -- with as many rounds as the collective fills (one for a
// collective of at most 16F pieces, four for a large one).  The pieces after
// the fixed rounds are claimed from the group's counter (work[0]) four at a
// time (16 KiB), so a warp that shares its SM with a GEMM CTA, or a CTA that
// starts late because its SM was busy, simply moves fewer.  Lane 0 claims the
// warp's next four while the current four are copied and broadcasts the claim
// by shuffle.  The kernel uses no shared memory, so it still fits beside a
// GEMM CTA.  A CTA none of whose warps found work leaves at once and records
// no residency.
constexpr uint64_t kVecPiece = 32 * kVecUnroll;  // vectors per piece (4 KiB)
constexpr unsigned kVecClaim = 4;                // pieces per claim
constexpr int kVecWarps = kVecThreads / 32;

template <bool kStream>
__global__ void __launch_bounds__(kVecThreads, 2)
    copy_vec_kernel(SegTable t, DevStatus* st, unsigned int* work, int cta_base, int total_ctas,
                    unsigned static_units, unsigned gate_need) {
    const unsigned long long t_enter = globaltimer();
    if (gate_closed(st, gate_need)) {
        if (threadIdx.x == 0) group_done(work, total_ctas);
        return;
    }
    const int lane = threadIdx.x & 31;
    const uint64_t pol = kStream ? policy_evict_first() : 0;
    const uint64_t vecs_per_seg = t.seg_bytes >> 4;
    // piece counts fit in 32 bits (copy_units_fit bounds the collective)
    const uint32_t pieces_per_seg = (uint32_t)((vecs_per_seg + kVecPiece - 1) / kVecPiece);
    const uint64_t total = (uint64_t)pieces_per_seg * (uint64_t)t.nseg;
    auto copy_piece = [&](uint32_t p) {
        const uint32_t seg = p / pieces_per_seg;
        const uint64_t vbase = (uint64_t)(p - seg * pieces_per_seg) * kVecPiece;
        const uint8_t* src = t.src[seg] + ((vbase + (uint64_t)lane) << 4);
        uint8_t* dst = t.dst[seg] + ((vbase + (uint64_t)lane) << 4);
        uint4 v[kVecUnroll];
        if (vbase + kVecPiece <= vecs_per_seg) {
            // a whole piece: 8 loads at fixed 512-byte strides from one base, then 8 stores
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) v[u] = kStream ? ld_vec_stream(src + u * 512, pol) : ld_vec(src + u * 512);
#pragma unroll
            for (int u = 0; u < kVecUnroll; ++u) {
                if (kStream)
                    st_vec_stream(dst + u * 512, v[u], pol);
                else
                    st_vec(dst + u * 512, v[u]);
            }
            return;
        }
        // the segment's ragged last piece
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u)
            if (vbase + (uint64_t)(u * 32 + lane) < vecs_per_seg)
                v[u] = kStream ? ld_vec_stream(src + u * 512, pol) : ld_vec(src + u * 512);
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u)
            if (vbase + (uint64_t)(u * 32 + lane) < vecs_per_seg) {
                if (kStream)
                    st_vec_stream(dst + u * 512, v[u], pol);
                else
                    st_vec(dst + u * 512, v[u]);
            }
    };
    const unsigned cta = (unsigned)cta_base + blockIdx.x;
    const unsigned first_ctas = static_units / kVecWarps;  // CTAs of the first part
    const uint64_t round = static_units;                     // 16 F pieces per fixed round
    const uint64_t rounds = round ? (total + round - 1) / round < kVecClaim ? (total + round - 1) / round
                                                                               : kVecClaim
                                  : 0;
    const uint64_t fixed = rounds * round;  // pieces 0 .. fixed-1 are dealt without the counter
    bool worked = false;
    if (cta < first_ctas) {
#pragma unroll 1
        for (uint64_t j = 0; j < rounds; ++j) {
            const uint64_t p = j * round + (uint64_t)(threadIdx.x >> 5) * first_ctas + cta;
            if (p < total) {
                copy_piece((uint32_t)p);
                worked = true;
            }
        }
    }
    // pieces fixed + 4c .. fixed + 4c + 3 belong to claim c (none to claim when
    // the fixed rounds cover the whole collective)
    unsigned c = 0;
    if (lane == 0 && fixed < total) c = atomicAdd(&work[0], 1u);
    c = __shfl_sync(0xffffffffu, c, 0);
    uint64_t p0 = fixed < total ? fixed + (uint64_t)c * kVecClaim : total;
    while (p0 < total) {
        worked = true;
        unsigned next = 0;
        if (lane == 0) next = atomicAdd(&work[0], 1u);
#pragma unroll 1
        for (unsigned q = 0; q < kVecClaim; ++q)
            if (p0 + q < total) copy_piece((uint32_t)(p0 + q));
        c = __shfl_sync(0xffffffffu, next, 0);
        p0 = fixed + (uint64_t)c * kVecClaim;
    }
    // a hardware barrier reduction: did any warp of this CTA move a piece?
    const int cta_worked = __syncthreads_or(worked ? 1 : 0);
    if (threadIdx.x == 0) {
        if (cta_worked) stamp_window(st, false, cta, t_enter, globaltimer());
        group_done(work, total_ctas);
    }
}

// bulk kernel: chunk c of the collective is segment c / chunks_per_seg at
// byte offset (c % chunks_per_seg) * kBulkChunk (the last chunk of a segment
// may be shorter; every size is a multiple of 16 bytes).  One thread claims
// chunks from the group's counter as it issues their loads, remembers which
// chunk each ring buffer holds, and stores them in the order loaded.
template <bool kStream>
__global__ void __launch_bounds__(kBulkThreads, 1)
    copy_bulk_kernel(SegTable t, DevStatus* st, unsigned int* work, int cta_base, int total_ctas,
                     unsigned static_units, unsigned gate_need) {
    if (gate_closed(st, gate_need)) {
        if (threadIdx.x == 0) group_done(work, total_ctas);
        return;
    }
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kBulkBufs];
    __shared__ int abort_flag;
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int b = 0; b < kBulkBufs; ++b) mbar_init(smem_addr(&full_bar[b]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t pol = kStream ? policy_evict_first() : 0;
        const uint64_t chunks_per_seg = (t.seg_bytes + kBulkChunk - 1) / kBulkChunk;
        const uint64_t total = chunks_per_seg * (uint64_t)t.nseg;
        const unsigned rec = (unsigned)cta_base + blockIdx.x;
        uint32_t held[kBulkBufs];   // chunk id in each ring buffer
        uint32_t issued = 0;        // loads issued (buffer issued % kBulkBufs next)
        bool exhausted = false;
        auto chunk_of = [&](uint32_t c, const uint8_t*& src, uint8_t*& dst, uint32_t& bytes) {
            const uint64_t seg = c / chunks_per_seg;
            const uint64_t off = (c - seg * chunks_per_seg) * kBulkChunk;
            const uint64_t left = t.seg_bytes - off;
            bytes = (uint32_t)(left < kBulkChunk ? left : kBulkChunk);
            src = t.src[seg] + off;
            dst = t.dst[seg] + off;
        };
        // Claims the next chunk and issues its load into buffer issued % kBulkBufs.
        // CTA b of the group's first launch part (F CTAs) takes chunks
        // i * F + b, i = 0 .. kBulkBufs-1, without asking (interleaved, so a
        // small collective still spreads over every SM of the part); every other
        // chunk comes from the counter, numbered after those.
        const uint32_t cta = (unsigned)cta_base + blockIdx.x;
        const uint32_t first_ctas = static_units / (uint32_t)kBulkBufs;
        auto try_issue = [&]() {
            if (exhausted) return;
            const bool fixed = cta < first_ctas && issued < (uint32_t)kBulkBufs;
            if (!fixed && (uint64_t)static_units >= total) {  // the fixed chunks cover everything
                exhausted = true;
                return;
            }
            const uint32_t c = fixed ? issued * first_ctas + cta : static_units + atomicAdd(&work[0], 1u);
            if (c >= total) {
                exhausted = true;
                return;
            }
            if (issued == 0) stamp_begin(st, false, rec);
            const uint8_t* src;
            uint8_t* dst;
            uint32_t bytes;
            chunk_of(c, src, dst, bytes);
            const int b = (int)(issued % kBulkBufs);
            held[b] = c;
            const uint32_t bar = smem_addr(&full_bar[b]);
            mbar_arrive_expect_tx(bar, bytes);
            if (kStream)
                bulk_load_hint(base + (uint32_t)b * kBulkChunk, src, bytes, bar, pol);
            else
                bulk_load(base + (uint32_t)b * kBulkChunk, src, bytes, bar);
            ++issued;
        };
        for (int b = 0; b < kBulkBufs && !exhausted; ++b) try_issue();
        uint32_t done = 0;  // chunks stored (in load order)
        bool ok = true;
        for (; done < issued; ++done) {
            const int b = (int)(done % kBulkBufs);
            if (!mbar_wait(smem_addr(&full_bar[b]), (done / kBulkBufs) & 1u, &abort_flag)) {
                report_error(st, -4, kSiteBulkLoad);
                ok = false;
                break;
            }
            const uint8_t* src;
            uint8_t* dst;
            uint32_t bytes;
            chunk_of(held[b], src, dst, bytes);
            if (kStream)
                bulk_store_hint(dst, base + (uint32_t)b * kBulkChunk, bytes, pol);
            else
                bulk_store(dst, base + (uint32_t)b * kBulkChunk, bytes);
            bulk_commit();
            // Refill the buffer of chunk done-1 (the one the next load goes to)
            // once its store has read it.
            if (done >= 1 && !exhausted) {
                bulk_wait_read<1>();
                try_issue();
            }
        }
        if (!ok) {
            // Gave up: let every load still in flight land before the CTA's
            // shared memory is released.
            for (uint32_t j = done; j < issued; ++j) {
                const int b = (int)(j % kBulkBufs);
                volatile int dummy = 0;
                if (!mbar_wait(smem_addr(&full_bar[b]), (j / kBulkBufs) & 1u, &dummy))
                    report_error(st, -4, kSiteBulkDrain);
            }
        }
        bulk_wait_all();
        if (issued > 0) stamp_end(st, false, rec);
        group_done(work, total_ctas);
    }
    __syncthreads();
}

// Reduce-scatter half of the all-reduce (the part that needs arithmetic and so
// stays on SMs; the pages offload only the all-gather half to DMA).  Element i
// of the vector belongs to chunk c = i / chunk; its rank-order fp32 sum
// ((0 + in_0[i]) + in_1[i]) + ... is written into rank c's output row at
// position i.  16-byte vectors; all R loads issued before the adds.
__global__ void __launch_bounds__(kVecThreads, 2) reduce_scatter_kernel(RsTable t, DevStatus* st) {
    if (threadIdx.x == 0) stamp_begin(st, false);
    const uint64_t nvec = t.count >> 2;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        float4 x[kMaxRanksAr];
#pragma unroll
        for (int q = 0; q < kMaxRanksAr; ++q)
            if (q < t.nranks) x[q] = __ldg(reinterpret_cast<const float4*>(t.in[q]) + v);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxRanksAr; ++q)
            if (q < t.nranks) {
                acc.x = __fadd_rn(acc.x, x[q].x);
                acc.y = __fadd_rn(acc.y, x[q].y);
                acc.z = __fadd_rn(acc.z, x[q].z);
                acc.w = __fadd_rn(acc.w, x[q].w);
            }
        const uint64_t c = (v << 2) / t.chunk;
        reinterpret_cast<float4*>(t.out + c * t.count)[v] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) stamp_end(st, false);
}

// The whole all-reduce on SMs in one pass: every 16-byte vector of the sum is
// computed once -- the rank-order fp32 sum (0 + in_0[i]) + in_1[i] + ...,
// all ranks' loads in flight at once -- and stored into every rank's row.  So
// each input byte is read once and each output byte written once, the least an
// all-reduce of R vectors inside one HBM moves: R + R vectors' worth, against
// (R + 1) + 2 (R - 1) for a reduce-scatter followed by copies of its chunks.
// (The pages split the all-reduce in two to hand the all-gather half to DMA
// engines; the copy-engine path keeps that split.)  The result is the same bit
// for bit on every row.  The work is a list of slices of 32 vectors (one a
// lane), dealt and claimed the way the copy kernel deals its pieces: the first
// part's warps start on up to four fixed rounds of slices (interleaved across
// its CTAs, so a small all-reduce spreads over every SM of the part), the rest
// are claimed from the group's counter eight at a time (fewer when the group's
// warps would otherwise not get a claim each).  Nothing waits on anything, so
// a partitioned all-reduce widens onto the SMs a GEMM leaves, as the copies do.
constexpr uint64_t kArSlice = 32;   // vectors a slice (one a lane)
constexpr unsigned kArClaim = 8;    // most slices a claim

// units a claim: `most`, or fewer so that `units` make at least one claim a warp of the group
__device__ __forceinline__ uint32_t claim_size(uint32_t units, unsigned most, int total_ctas) {
    const uint32_t per = units / ((uint32_t)kVecWarps * (uint32_t)total_ctas);
    return per < 1u ? 1u : per > most ? most : per;
}

template <bool kStream>
__global__ void __launch_bounds__(kVecThreads, 2)
    allreduce_push_kernel(RsTable r, DevStatus* st, unsigned int* work, int cta_base, int total_ctas,
                          unsigned static_units, unsigned gate_need) {
    const unsigned long long t_enter = globaltimer();
    if (gate_closed(st, gate_need)) {
        if (threadIdx.x == 0) group_done(work, total_ctas);
        return;
    }
    const int lane = threadIdx.x & 31;
    const uint64_t pol = kStream ? policy_evict_first() : 0;
    const uint64_t nvec = r.count >> 2;  // 16-byte vectors of a rank's vector
    // slice counts fit in 32 bits (allreduce_sm_launch bounds them)
    const uint32_t slices = (uint32_t)((nvec + kArSlice - 1) / kArSlice);
    auto slice = [&](uint32_t sl) {
        const uint64_t v = (uint64_t)sl * kArSlice + (uint64_t)lane;
        if (v >= nvec) return;
        uint4 x[kMaxRanksAr];
#pragma unroll
        for (int q = 0; q < kMaxRanksAr; ++q)
            if (q < r.nranks) {
                const uint8_t* in = reinterpret_cast<const uint8_t*>(r.in[q]) + (v << 4);
                x[q] = kStream ? ld_vec_stream(in, pol) : ld_vec(in);
            }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kMaxRanksAr; ++q)
            if (q < r.nranks) {
                acc.x = __fadd_rn(acc.x, __uint_as_float(x[q].x));
                acc.y = __fadd_rn(acc.y, __uint_as_float(x[q].y));
                acc.z = __fadd_rn(acc.z, __uint_as_float(x[q].z));
                acc.w = __fadd_rn(acc.w, __uint_as_float(x[q].w));
            }
        const uint4 a = make_uint4(__float_as_uint(acc.x), __float_as_uint(acc.y), __float_as_uint(acc.z),
                                   __float_as_uint(acc.w));
#pragma unroll
        for (int q = 0; q < kMaxRanksAr; ++q)
            if (q < r.nranks) {
                uint8_t* out = reinterpret_cast<uint8_t*>(r.out + (uint64_t)q * r.count) + (v << 4);
                if (kStream)
                    st_vec_stream(out, a, pol);
                else
                    st_vec(out, a);
            }
    };

    const unsigned cta = (unsigned)cta_base + blockIdx.x;
    const unsigned first_ctas = static_units / kVecWarps;  // CTAs of the first part
    const uint64_t round = static_units;                     // slices a fixed round
    const uint64_t rounds = round ? ((slices + round - 1) / round < kVecClaim ? (slices + round - 1) / round
                                                                              : kVecClaim)
                                  : 0;
    const uint32_t fixed = (uint32_t)(rounds * round < slices ? rounds * round : slices);
    const uint32_t sc = claim_size(slices - fixed, kArClaim, total_ctas);
    const uint32_t claims = (slices - fixed + sc - 1) / sc;
    bool worked = false;
    if (cta < first_ctas) {
#pragma unroll 1
        for (uint64_t j = 0; j < rounds; ++j) {
            const uint64_t sl = j * round + (uint64_t)(threadIdx.x >> 5) * first_ctas + cta;
            if (sl < fixed) {
                slice((uint32_t)sl);
                worked = true;
            }
        }
    }
    // claim q: slices fixed + sc q .. + sc - 1; lane 0 claims the warp's next while the current one runs
    unsigned q = claims;
    if (claims > 0) {
        unsigned c0 = 0;
        if (lane == 0) c0 = atomicAdd(&work[0], 1u);
        q = __shfl_sync(0xffffffffu, c0, 0);
    }
    while (q < claims) {
        worked = true;
        unsigned next = 0;
        if (lane == 0) next = atomicAdd(&work[0], 1u);
        const uint32_t s0 = fixed + q * sc;
#pragma unroll 1
        for (uint32_t i = 0; i < sc && s0 + i < slices; ++i) slice(s0 + i);
        q = __shfl_sync(0xffffffffu, next, 0);
    }
    const int cta_worked = __syncthreads_or(worked ? 1 : 0);
    if (threadIdx.x == 0) {
        if (cta_worked) stamp_window(st, false, cta, t_enter, globaltimer());
        group_done(work, total_ctas);
    }
}

// ---------------------------------------------------------------- host side

int reduce_scatter_launch(const RsTable& t, int ctas, int smem_reserve, cudaStream_t s, DevStatus* st,
                          int* ctas_out) {
    if (ctas_out) *ctas_out = 0;
    if (t.count == 0) return 0;
    if (take_fault(kFaultSmCollLaunch)) return set_error(-3, "injected failure: SM collective launch");
    if (ctas < 1) ctas = 1;
    reduce_scatter_kernel<<<ctas, kVecThreads, smem_reserve, s>>>(t, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "reduce-scatter launch");
    count_launch();
    if (ctas_out) *ctas_out = ctas;
    return 0;
}

int copy_init_device(int max_reserve) {
    cudaError_t e = cudaSuccess;
    if (max_reserve > 0) {
        e = cudaFuncSetAttribute(reduce_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_reserve);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(reduce_scatter_kernel)");
    }
    for (auto fn : {copy_bulk_kernel<false>, copy_bulk_kernel<true>}) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(copy_bulk_kernel)");
    }
    if (max_reserve > 0) {
        for (auto fn : {copy_vec_kernel<false>, copy_vec_kernel<true>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_reserve);
            if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(copy_vec_kernel)");
        }
        for (auto fn : {allreduce_push_kernel<false>, allreduce_push_kernel<true>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_reserve);
            if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(allreduce_push_kernel)");
        }
    }
    return 0;
}

CopyGroup copy_group(DeviceState& ds, int total_ctas, int first_ctas) {
    CopyGroup g;
    g.work = ds.status->coll_sched[ds.next_coll_sched++ % kSchedSlots];
    g.total_ctas = total_ctas;
    g.static_ctas = first_ctas;
    return g;
}

static uint64_t copy_units(const SegTable& t, uint64_t unit_bytes) {
    return (t.seg_bytes + unit_bytes - 1) / unit_bytes * (uint64_t)t.nseg;
}

bool copy_units_fit(const SegTable& t) {
    // 4 KiB pieces (vec) and 32 KiB chunks (bulk) are numbered in 32 bits: keep
    // the piece count, plus the overshooting claims, well inside that
    return copy_units(t, 4 * 1024) < (1ull << 31);
}

// One launch of `kernel` with its arguments; `dependent` adds programmatic
// stream serialization.
template <class K, class... Args>
static cudaError_t launch_part(K kernel, int ctas, int threads, int smem, cudaStream_t s, bool dependent,
                               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = dependent ? attr : nullptr;
    cfg.numAttrs = dependent ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

static bool group_covers(const CopyGroup& g, int ctas, int cta_base) {
    return g.work && g.total_ctas >= ctas && cta_base >= 0 && cta_base + ctas <= g.total_ctas && g.static_ctas >= 0 &&
           g.static_ctas <= g.total_ctas && !(cta_base > 0 && cta_base < g.static_ctas);
}

int copy_sm_launch(const SegTable& t, int ctas, int cta_base, const CopyGroup& g, int flavour, int smem_reserve,
                   int l2_stream, cudaStream_t s, DevStatus* st, int* ctas_out, unsigned gate_need, bool dependent) {
    if (ctas_out) *ctas_out = 0;
    if (t.nseg <= 0 || t.seg_bytes == 0) return 0;
    if (!group_covers(g, ctas, cta_base)) return set_error(-1, "copy launch group does not cover this launch");
    if (!copy_units_fit(t)) return set_error(-5, "collective has more than 2^31 4 KiB pieces");
    if (take_fault(kFaultSmCollLaunch)) return set_error(-3, "injected failure: SM collective launch");
    if (ctas < 1) return set_error(-1, "copy launch needs at least one CTA");
    // the group's first part (its first g.static_ctas CTAs) starts on fixed units
    cudaError_t e;
    if (flavour == kSmkBulk) {
        const unsigned su = (unsigned)g.static_ctas * (unsigned)kBulkBufs;
        e = launch_part(l2_stream ? copy_bulk_kernel<true> : copy_bulk_kernel<false>, ctas, kBulkThreads, kBulkSmem,
                        s, dependent, t, st, g.work, cta_base, g.total_ctas, su, gate_need);
    } else {
        const unsigned su = (unsigned)g.static_ctas * (unsigned)kVecWarps;
        e = launch_part(l2_stream ? copy_vec_kernel<true> : copy_vec_kernel<false>, ctas, kVecThreads, smem_reserve,
                        s, dependent, t, st, g.work, cta_base, g.total_ctas, su, gate_need);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "copy kernel launch");
    count_launch();
    if (ctas_out) *ctas_out = ctas;
    return 0;
}

int allreduce_sm_launch(const RsTable& r, int ctas, int cta_base, const CopyGroup& g, int smem_reserve,
                        int l2_stream, cudaStream_t s, DevStatus* st, int* ctas_out, unsigned gate_need,
                        bool dependent) {
    if (ctas_out) *ctas_out = 0;
    if (r.count == 0) return 0;
    if (r.nranks < 1 || r.nranks > kMaxRanksAr || (r.count & 3u)) return set_error(-1, "all-reduce table is inconsistent");
    if (!group_covers(g, ctas, cta_base)) return set_error(-1, "all-reduce launch group does not cover this launch");
    // 512-byte slices: the slice count, and the claims past it, stay far inside 32 bits
    if (((r.count >> 2) + kArSlice - 1) / kArSlice >= (1ull << 30))
        return set_error(-5, "all-reduce has too many 512-byte slices");
    if (take_fault(kFaultSmCollLaunch)) return set_error(-3, "injected failure: SM collective launch");
    if (ctas < 1) return set_error(-1, "all-reduce launch needs at least one CTA");
    const unsigned su = (unsigned)g.static_ctas * (unsigned)kVecWarps;
    cudaError_t e = launch_part(l2_stream ? allreduce_push_kernel<true> : allreduce_push_kernel<false>, ctas,
                                kVecThreads, smem_reserve, s, dependent, r, st, g.work, cta_base, g.total_ctas, su,
                                gate_need);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "all-reduce kernel launch");
    count_launch();
    if (ctas_out) *ctas_out = ctas;
    return 0;
}

int bulk_copy_smem_bytes() { return kBulkSmem; }

}  // namespace c3
