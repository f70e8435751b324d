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

// Work unit of the vec kernel: a "round" of kVecThreads * kVecUnroll vectors
// (64 KiB) inside one segment.  Rounds are dealt to CTAs grid-stride.
template <bool kStream>
__global__ void __launch_bounds__(kVecThreads, 2)
    copy_vec_kernel(SegTable t, DevStatus* st) {
    if (threadIdx.x == 0) stamp_begin(st, false);
    const uint64_t pol = kStream ? policy_evict_first() : 0;
    const uint64_t vecs_per_seg = t.seg_bytes >> 4;
    constexpr uint64_t kRound = (uint64_t)kVecThreads * kVecUnroll;
    const uint64_t rounds_per_seg = (vecs_per_seg + kRound - 1) / kRound;
    const uint64_t total_rounds = rounds_per_seg * (uint64_t)t.nseg;
    for (uint64_t r = blockIdx.x; r < total_rounds; r += gridDim.x) {
        const uint64_t seg = r / rounds_per_seg;
        const uint64_t v0 = (r - seg * rounds_per_seg) * kRound + threadIdx.x;
        const uint8_t* src = t.src[seg];
        uint8_t* dst = t.dst[seg];
        uint4 v[kVecUnroll];
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u) {
            const uint64_t i = v0 + (uint64_t)u * kVecThreads;
            if (i < vecs_per_seg) v[u] = kStream ? ld_vec_stream(src + (i << 4), pol) : ld_vec(src + (i << 4));
        }
#pragma unroll
        for (int u = 0; u < kVecUnroll; ++u) {
            const uint64_t i = v0 + (uint64_t)u * kVecThreads;
            if (i < vecs_per_seg) {
                if (kStream)
                    st_vec_stream(dst + (i << 4), v[u], pol);
                else
                    st_vec(dst + (i << 4), v[u]);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) stamp_end(st, false);
}

// bulk kernel: chunk c of the collective is segment c / chunks_per_seg at
// byte offset (c % chunks_per_seg) * kBulkChunk (the last chunk of a segment
// may be shorter; every size is a multiple of 16 bytes).
template <bool kStream>
__global__ void __launch_bounds__(kBulkThreads, 1) copy_bulk_kernel(SegTable t, DevStatus* st) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kBulkBufs];
    __shared__ int abort_flag;
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        stamp_begin(st, false);
        abort_flag = 0;
        for (int b = 0; b < kBulkBufs; ++b) mbar_init(smem_addr(&full_bar[b]), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t pol = kStream ? policy_evict_first() : 0;
        const uint64_t chunks_per_seg = (t.seg_bytes + kBulkChunk - 1) / kBulkChunk;
        const uint64_t total = chunks_per_seg * (uint64_t)t.nseg;
        const uint64_t n_my = (blockIdx.x < total) ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
        auto chunk_of = [&](uint64_t i, const uint8_t*& src, uint8_t*& dst, uint32_t& bytes) {
            const uint64_t c = blockIdx.x + i * gridDim.x;
            const uint64_t seg = c / chunks_per_seg;
            const uint64_t off = (c - seg * chunks_per_seg) * kBulkChunk;
            const uint64_t left = t.seg_bytes - off;
            bytes = (uint32_t)(left < kBulkChunk ? left : kBulkChunk);
            src = t.src[seg] + off;
            dst = t.dst[seg] + off;
        };
        auto issue_load = [&](uint64_t i) {
            const uint8_t* src;
            uint8_t* dst;
            uint32_t bytes;
            chunk_of(i, src, dst, bytes);
            const int b = (int)(i % kBulkBufs);
            const uint32_t bar = smem_addr(&full_bar[b]);
            mbar_arrive_expect_tx(bar, bytes);
            if (kStream)
                bulk_load_hint(base + (uint32_t)b * kBulkChunk, src, bytes, bar, pol);
            else
                bulk_load(base + (uint32_t)b * kBulkChunk, src, bytes, bar);
        };
        const uint64_t pro = n_my < (uint64_t)kBulkBufs ? n_my : (uint64_t)kBulkBufs;
        for (uint64_t i = 0; i < pro; ++i) issue_load(i);
        uint64_t issued = pro;  // loads issued so far (chunks 0 .. issued-1)
        uint64_t i = 0;
        for (; i < n_my; ++i) {
            const int b = (int)(i % kBulkBufs);
            if (!mbar_wait(smem_addr(&full_bar[b]), (uint32_t)((i / kBulkBufs) & 1), &abort_flag)) {
                report_error(st, -4, kSiteBulkLoad);
                break;
            }
            const uint8_t* src;
            uint8_t* dst;
            uint32_t bytes;
            chunk_of(i, src, dst, bytes);
            if (kStream)
                bulk_store_hint(dst, base + (uint32_t)b * kBulkChunk, bytes, pol);
            else
                bulk_store(dst, base + (uint32_t)b * kBulkChunk, bytes);
            bulk_commit();
            // Refill the buffer of chunk i-1 once its store has read it.
            if (i >= 1 && i - 1 + kBulkBufs < n_my) {
                bulk_wait_read<1>();
                issue_load(i - 1 + kBulkBufs);
                ++issued;
            }
        }
        if (i < n_my) {
            // Gave up: let every load still in flight land before the CTA's
            // shared memory is released.
            for (uint64_t j = i; j < issued; ++j) {
                const int b = (int)(j % kBulkBufs);
                volatile int dummy = 0;
                if (!mbar_wait(smem_addr(&full_bar[b]), (uint32_t)((j / kBulkBufs) & 1), &dummy))
                    report_error(st, -4, kSiteBulkDrain);
            }
        }
        bulk_wait_all();
        stamp_end(st, false);
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
    if (max_reserve > 0)
        for (auto fn : {copy_vec_kernel<false>, copy_vec_kernel<true>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_reserve);
            if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(copy_vec_kernel)");
        }
    return 0;
}

int copy_sm_launch(const SegTable& t, int ctas, int flavour, int smem_reserve, int l2_stream, cudaStream_t s,
                   DevStatus* st, int* ctas_out) {
    if (ctas_out) *ctas_out = 0;
    if (t.nseg <= 0 || t.seg_bytes == 0) return 0;
    if (take_fault(kFaultSmCollLaunch)) return set_error(-3, "injected failure: SM collective launch");
    if (ctas < 1) ctas = 1;
    if (flavour == kSmkBulk) {
        if (l2_stream)
            copy_bulk_kernel<true><<<ctas, kBulkThreads, kBulkSmem, s>>>(t, st);
        else
            copy_bulk_kernel<false><<<ctas, kBulkThreads, kBulkSmem, s>>>(t, st);
    } else {
        if (l2_stream)
            copy_vec_kernel<true><<<ctas, kVecThreads, smem_reserve, s>>>(t, st);
        else
            copy_vec_kernel<false><<<ctas, kVecThreads, smem_reserve, s>>>(t, st);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "copy kernel launch");
    count_launch();
    if (ctas_out) *ctas_out = ctas;
    return 0;
}

int bulk_copy_smem_bytes() { return kBulkSmem; }

}  // namespace c3
