// gemm_tcgen05.cu -- the computation half of C3: C = A * B^T in bf16 with fp32
// accumulation on the sm_103a tensor cores (tcgen05.mma, accumulator in TMEM),
// operands brought in by TMA, persistent CTAs whose number can be capped.
//
// The pages pair a library GEMM with a collective and study how the two
// interfere ("Optimizing ML Concurrent Computation and Communication with GPU
// DMA Engines": the GEMM loses time when compute units are taken away or
// shared, Figure 5a and Section IV-B1).  Capping the persistent grid is how
// this library gives the GEMM a fixed SM budget.
//
// Kernel layout (one CTA per SM, 192 threads):
//   warp 0      TMA producer: A tile 128 x 64 and B tile BN x 64 per stage,
//               128-byte swizzle, into a STAGES-deep shared-memory ring;
//   warp 1      TMEM owner and MMA issuer (one thread): 4 x tcgen05.mma
//               (M=128, N=BN, K=16) per stage into one of two TMEM
//               accumulators, tcgen05.commit frees the stage / publishes the tile;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns, fp32 stores to C
//               with edge masking, then release the accumulator.
// The two accumulators let the epilogue of tile i overlap the main loop of
// tile i+1.  Tiles are dealt round-robin (tile = blockIdx.x + i * gridDim.x)
// in a grouped order: GROUP_M row blocks advance together so that the CTAs
// in flight share A row blocks and B column blocks in L2.
#include "c3_device.cuh"
#include "c3_internal.h"

#include <cstdio>
#include <mutex>

namespace c3 {

constexpr int kBM = 128;
constexpr int kBK = 64;           // 64 bf16 = 128 bytes = one swizzle row
constexpr int kUmmaK = 16;        // K of one kind::f16 MMA
constexpr int kGemmThreads = 192;
constexpr int kGroupM = 16;

template <int BN>
struct GemmCfg {
    static constexpr int kStages = (BN == 256) ? 4 : 6;
    static constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KiB
    static constexpr uint32_t kBBytes = BN * kBK * 2;    // 32 or 16 KiB
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;        // two accumulators
    // ring + barriers + TMEM slot + abort flag, plus 1 KiB for 1024-byte alignment
    static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
};

// Instruction descriptor of kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
template <int BN>
__device__ __forceinline__ uint32_t make_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128-byte swizzle: start address >> 4 (bits 0-13), leading byte offset
// (unused for swizzled K-major, 1), stride byte offset 1024 >> 4 between
// 8-row groups (bits 32-45), descriptor version 1 (bits 46-47), swizzle mode
// 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mb, int& nb) {
    const int per_group = kGroupM * num_n;
    const int g = t / per_group;
    const int first_m = g * kGroupM;
    const int gm = min(num_m - first_m, kGroupM);
    const int r = t - g * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     float* __restrict__ C, int M, int N, int num_m, int num_n, int num_kb,
                     DevStatus* st) {
    using Cfg = GemmCfg<BN>;
    constexpr int S = Cfg::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // ring: [A stage 0..S-1][B stage 0..S-1], then barriers
    const uint32_t sA = base;
    const uint32_t sB = base + S * Cfg::kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * Cfg::kStageBytes);
    // bars[0..S) full, [S..2S) empty, [2S..2S+2) tmem_full, [2S+2..2S+4) tmem_empty, [2S+4] drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = num_m * num_n;

    if (threadIdx.x == 0) {
        stamp_begin(st, true);
        *abort_flag = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(bar(i), 1);
            mbar_init(bar(S + i), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(2 * S + b), 1);
            mbar_init(bar(2 * S + 2 + b), 4 * 32);
        }
        mbar_init(bar(2 * S + 4), 1);
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(bar(S + stage), phase ^ 1u, abort_flag)) {
                        report_error(st, -4, kSiteGemmProducer);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(stage), Cfg::kStageBytes);
                    tma_load_2d(sA + stage * Cfg::kABytes, &tmA, bar(stage), kb * kBK, mb * kBM, pol_a);
                    tma_load_2d(sB + stage * Cfg::kBBytes, &tmB, bar(stage), kb * kBK, nb * BN, pol_b);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: the last load issued into each stage must have landed before
            // the CTA exits (a no-op when the MMA warp consumed everything).  The
            // last load into stage i belongs to the current pass when i < stage
            // and to the previous pass otherwise; on a stage never loaded the
            // parity-1 wait returns at once.
            volatile int no_abort = 0;
            for (int i = 0; i < S; ++i) {
                if (!mbar_wait(bar(i), (i < stage) ? phase : (phase ^ 1u), &no_abort))
                    report_error(st, -4, kSiteGemmDrain);
            }
            (void)ok;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = make_idesc<BN>();
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!mbar_wait(bar(2 * S + 2 + buf), (use & 1u) ^ 1u, abort_flag)) {
                    report_error(st, -4, kSiteGemmMma);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(bar(stage), phase, abort_flag)) {
                        report_error(st, -4, kSiteGemmMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = make_sdesc(sA + stage * Cfg::kABytes);
                    const uint64_t bdesc = make_sdesc(sB + stage * Cfg::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // advance 16 elements = 32 bytes inside the swizzled row
                        tc_mma_bf16(d_tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                                    (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(bar(S + stage));  // stage free once these MMAs have read it
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(bar(2 * S + buf));  // accumulator ready
            }
            // Whatever happened, make sure no MMA is still running before TMEM is freed.
            tc_commit(bar(2 * S + 4));
            volatile int no_abort = 0;
            if (!mbar_wait(bar(2 * S + 4), 0, &no_abort)) report_error(st, -4, kSiteGemmDrain);
        }
    } else {
        // ---------------- epilogue: warps 2..5 -> TMEM lane quarter (warp % 4)
        const int q = warp & 3;
        const bool vec_ok = (N & 3) == 0;
        int local = 0;
        for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++local) {
            const int buf = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            // tcgen05.ld is warp-collective: the whole warp leaves together if
            // any lane's wait gave up.
            const bool ready = mbar_wait(bar(2 * S + buf), use & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, ready)) {
                report_error(st, -4, kSiteGemmEpilogue);
                break;
            }
            tc_fence_after();
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb);
            const int row = mb * kBM + q * 32 + lane;
            float* crow = C + (size_t)row * (size_t)N;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(taddr + (uint32_t)(c * 32), r);
                tmem_ld_wait();
                const int col0 = nb * BN + c * 32;
                if (row < M) {
                    if (vec_ok && col0 + 32 <= N) {
                        float4* dst = reinterpret_cast<float4*>(crow + col0);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + j < N) crow[col0 + j] = __uint_as_float(r[j]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(2 * S + 2 + buf));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
    if (threadIdx.x == 0) stamp_end(st, true);
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 [rows][K] row-major, box 64 (K) x box_rows, 128-byte swizzle, zero fill
// outside the tensor (ragged M, N and K tails read as zeros).
static int make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(-3, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(-3, "cuTensorMapEncodeTiled failed");
    return 0;
}

int gemm_smem_bytes() { return GemmCfg<256>::kSmem > GemmCfg<128>::kSmem ? GemmCfg<256>::kSmem : GemmCfg<128>::kSmem; }

int gemm_init_device() {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GemmCfg<256>::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 GemmCfg<128>::kSmem);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(gemm)");
    return 0;
}

// Pick the tile width: the one whose busiest CTA has the least work, with a
// fixed per-tile overhead (epilogue, pipeline fill) that favours wide tiles.
static int choose_bn(int64_t M, int64_t N, int grid_cap) {
    const int64_t num_m = (M + kBM - 1) / kBM;
    int best_bn = 256;
    double best = 1e300;
    for (int bn : {256, 128}) {
        const int64_t tiles = num_m * ((N + bn - 1) / bn);
        const int64_t grid = tiles < grid_cap ? tiles : grid_cap;
        const int64_t waves = (tiles + grid - 1) / grid;
        const double cost = (double)waves * (bn + 32);
        if (cost < best - 1e-9) {
            best = cost;
            best_bn = bn;
        }
    }
    return best_bn;
}

int gemm_launch(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int sm_budget,
                cudaStream_t s, DevStatus* st, int* ctas_out) {
    if (ctas_out) *ctas_out = 0;
    if (M == 0 || N == 0) return 0;
    if (K == 0) return zero_fill_launch(C, (size_t)M * (size_t)N * sizeof(float), s);
    DeviceState* ds = device_state();
    if (!ds) return -3;
    int cap = (sm_budget <= 0 || sm_budget > ds->sm_count) ? ds->sm_count : sm_budget;
    const int bn = choose_bn(M, N, cap);
    const int64_t num_m = (M + kBM - 1) / kBM;
    const int64_t num_n = (N + bn - 1) / bn;
    const int64_t tiles = num_m * num_n;
    if (tiles > 0x7FFFFFFF) return set_error(-5, "GEMM has more than 2^31 tiles");
    const int grid = (int)(tiles < cap ? tiles : cap);
    const int num_kb = (int)((K + kBK - 1) / kBK);
    CUtensorMap ma, mb;
    int rc = make_map(&ma, A, M, K, kBM);
    if (rc) return rc;
    rc = make_map(&mb, B, N, K, bn);
    if (rc) return rc;
    if (bn == 256)
        gemm_bf16_kernel<256><<<grid, kGemmThreads, GemmCfg<256>::kSmem, s>>>(
            ma, mb, C, (int)M, (int)N, (int)num_m, (int)num_n, num_kb, st);
    else
        gemm_bf16_kernel<128><<<grid, kGemmThreads, GemmCfg<128>::kSmem, s>>>(
            ma, mb, C, (int)M, (int)N, (int)num_m, (int)num_n, num_kb, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "gemm kernel launch");
    count_launch();
    if (ctas_out) *ctas_out = grid;
    return 0;
}

}  // namespace c3

// ---------------------------------------------------------------- allocation-free GEMM entry point
//
// c3_gemm_noalloc: the GEMM for callers that must not allocate device memory
// (see include/c3_api.h).  Its scratch -- the error word, the %globaltimer
// window and the per-CTA residency records the kernel writes -- lives in the
// file-scope array below instead of the library's cudaMalloc'd status block.
// Host code cannot use the array's name as a device address, so the address
// is looked up once per device with cudaGetSymbolAddress and cached.

namespace c3 {

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStatusBytes];

struct NoAllocDevice {
    bool ready = false;
    int sm_count = 0;
    DevStatus* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
static NoAllocDevice g_noalloc[64];
static std::mutex g_noalloc_mu;

// Once per device, with that device current: the array's device address, the
// SM count and the kernels' shared-memory attribute.  No allocation.
static int noalloc_setup(NoAllocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return set_error(-5, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& d = g_noalloc[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return set_cuda_error(e, "device attributes");
        if (major != 10 || minor != 3) return set_error(-5, "libc3 is built for sm_103a (GB300) only");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
        d.scratch = static_cast<DevStatus*>(p);
        int rc = gemm_init_device();
        if (rc) return rc;
        d.ready = true;
    }
    *out = &d;
    return 0;
}

}  // namespace c3

extern "C" int c3_gemm_noalloc(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                               int sm_budget, void* stream, int check) {
    using namespace c3;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M < 0 || N < 0 || K < 0 || sm_budget < 0) return set_error(-1, "negative size or sm_budget");
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return set_error(-5, "GEMM dimension above 2^31-1");
    if (M == 0 || N == 0) return 0;
    if (!C) return set_error(-1, "C is NULL");
    if ((uintptr_t)C & 15u) return set_error(-2, "C must be 16-byte aligned");
    if (K > 0) {
        if (!A || !B) return set_error(-1, "A or B is NULL");
        if (((uintptr_t)A | (uintptr_t)B) & 15u) return set_error(-2, "A and B must be 16-byte aligned");
        if (K % 8) return set_error(-2, "K must be a multiple of 8 (16-byte TMA row pitch)");
    }
    NoAllocDevice* d = nullptr;
    int rc = noalloc_setup(&d);
    if (rc) return rc;
    const int cap = (sm_budget <= 0 || sm_budget > d->sm_count) ? d->sm_count : sm_budget;
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * sizeof(float), s);
        return e == cudaSuccess ? 0 : set_cuda_error(e, "cudaMemsetAsync");
    }
    const int bn = choose_bn(M, N, cap);
    const int64_t num_m = (M + kBM - 1) / kBM;
    const int64_t num_n = (N + bn - 1) / bn;
    const int64_t tiles = num_m * num_n;
    if (tiles > 0x7FFFFFFF) return set_error(-5, "GEMM has more than 2^31 tiles");
    const int grid = (int)(tiles < cap ? tiles : cap);
    // The static block records at most kCtaRecs CTAs: refuse a launch that would need more.
    if (grid > kCtaRecs)
        return set_error(-5, "c3_gemm_noalloc: more than 256 CTAs would need more than its 16 KiB scratch");
    CUtensorMap ma, mb;
    if ((rc = make_map(&ma, A, M, K, kBM))) return rc;
    if ((rc = make_map(&mb, B, N, K, bn))) return rc;
    // The block keeps the previous call's contents: clear it on this stream first.
    if ((rc = status_reset_launch(d->scratch, s))) return rc;
    const int num_kb = (int)((K + kBK - 1) / kBK);
    if (bn == 256)
        gemm_bf16_kernel<256><<<grid, kGemmThreads, GemmCfg<256>::kSmem, s>>>(
            ma, mb, C, (int)M, (int)N, (int)num_m, (int)num_n, num_kb, d->scratch);
    else
        gemm_bf16_kernel<128><<<grid, kGemmThreads, GemmCfg<128>::kSmem, s>>>(
            ma, mb, C, (int)M, (int)N, (int)num_m, (int)num_n, num_kb, d->scratch);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "gemm kernel launch");
    count_launch();
    if (!check) return 0;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return set_cuda_error(e, "stream synchronize");
    int err = 0, where = 0;
    e = cudaMemcpy(&err, &d->scratch->error, sizeof err, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(&where, &d->scratch->where, sizeof where, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e, "reading the scratch status word");
    if (err) {
        char buf[96];
        std::snprintf(buf, sizeof buf, "device wait gave up (site %d)", where);
        return set_error(err, buf);
    }
    return 0;
}
