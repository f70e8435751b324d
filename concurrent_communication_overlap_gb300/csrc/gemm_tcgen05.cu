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
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns, then out to C.
//               Staged: each 32 x 32 fp32 block goes through shared memory in
//               the 128-byte swizzle and leaves by TMA store, whole cache lines
//               at a time, and the accumulator is released as soon as it has
//               been read out.  Direct (no staging space for this tile, or
//               N % 4 != 0): per-thread row stores with edge masking.
// Two accumulator sets, where TMEM holds them, let the epilogue of tile i
// overlap the main loop of tile i+1.  Tiles are claimed one by one from an atomic counter (a
// scheduler slot in the status block), in a grouped order: GROUP_M row blocks
// advance together so that the tiles in flight share A row blocks and B
// column blocks in L2.  A CTA slowed by a neighbour, or started late because
// its SM was held by a collective, claims fewer tiles.
#include "c3_device.cuh"
#include "c3_internal.h"

#include <cstdio>
#include <mutex>

namespace c3 {

constexpr int kBM = 128;          // rows of one MMA / one accumulator
constexpr int kBK = 64;           // 64 bf16 = 128 bytes = one swizzle row
constexpr int kUmmaK = 16;        // K of one kind::f16 MMA
constexpr int kGemmThreads = 192;
constexpr int kGroupM = 16;
constexpr int kSmemLimit = 232448;  // opt-in shared memory per CTA (227 KiB)

// Tile of one CTA: MSUB x 128 rows (MSUB accumulators side by side in TMEM,
// all fed by the same B tile) by BN columns.  Two accumulator sets when they
// fit in TMEM's 512 columns, so the epilogue of one tile overlaps the main
// loop of the next; one set otherwise.
template <int BN, int MSUB>
struct GemmCfg {
    static constexpr uint32_t kABytes = kBM * kBK * 2;           // 16 KiB per 128-row sub-tile
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = MSUB * kABytes + kBBytes;
    static constexpr int kStagesFit = (kSmemLimit - 1024 - 512) / (int)kStageBytes;
    static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
    static constexpr uint32_t kAccCols = MSUB * BN;              // fp32 columns of one accumulator set
    static constexpr int kAccBufs = (2 * kAccCols <= 512) ? 2 : 1;
    static constexpr uint32_t kUsedCols = kAccCols * kAccBufs;
    static constexpr uint32_t kTmemCols = kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128
                                          : kUsedCols <= 256 ? 256 : 512;
    // Epilogue staging: two 4 KiB blocks (32 rows x 128 B) per epilogue warp.
    // Its own region when the ring leaves room for it; otherwise the CTA's
    // last tile borrows the (then idle) ring, and earlier tiles store
    // directly.
    static constexpr int kStagingBytes = 4 * 2 * 4096;
    static constexpr bool kOwnStaging =
        kSmemLimit - 1024 - 512 - kStages * (int)kStageBytes >= kStagingBytes;
    // A last tile staged in the idle ring gives each epilogue warp a quarter of
    // it: room for every 4 KiB block of its lane quarter, so no block is reused
    // and no store has to be waited for before the next block is written.
    static constexpr int kRingBlocksPerWarp = kStages * (int)kStageBytes / (4 * 4096);
    static constexpr int kBlocksPerWarp = MSUB * BN / 32;
    static_assert(kOwnStaging || kRingBlocksPerWarp >= kBlocksPerWarp, "no room to stage the epilogue");
    // ring, [staging], then barriers / TMEM slot / abort flag (512 B), plus 1 KiB for alignment
    static constexpr int kSmem = kStages * kStageBytes + (kOwnStaging ? kStagingBytes : 0) + 1024 + 512;
    static_assert(kStages >= 2, "tile too large for the shared-memory ring");
    static_assert(kUsedCols <= 512, "accumulators exceed TMEM");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128 is 16..256 step 16");
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

template <int BN, int MSUB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, int has_mc, float* __restrict__ C, int M, int N,
                     int num_m, int num_n, int num_kb, unsigned int* sched, int static_first, DevStatus* st) {
    using Cfg = GemmCfg<BN, MSUB>;
    constexpr int S = Cfg::kStages;
    constexpr int NB = Cfg::kAccBufs;
    constexpr int kRowsCta = kBM * MSUB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // ring: stage i = [A sub-tile 0 .. MSUB-1][B], then the staging region (if own), then barriers
    const uint32_t own_staging = base + S * Cfg::kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + S * Cfg::kStageBytes +
                                                 (Cfg::kOwnStaging ? Cfg::kStagingBytes : 0));
    // bars[0..S) full, [S..2S) empty, [2S..2S+NB) tmem_full, [2S+NB..2S+2NB) tmem_empty, [2S+2NB] drain,
    // then the tile ring's full and empty barriers
    constexpr int kTR = 4;  // tile-id ring between the producer and the MMA / epilogue roles
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * NB + 1 + 2 * kTR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* tile_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    auto stage_a = [&](int stage, int sub) { return base + (uint32_t)stage * Cfg::kStageBytes + (uint32_t)sub * Cfg::kABytes; };
    auto stage_b = [&](int stage) { return base + (uint32_t)stage * Cfg::kStageBytes + MSUB * Cfg::kABytes; };
    const int BAR_TFULL = 2 * S, BAR_TEMPTY = 2 * S + NB, BAR_DRAIN = 2 * S + 2 * NB;
    const int BAR_RFULL = BAR_DRAIN + 1, BAR_REMPTY = BAR_RFULL + kTR;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = num_m * num_n;

    // A kernel launched after this one on its stream with programmatic stream
    // serialization (the second part of a partitioned collective) may be
    // scheduled once every CTA of this grid has passed this point: from then
    // on no GEMM CTA waits for an SM, and the dependent's CTAs take only the
    // SMs the GEMM leaves.  A no-op for any other successor.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        stamp_begin(st, true);
        if (st) atomicAdd(&st->gemm_started, 1u);  // read by collective CTAs that wait for the GEMM's SMs
        *abort_flag = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(bar(i), 1);
            mbar_init(bar(S + i), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(bar(BAR_TFULL + b), 1);
            mbar_init(bar(BAR_TEMPTY + b), 4 * 32);
        }
        mbar_init(bar(BAR_DRAIN), 1);
        for (int i = 0; i < kTR; ++i) {
            mbar_init(bar(BAR_RFULL + i), 1);
            mbar_init(bar(BAR_REMPTY + i), 1 + 4);  // the MMA thread + one arrival per epilogue warp
        }
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (has_mc) prefetch_tensormap(&tmC);
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
            // ---------------- TMA producer (and tile scheduler)
            // Tiles are claimed one at a time from the launch's counter (or
            // dealt round-robin when there is none), published to the other
            // roles through the tile ring, and the sentinel total_tiles ends
            // every role's loop.  A CTA that starts late (its SM was busy)
            // simply claims fewer tiles.  With static_first, CTA b starts on
            // tile b without waiting for the counter (every CTA starts at
            // once) and the counter hands out tiles from gridDim.x on.
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            const unsigned claim_base = static_first ? gridDim.x : 0u;
            int t = (sched && !static_first) ? (int)min(atomicAdd(&sched[0], 1u), (unsigned)total_tiles)
                                             : (int)blockIdx.x;
            for (int i = 0;; ++i) {
                const int slot = i & (kTR - 1);
                if (!mbar_wait(bar(BAR_REMPTY + slot), ((uint32_t)(i / kTR) & 1u) ^ 1u, abort_flag)) {
                    report_error(st, -4, kSiteGemmProducer);
                    break;
                }
                tile_ring[slot] = t < total_tiles ? t : total_tiles;
                mbar_arrive(bar(BAR_RFULL + slot));
                if (t >= total_tiles) break;
                // The next tile is claimed once this tile's first loads are in
                // flight; its value is needed only after the last one.
                unsigned next_raw = 0;
                int mb, nb;
                tile_coords(t, num_m, num_n, mb, nb);
                // With a single row block every tile reads the same A panel.
                // Each tile then walks K from its own starting block (spread
                // evenly over the column blocks), so that at any moment the
                // CTAs read different parts of A instead of all asking L2 for
                // the same lines.  The accumulation order follows the loads.
                int kx = (num_m == 1) ? (int)(((long long)nb * num_kb) / num_n) : 0;
                bool ok = true;
                for (int kb = 0; kb < num_kb; ++kb, kx = (kx + 1 == num_kb) ? 0 : kx + 1) {
                    if (!mbar_wait(bar(S + stage), phase ^ 1u, abort_flag)) {
                        report_error(st, -4, kSiteGemmProducer);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(stage), Cfg::kStageBytes);
#pragma unroll
                    for (int sub = 0; sub < MSUB; ++sub)
                        tma_load_2d(stage_a(stage, sub), &tmA, bar(stage), kx * kBK, mb * kRowsCta + sub * kBM, pol_a);
                    tma_load_2d(stage_b(stage), &tmB, bar(stage), kx * kBK, nb * BN, pol_b);
                    if (kb == 0 && sched) next_raw = atomicAdd(&sched[0], 1u);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                t = sched ? (int)min(claim_base + next_raw, (unsigned)total_tiles) : t + (int)gridDim.x;
            }
            // The launch's last CTA to finish puts its scheduler slot back to zero.
            if (sched) {
                __threadfence();
                if (atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
                    atomicExch(&sched[0], 0u);
                    atomicExch(&sched[1], 0u);
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
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = make_idesc<BN>();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int local = 0; ok; ++local) {
                const int slot = local & (kTR - 1);
                if (!mbar_wait(bar(BAR_RFULL + slot), (uint32_t)(local / kTR) & 1u, abort_flag)) {
                    report_error(st, -4, kSiteGemmMma);
                    break;
                }
                const int t = tile_ring[slot];
                mbar_arrive(bar(BAR_REMPTY + slot));
                if (t >= total_tiles) break;
                const int buf = local % NB;
                const uint32_t use = (uint32_t)(local / NB);
                if (!mbar_wait(bar(BAR_TEMPTY + buf), (use & 1u) ^ 1u, abort_flag)) {
                    report_error(st, -4, kSiteGemmMma);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * Cfg::kAccCols);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(bar(stage), phase, abort_flag)) {
                        report_error(st, -4, kSiteGemmMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = make_sdesc(stage_b(stage));
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
#pragma unroll
                        for (int sub = 0; sub < MSUB; ++sub) {
                            // advance 16 elements = 32 bytes inside the swizzled row
                            const uint64_t adesc = make_sdesc(stage_a(stage, sub));
                            tc_mma_bf16(d_tmem + (uint32_t)(sub * BN), adesc + (uint64_t)(2 * k),
                                        bdesc + (uint64_t)(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(bar(S + stage));  // stage free once these MMAs have read it
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(bar(BAR_TFULL + buf));  // accumulator set ready
            }
            // Whatever happened, make sure no MMA is still running before TMEM is freed.
            tc_commit(bar(BAR_DRAIN));
            volatile int no_abort = 0;
            if (!mbar_wait(bar(BAR_DRAIN), 0, &no_abort)) report_error(st, -4, kSiteGemmDrain);
        }
    } else {
        // ---------------- epilogue: warps 2..5 -> TMEM lane quarter (warp % 4)
        const int q = warp & 3;
        const bool vec_ok = (N & 3) == 0;
        for (int local = 0;; ++local) {
            const int slot = local & (kTR - 1);
            const bool have = mbar_wait(bar(BAR_RFULL + slot), (uint32_t)(local / kTR) & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, have)) {
                report_error(st, -4, kSiteGemmEpilogue);
                break;
            }
            const int t = tile_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_REMPTY + slot));
            if (t >= total_tiles) break;
            // Where this tile's output is staged: the own region, or the ring
            // when this is the CTA's last tile (the producer then loads nothing
            // more, and every stage has been consumed once the accumulator is
            // ready).  The next tile-ring entry is already
            // published by then: the producer writes it as soon as it has
            // issued this tile's last load.
            bool staged = false;
            uint32_t stg = own_staging;
            if (has_mc) {
                if (Cfg::kOwnStaging) {
                    staged = true;
                } else {
                    const int nslot = (local + 1) & (kTR - 1);
                    const bool seen =
                        mbar_wait(bar(BAR_RFULL + nslot), (uint32_t)((local + 1) / kTR) & 1u, abort_flag);
                    if (!__all_sync(0xffffffffu, seen)) {
                        report_error(st, -4, kSiteGemmEpilogue);
                        break;
                    }
                    staged = tile_ring[nslot] >= total_tiles;
                    stg = base;
                }
            }
            const int buf = local % NB;
            const uint32_t use = (uint32_t)(local / NB);
            // tcgen05.ld is warp-collective: the whole warp leaves together if
            // any lane's wait gave up.
            const bool ready = mbar_wait(bar(BAR_TFULL + buf), use & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, ready)) {
                report_error(st, -4, kSiteGemmEpilogue);
                break;
            }
            tc_fence_after();
            int mb, nb;
            tile_coords(t, num_m, num_n, mb, nb);
            if (staged) {
                // Own region: two 4 KiB blocks per warp, alternating; a block is
                // rewritten only after the TMA store issued from it two blocks
                // ago has read it.  Idle ring (last tile): one block per 32x32
                // piece, never reused.  Row `lane` of a block holds 32 fp32 in
                // eight 16-byte chunks, chunk j at position j ^ (lane & 7): the
                // 128-byte swizzle the store's tensor map undoes, and no bank
                // conflicts beyond the four wavefronts 512 bytes need.
                const uint32_t wstg =
                    stg + (uint32_t)q * (Cfg::kOwnStaging ? 8192u : (uint32_t)Cfg::kRingBlocksPerWarp * 4096u);
                int issued = 0;
                // The 32 x 32 pieces j = 0 .. MSUB * BN/32 - 1 (sub-tile j / (BN/32),
                // column block j % (BN/32)) are read out of TMEM one ahead of the one
                // being staged: the load of piece j+1 is in flight while piece j goes
                // to shared memory, and the accumulator set is released as soon as its
                // last piece has landed in registers.
                constexpr int kPieces = MSUB * (BN / 32);
                const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * Cfg::kAccCols);
                auto piece_taddr = [&](int j) {
                    return tq + (uint32_t)((j / (BN / 32)) * BN + (j % (BN / 32)) * 32);
                };
                auto release_if_last = [&](int j_landed) {
                    if (j_landed == kPieces - 1) {
                        // the accumulator set has been read out: the MMA may reuse it
                        tc_fence_before();
                        mbar_arrive(bar(BAR_TEMPTY + buf));
                    }
                };
                auto stage_piece = [&](const uint32_t (&r)[32], int j) {
                    const int sub = j / (BN / 32), c = j % (BN / 32);
                    const int row0 = mb * kRowsCta + sub * kBM + q * 32;
                    const int col0 = nb * BN + c * 32;
                    if (row0 >= M || col0 >= N) return;  // wholly outside C (uniform per warp)
                    const uint32_t blk = wstg + (uint32_t)(Cfg::kOwnStaging ? (issued & 1) : issued) * 4096u;
                    if (Cfg::kOwnStaging && issued >= 2) {
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                    }
                    const uint32_t rowp = blk + (uint32_t)lane * 128u;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        st_shared_v4(rowp + ((uint32_t)(jj ^ (lane & 7)) << 4), r[4 * jj], r[4 * jj + 1],
                                     r[4 * jj + 2], r[4 * jj + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, blk, col0, row0);  // clipped to M x N by the tensor map
                        bulk_commit();
                    }
                    ++issued;
                };
                uint32_t ra[32], rb[32];
                tmem_ld32(piece_taddr(0), ra);
                tmem_ld_wait();
                release_if_last(0);
#pragma unroll 1
                for (int j = 0; j < kPieces; j += 2) {
                    // ra holds piece j; rb receives piece j+1 meanwhile
                    if (j + 1 < kPieces) tmem_ld32(piece_taddr(j + 1), rb);
                    stage_piece(ra, j);
                    if (j + 1 >= kPieces) break;
                    tmem_ld_wait();
                    release_if_last(j + 1);
                    if (j + 2 < kPieces) tmem_ld32(piece_taddr(j + 2), ra);
                    stage_piece(rb, j + 1);
                    if (j + 2 < kPieces) {
                        tmem_ld_wait();
                        release_if_last(j + 2);
                    }
                }
                if (lane == 0) bulk_wait_read<0>();  // staging free for the next tile
                __syncwarp();
            } else {
#pragma unroll 1
                for (int sub = 0; sub < MSUB; ++sub) {
                    const int row = mb * kRowsCta + sub * kBM + q * 32 + lane;
                    float* crow = C + (size_t)row * (size_t)N;
                    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                           (uint32_t)(buf * Cfg::kAccCols + sub * BN);
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
                                                         __uint_as_float(r[4 * j + 2]),
                                                         __uint_as_float(r[4 * j + 3]));
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (col0 + j < N) crow[col0 + j] = __uint_as_float(r[j]);
                            }
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(BAR_TEMPTY + buf));
            }
        }
        // Every TMA store this warp issued has finished reading shared memory
        // before the CTA ends; their writes to C are complete when the grid is.
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
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

// The fp32 output C [M][N] as a TMA store target: box 32 x 32, the 128-byte
// swizzle the epilogue writes its staging blocks in.  Needs a row pitch that
// is a multiple of 16 bytes (N % 4 == 0); returns 1 when the map was made, 0
// when the epilogue must store directly.
static int make_out_map(CUtensorMap* map, float* C, int64_t M, int64_t N) {
    if (N % 4 != 0) return 0;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_error(-3, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)N * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(-3, "cuTensorMapEncodeTiled (output) failed");
    return 1;
}

// The tile configurations this build carries (BN x MSUB), in the order the
// cost model breaks ties.
struct TileCfg {
    int bn, msub, stages, acc_bufs, smem;
};
#define C3_CFG(BN_, MS_) {BN_, MS_, GemmCfg<BN_, MS_>::kStages, GemmCfg<BN_, MS_>::kAccBufs, GemmCfg<BN_, MS_>::kSmem}
static const TileCfg kCfgs[] = {C3_CFG(256, 1), C3_CFG(128, 1), C3_CFG(256, 2), C3_CFG(224, 2), C3_CFG(192, 2),
                                C3_CFG(128, 2)};
#undef C3_CFG
constexpr int kNumCfgs = sizeof(kCfgs) / sizeof(kCfgs[0]);

int gemm_smem_bytes() {
    int m = 0;
    for (const auto& c : kCfgs) m = c.smem > m ? c.smem : m;
    return m;
}

template <int BN, int MS>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemm_bf16_kernel<BN, MS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<BN, MS>::kSmem);
}

int gemm_init_device() {
    cudaError_t e = set_attr<256, 1>();
    if (e == cudaSuccess) e = set_attr<128, 1>();
    if (e == cudaSuccess) e = set_attr<256, 2>();
    if (e == cudaSuccess) e = set_attr<224, 2>();
    if (e == cudaSuccess) e = set_attr<192, 2>();
    if (e == cudaSuccess) e = set_attr<128, 2>();
    if (e != cudaSuccess) return set_cuda_error(e, "cudaFuncSetAttribute(gemm)");
    return 0;
}

// Cost model for picking the tile configuration, in SM clock cycles of the
// busiest CTA: per tile, the larger of the tensor-core time (4096 bf16 MACs
// per cycle per SM) and the operand-load time (bytes into shared memory at an
// assumed ~48 bytes per cycle per SM, the rate the single-tile kernel reached
// on a latency-bound load), times the number of waves; with one accumulator
// set the epilogue (fp32 tile out at ~64 bytes per cycle) does not overlap
// and is added per tile.
static int choose_cfg(int64_t M, int64_t N, int64_t K, int cap) {
    int best = 0;
    double best_cost = 1e300;
    for (int i = 0; i < kNumCfgs; ++i) {
        const TileCfg& c = kCfgs[i];
        const int64_t rows = 128LL * c.msub;
        const int64_t units = ((M + rows - 1) / rows) * ((N + c.bn - 1) / c.bn);
        const int64_t grid = units < cap ? units : cap;
        const int64_t waves = (units + grid - 1) / grid;
        const double kk = (double)((K + 63) / 64 * 64);
        const double mma = (double)rows * c.bn * kk / 4096.0;
        const double load = (double)(rows + c.bn) * kk * 2.0 / 48.0;
        const double epi = (double)rows * c.bn * 4.0 / 64.0;
        const double per_tile = (mma > load ? mma : load) + (c.acc_bufs == 1 ? epi : 0.0);
        const double cost = (double)waves * per_tile + epi;
        if (cost < best_cost * 0.999) {
            best_cost = cost;
            best = i;
        }
    }
    return best;
}

static int launch_cfg(int ci, int grid, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                      int has_mc, float* C, int64_t M, int64_t N, int64_t num_m, int64_t num_n, int num_kb,
                      unsigned int* sched, int static_first, DevStatus* st, cudaStream_t s) {
    if (take_fault(kFaultGemmLaunch)) return set_error(-3, "injected failure: GEMM launch");
    const TileCfg& c = kCfgs[ci];
#define C3_LAUNCH(BN_, MS_)                                                                                  \
    gemm_bf16_kernel<BN_, MS_><<<grid, kGemmThreads, GemmCfg<BN_, MS_>::kSmem, s>>>(                           \
        ma, mb, mc, has_mc, C, (int)M, (int)N, (int)num_m, (int)num_n, num_kb, sched, static_first, st)
    if (c.bn == 256 && c.msub == 1) C3_LAUNCH(256, 1);
    else if (c.bn == 128 && c.msub == 1) C3_LAUNCH(128, 1);
    else if (c.bn == 256 && c.msub == 2) C3_LAUNCH(256, 2);
    else if (c.bn == 224 && c.msub == 2) C3_LAUNCH(224, 2);
    else if (c.bn == 192 && c.msub == 2) C3_LAUNCH(192, 2);
    else C3_LAUNCH(128, 2);
#undef C3_LAUNCH
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "gemm kernel launch");
    count_launch();
    return 0;
}

// Plans one GEMM: configuration, grid, tensor maps.
struct GemmPlan {
    int ci, grid, num_kb, has_mc;
    int64_t num_m, num_n;
    CUtensorMap ma, mb, mc;
};

static int plan_gemm(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int cap,
                     GemmPlan* p) {
    p->ci = choose_cfg(M, N, K, cap);
    const TileCfg& c = kCfgs[p->ci];
    p->num_m = (M + 128LL * c.msub - 1) / (128LL * c.msub);
    p->num_n = (N + c.bn - 1) / c.bn;
    const int64_t tiles = p->num_m * p->num_n;
    if (tiles > 0x7FFFFFFF) return set_error(-5, "GEMM has more than 2^31 tiles");
    p->grid = (int)(tiles < cap ? tiles : cap);
    p->num_kb = (int)((K + kBK - 1) / kBK);
    int rc = make_map(&p->ma, A, M, K, kBM);
    if (rc) return rc;
    if ((rc = make_map(&p->mb, B, N, K, c.bn))) return rc;
    rc = make_out_map(&p->mc, C, M, N);
    if (rc < 0) return rc;
    p->has_mc = rc;
    return 0;
}

int gemm_prepare(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int sm_budget,
                 GemmLaunch* g) {
    g->kind = 0;
    g->C = C;
    g->M = M;
    g->N = N;
    g->K = K;
    if (M == 0 || N == 0) return 0;
    if (K == 0) {
        g->kind = 1;
        return 0;
    }
    DeviceState* ds = device_state();
    if (!ds) return -3;
    const int cap = (sm_budget <= 0 || sm_budget > ds->sm_count) ? ds->sm_count : sm_budget;
    GemmPlan p;
    int rc = plan_gemm(A, B, C, M, N, K, cap, &p);
    if (rc) return rc;
    g->kind = 2;
    g->ci = p.ci;
    g->grid = p.grid;
    g->num_kb = p.num_kb;
    g->num_m = p.num_m;
    g->num_n = p.num_n;
    g->ma = p.ma;
    g->mb = p.mb;
    g->mc = p.mc;
    g->has_mc = p.has_mc;
    return 0;
}

int gemm_enqueue(const GemmLaunch& g, cudaStream_t s, DevStatus* st, int* ctas_out) {
    if (ctas_out) *ctas_out = 0;
    if (g.kind == 0) return 0;
    if (g.kind == 1) return zero_fill_launch(g.C, (size_t)g.M * (size_t)g.N * sizeof(float), s);
    DeviceState* ds = device_state();
    if (!ds) return -3;
    unsigned int* sched = st ? st->sched[ds->next_sched++ % kSchedSlots] : nullptr;
    int rc = launch_cfg(g.ci, g.grid, g.ma, g.mb, g.mc, g.has_mc, g.C, g.M, g.N, g.num_m, g.num_n, g.num_kb, sched,
                        g.static_first, st, s);
    if (rc) return rc;
    if (ctas_out) *ctas_out = g.grid;
    return 0;
}

int gemm_launch(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int sm_budget,
                cudaStream_t s, DevStatus* st, int* ctas_out) {
    GemmLaunch g;
    int rc = gemm_prepare(A, B, C, M, N, K, sm_budget, &g);
    if (rc) return rc;
    return gemm_enqueue(g, s, st, ctas_out);
}

void gemm_sched_reset(DevStatus* st) {
    if (st) cudaMemset(st->sched, 0, sizeof st->sched);
}

int gemm_describe(int64_t M, int64_t N, int64_t K, int cap, int* bn, int* msub, int* grid) {
    const int ci = choose_cfg(M, N, K, cap);
    const TileCfg& c = kCfgs[ci];
    const int64_t tiles = ((M + 128LL * c.msub - 1) / (128LL * c.msub)) * ((N + c.bn - 1) / c.bn);
    *bn = c.bn;
    *msub = c.msub;
    *grid = (int)(tiles < cap ? tiles : cap);
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
    unsigned int next_sched = 0;
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
    GemmPlan plan;
    if ((rc = plan_gemm(A, B, C, M, N, K, cap, &plan))) return rc;
    // The static block records at most kCtaRecs CTAs: refuse a launch that would need more.
    if (plan.grid > kCtaRecs)
        return set_error(-5, "c3_gemm_noalloc: more than 256 CTAs would need more than its 16 KiB scratch");
    // The block keeps the previous call's contents: clear it on this stream first,
    // the scheduler slot this launch takes included (a launch that gave up a wait
    // may have left its slot non-zero, and the status reset leaves slots alone).
    if ((rc = status_reset_launch(d->scratch, s))) return rc;
    unsigned int* sched = d->scratch->sched[d->next_sched++ % kSchedSlots];
    cudaError_t ez = cudaMemsetAsync(sched, 0, 2 * sizeof(unsigned int), s);
    if (ez != cudaSuccess) return set_cuda_error(ez, "clearing the scheduler slot");
    if ((rc = launch_cfg(plan.ci, plan.grid, plan.ma, plan.mb, plan.mc, plan.has_mc, C, M, N, plan.num_m,
                         plan.num_n, plan.num_kb, sched, 1, d->scratch, s)))
        return rc;
    cudaError_t e;
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
