// c3_runtime.cpp -- host side of libc3.so: the C ABI of include/c3_api.h.
//
// Per-device state, argument checks, the four ways of running a GEMM and a
// collective together (baseline, schedule prioritisation, SM partitioning,
// copy-engine offload with an optional GEMM SM cap) and the C3 timer.  The
// modes and the yardstick follow "Optimizing ML Concurrent Computation and
// Communication with GPU DMA Engines" as its review pages state them:
//   ideal speedup    = (T_gemm + T_comm) / max(T_gemm, T_comm), isolated times
//                      (abstract; referee report summary; Section IV-B3);
//   c3_sp            = communication kernel scheduled first, at high priority
//                      ("If this is right": schedule the lower-workgroup-count
//                      kernel first);
//   c3_rp            = disjoint compute-unit budgets (Section V-B);
//   ConCCL / _rp     = the collective on DMA engines, optionally with compute
//                      units taken from the GEMM (Sections VI-B, VI-F).
// The pages call the achieved fraction "% of ideal speedup"; this library
// reports both readings of it: the share of the ideal gain realized,
// (S_real - 1) / (S_ideal - 1), and the ratio S_real / S_ideal.
#include "../../include/c3_api.h"
#include "c3_internal.h"

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <thread>

namespace c3 {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int set_cuda_error(cudaError_t e, const char* what) {
    std::snprintf(g_err, sizeof g_err, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    cudaGetLastError();  // clear the sticky-free error so later calls are not blamed
    return C3_ECUDA;
}

int set_error(int code, const char* what) {
    std::snprintf(g_err, sizeof g_err, "%s", what);
    return code;
}

static std::atomic<int> g_fault{0};

bool take_fault(int site) {
    int armed = site;
    return site != 0 && g_fault.compare_exchange_strong(armed, 0);
}

static_assert(kFaultGemmLaunch == C3_FAULT_GEMM_LAUNCH && kFaultSmCollLaunch == C3_FAULT_SM_COLL_LAUNCH &&
                  kFaultMemcpy == C3_FAULT_MEMCPY && kFaultDeviceInit == C3_FAULT_DEVICE_INIT,
              "fault site values");

constexpr int kMaxDevices = 64;
static DeviceState g_dev[kMaxDevices];

static int init_device(DeviceState& ds, int dev) {
    ds.device = dev;
    cudaError_t e;
#define C3_TRY(call, what)                                \
    do {                                                  \
        e = (call);                                       \
        if (e != cudaSuccess) return set_cuda_error(e, what); \
    } while (0)
    C3_TRY(cudaDeviceGetAttribute(&ds.sm_count, cudaDevAttrMultiProcessorCount, dev), "sm count");
    C3_TRY(cudaDeviceGetAttribute(&ds.l2_bytes, cudaDevAttrL2CacheSize, dev), "l2 size");
    C3_TRY(cudaDeviceGetAttribute(&ds.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev),
           "smem per sm");
    C3_TRY(cudaDeviceGetAttribute(&ds.smem_per_block, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
           "smem per block");
    C3_TRY(cudaDeviceGetAttribute(&ds.cc_major, cudaDevAttrComputeCapabilityMajor, dev), "cc major");
    C3_TRY(cudaDeviceGetAttribute(&ds.cc_minor, cudaDevAttrComputeCapabilityMinor, dev), "cc minor");
    if (ds.cc_major != 10 || ds.cc_minor != 3)
        return set_error(C3_EUNSUP, "libc3 is built for sm_103a (GB300) only");
    if (ds.sm_count > 256) return set_error(C3_EUNSUP, "more than 256 SMs: %smid maps hold 256");
    int lo = 0, hi = 0;
    C3_TRY(cudaDeviceGetStreamPriorityRange(&lo, &hi), "stream priority range");
    C3_TRY(cudaStreamCreateWithPriority(&ds.s_comm, cudaStreamNonBlocking, lo), "stream");
    C3_TRY(cudaStreamCreateWithPriority(&ds.s_comm_hi, cudaStreamNonBlocking, hi), "stream");
    C3_TRY(cudaStreamCreateWithFlags(&ds.s_capture, cudaStreamNonBlocking), "stream");
    for (auto& ev : ds.ev) C3_TRY(cudaEventCreate(&ev), "event");
    if (take_fault(kFaultDeviceInit))
        return set_error(C3_ECUDA, "injected failure: device initialisation (status block allocation refused)");
    C3_TRY(cudaMalloc(reinterpret_cast<void**>(&ds.status), kStatusBytes), "status block");
    C3_TRY(cudaMemset(ds.status, 0, kStatusBytes), "status block");
#undef C3_TRY
    int rc = gemm_init_device();
    if (rc) return rc;
    rc = copy_init_device(ds.smem_per_block);
    if (rc) return rc;
    ds.ready = true;
    return 0;
}

static void release_device(DeviceState& ds) {
    if (ds.s_comm) cudaStreamDestroy(ds.s_comm);
    if (ds.s_comm_hi) cudaStreamDestroy(ds.s_comm_hi);
    if (ds.s_capture) cudaStreamDestroy(ds.s_capture);
    if (ds.device >= 0) ce_release_graphs(ds.device);
    for (auto& ev : ds.ev)
        if (ev) cudaEventDestroy(ev);
    if (ds.status) cudaFree(ds.status);
    ds = DeviceState();
}

DeviceState* device_state() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_cuda_error(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_error(C3_EUNSUP, "device ordinal out of range");
        return nullptr;
    }
    DeviceState& ds = g_dev[dev];
    if (!ds.ready) {
        int rc = init_device(ds, dev);
        if (rc) {
            release_device(ds);
            return nullptr;
        }
    }
    return &ds;
}

static int default_comm_sms(const DeviceState& ds) {
    // One vector-copy CTA per SM: the budget at which the SM collective is
    // fastest alone on GB300 (a fifth of the SMs, the share the pages' library
    // gives its all-gather by default -- 64 of 304 compute units, Figure 5
    // caption -- moves less than half as many bytes per second here).
    return ds.sm_count;
}

// Shared memory a partitioned collective CTA reserves so that neither a GEMM
// CTA nor a second collective CTA fits on its SM.
static int exclusive_reserve(const DeviceState& ds) {
    int need_vs_gemm = ds.smem_per_sm - gemm_smem_bytes() + 1024;
    int need_vs_self = ds.smem_per_sm / 2 + 1024;
    int r = need_vs_gemm > need_vs_self ? need_vs_gemm : need_vs_self;
    return r > ds.smem_per_block ? ds.smem_per_block : r;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return na && nb && x < y + nb && y < x + na;
}

static int check_gemm(const void* A, const void* B, const float* C, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return set_error(C3_EINVAL, "negative GEMM dimension");
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return set_error(C3_EUNSUP, "GEMM dimension above 2^31-1");
    if (M == 0 || N == 0) return C3_OK;
    if (!C) return set_error(C3_EINVAL, "C is NULL");
    if (!aligned16(C)) return set_error(C3_EALIGN, "C must be 16-byte aligned");
    if (K == 0) return C3_OK;
    if (!A || !B) return set_error(C3_EINVAL, "A or B is NULL");
    if (!aligned16(A) || !aligned16(B)) return set_error(C3_EALIGN, "A and B must be 16-byte aligned");
    if (K % 8) return set_error(C3_EALIGN, "K must be a multiple of 8 (16-byte TMA row pitch)");
    return C3_OK;
}

static int build_allgather(const void* const* shards, void* out, size_t shard_bytes, int nranks,
                           SegTable* t) {
    if (nranks < 1 || nranks > kMaxSegs) return set_error(C3_EINVAL, "nranks must be 1..64");
    if (!shards || !out) return set_error(C3_EINVAL, "shards or out is NULL");
    if (shard_bytes % 16) return set_error(C3_EALIGN, "shard_bytes must be a multiple of 16");
    if (!aligned16(out)) return set_error(C3_EALIGN, "out must be 16-byte aligned");
    std::memset(t, 0, sizeof *t);
    for (int r = 0; r < nranks; ++r) {
        if (!shards[r]) return set_error(C3_EINVAL, "a shard pointer is NULL");
        if (!aligned16(shards[r])) return set_error(C3_EALIGN, "shards must be 16-byte aligned");
        if (overlaps(shards[r], shard_bytes, out, shard_bytes * (size_t)nranks))
            return set_error(C3_EINVAL, "out overlaps a shard");
        t->src[r] = static_cast<const uint8_t*>(shards[r]);
        t->dst[r] = static_cast<uint8_t*>(out) + (size_t)r * shard_bytes;
    }
    t->nseg = nranks;
    t->kind = kSegAllGather;
    t->nranks = nranks;
    t->seg_bytes = shard_bytes;
    return C3_OK;
}

static int build_alltoall(const void* in, void* out, size_t block_bytes, int nranks, SegTable* t) {
    if (nranks < 1 || nranks * nranks > kMaxSegs) return set_error(C3_EINVAL, "nranks must be 1..8");
    if (!in || !out) return set_error(C3_EINVAL, "in or out is NULL");
    if (block_bytes % 16) return set_error(C3_EALIGN, "block_bytes must be a multiple of 16");
    if (!aligned16(in) || !aligned16(out)) return set_error(C3_EALIGN, "in and out must be 16-byte aligned");
    const size_t total = block_bytes * (size_t)nranks * (size_t)nranks;
    if (overlaps(in, total, out, total)) return set_error(C3_EINVAL, "in and out overlap");
    std::memset(t, 0, sizeof *t);
    for (int i = 0; i < nranks; ++i)
        for (int j = 0; j < nranks; ++j) {
            t->src[i * nranks + j] = static_cast<const uint8_t*>(in) + (size_t)(i * nranks + j) * block_bytes;
            t->dst[i * nranks + j] = static_cast<uint8_t*>(out) + (size_t)(j * nranks + i) * block_bytes;
        }
    t->nseg = nranks * nranks;
    t->kind = kSegAllToAll;
    t->nranks = nranks;
    t->seg_bytes = block_bytes;
    return C3_OK;
}

static int build_allreduce(const void* const* inputs, void* out, size_t count, int nranks, CollPlan* cp) {
    if (nranks < 1 || nranks > kMaxRanksAr) return set_error(C3_EINVAL, "nranks must be 1..8 for the all-reduce");
    if (!inputs || !out) return set_error(C3_EINVAL, "inputs or out is NULL");
    if (count % ((size_t)nranks * 4))
        return set_error(C3_EALIGN, "count must be a multiple of 4 * nranks (16-byte chunks)");
    if (!aligned16(out)) return set_error(C3_EALIGN, "out must be 16-byte aligned");
    const size_t row = count * sizeof(float);
    std::memset(&cp->seg, 0, sizeof cp->seg);
    std::memset(&cp->rs, 0, sizeof cp->rs);
    for (int q = 0; q < nranks; ++q) {
        if (!inputs[q]) return set_error(C3_EINVAL, "an input pointer is NULL");
        if (!aligned16(inputs[q])) return set_error(C3_EALIGN, "inputs must be 16-byte aligned");
        if (overlaps(inputs[q], row, out, row * (size_t)nranks)) return set_error(C3_EINVAL, "out overlaps an input");
        cp->rs.in[q] = static_cast<const float*>(inputs[q]);
    }
    const size_t chunk = count / (size_t)nranks;
    float* o = static_cast<float*>(out);
    cp->rs.out = o;
    cp->rs.count = count;
    cp->rs.chunk = chunk ? chunk : 1;
    cp->rs.nranks = nranks;
    cp->has_rs = count > 0;
    int n = 0;
    for (int c = 0; c < nranks; ++c)
        for (int r = 0; r < nranks; ++r) {
            if (r == c) continue;
            cp->seg.src[n] = reinterpret_cast<const uint8_t*>(o + (size_t)c * count + (size_t)c * chunk);
            cp->seg.dst[n] = reinterpret_cast<uint8_t*>(o + (size_t)r * count + (size_t)c * chunk);
            ++n;
        }
    cp->seg.nseg = n;
    cp->seg.kind = kSegAllReduce;
    cp->seg.nranks = nranks;
    cp->seg.seg_bytes = chunk * sizeof(float);
    return C3_OK;
}

// Where one buffer lives.  Device memory of the current device (or managed
// memory) is used as given.  Page-locked host memory (cudaHostAlloc, or
// cudaHostRegister) is accepted as a collective's SOURCE only: the segment
// table then holds its device address, the copy engines reach it with
// host-to-device DMA and the SM copy kernel with plain loads over the CPU-GPU
// link.  Pageable memory and another device's memory are argument errors.
static int locate(const void* p, int dev, bool allow_host, bool* host, const void** dptr) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaPointerGetAttributes");
    *host = false;
    *dptr = p;
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        if (a.type == cudaMemoryTypeDevice && a.device != dev)
            return set_error(C3_EINVAL, "a buffer belongs to another device");
        return C3_OK;
    }
    if (a.type == cudaMemoryTypeHost) {
        if (!allow_host) return set_error(C3_EINVAL, "only a collective's sources may be host memory");
        if (!a.devicePointer) return set_error(C3_EINVAL, "page-locked host buffer has no device mapping");
        // the device address keeps the host address's offset within the allocation
        *host = true;
        *dptr = a.devicePointer;
        return C3_OK;
    }
    return set_error(C3_EINVAL, "a buffer is pageable host memory: use device or page-locked host memory");
}

// Resolves every buffer of a built plan against the current device: the
// destinations must be device memory; all-gather and all-to-all sources may
// be page-locked host memory (the all-reduce's inputs feed an SM reduction
// and must be device memory).
static int locate_plan(const DeviceState& ds, CollPlan* cp) {
    SegTable& t = cp->seg;
    t.host_src = 0;
    bool host = false;
    const void* d = nullptr;
    int rc;
    if (cp->has_rs) {
        for (int q = 0; q < cp->rs.nranks; ++q)
            if ((rc = locate(cp->rs.in[q], ds.device, false, &host, &d))) return rc;
        return locate(cp->rs.out, ds.device, false, &host, &d);
    }
    if (t.nseg == 0 || t.seg_bytes == 0) return C3_OK;
    if (t.kind == kSegAllToAll) {
        // one send buffer and one receive buffer; block (0,0) sits at both bases
        if ((rc = locate(t.dst[0], ds.device, false, &host, &d))) return rc;
        if ((rc = locate(t.src[0], ds.device, true, &host, &d))) return rc;
        if (host) {
            const intptr_t shift = (const uint8_t*)d - t.src[0];
            for (int i = 0; i < t.nseg; ++i) t.src[i] += shift;
            t.host_src = 1;
        }
        return C3_OK;
    }
    if ((rc = locate(t.dst[0], ds.device, false, &host, &d))) return rc;
    for (int i = 0; i < t.nseg; ++i) {
        if ((rc = locate(t.src[i], ds.device, true, &host, &d))) return rc;
        if (host) {
            t.src[i] = static_cast<const uint8_t*>(d);
            t.host_src = 1;
        }
    }
    return C3_OK;
}

// The SM copy kernel a collective runs on, and the shared memory its CTAs
// reserve: exclusive CTAs (partitioning) keep their SMs to themselves.
static int pick_flavour(const SegTable& t, int sm_kernel, bool exclusive) {
    return sm_kernel == C3_SMK_VEC ? kSmkVec
           : sm_kernel == C3_SMK_BULK ? kSmkBulk
           : (exclusive && !t.host_src ? kSmkBulk : kSmkVec);
}

// One collective launch.  SM engine: `budget` CTAs (0 = default), one launch
// group; exclusive = the CTAs keep their SMs to themselves (partitioning).
// With `split_total` > budget the collective is the first part of a split
// group of split_total CTAs (launch_coll_rest launches the others).  *group
// receives the group (SM engine).  An all-reduce on the SM engine runs as one
// pass of its own kernel, whatever p->sm_kernel asks for the copies; on the
// copy engine, as the reduce-scatter kernel and then memcpy of its chunks.
static int launch_coll(DeviceState& ds, const CollPlan& cp, int engine, int sm_kernel, int l2_stream, int ce_variant,
                       int budget, bool exclusive, cudaStream_t s, int* ctas, int split_total = 0,
                       CopyGroup* group = nullptr) {
    if (ctas) *ctas = 0;
    const SegTable& t = cp.seg;
    int k = budget > 0 ? budget : default_comm_sms(ds);
    if (k > ds.sm_count) k = ds.sm_count;
    const int total = split_total > k ? split_total : k;
    if (engine == C3_ENGINE_SM && t.host_src && sm_kernel == C3_SMK_BULK)
        return set_error(C3_EUNSUP, "the bulk copy kernel reads device memory only; host sources take the vector kernel");
    if (cp.has_rs) {
        if (engine == C3_ENGINE_SM) {
            // On the default budget (every SM), an unpartitioned all-reduce that moves
            // less than 512 MiB runs two CTAs an SM: more loads in flight through its
            // ramp and tail (16 MiB a rank: 42.6 us against 46.7 on one an SM).  Larger
            // ones keep one (64 MiB a rank: 161.5 against 167.6 us; one CTA an SM
            // already streams at the HBM rate there).  A budget the caller sets is kept.
            const uint64_t traffic = 2ull * (uint64_t)cp.rs.nranks * cp.rs.count * sizeof(float);
            const bool twice = budget <= 0 && !exclusive && split_total <= k && traffic < (512ull << 20);
            const int kk = twice ? 2 * k : k;
            CopyGroup g = copy_group(ds, split_total > k ? total : kk, kk);
            if (group) *group = g;
            return allreduce_sm_launch(cp.rs, kk, 0, g, exclusive ? exclusive_reserve(ds) : 0, l2_stream, s,
                                       ds.status, ctas);
        }
        // the reduce-scatter needs arithmetic, so it runs on SMs; the copy engine carries the all-gather
        int rc = reduce_scatter_launch(cp.rs, k, 0, s, ds.status, ctas);
        if (rc) return rc;
        if (t.nseg == 0) return 0;
        return copy_ce_launch(t, ce_variant, s, ds.s_capture, cp.stage);
    }
    if (engine == C3_ENGINE_CE) return copy_ce_launch(t, ce_variant, s, ds.s_capture, cp.stage);
    const int flavour = pick_flavour(t, sm_kernel, exclusive);
    const int reserve = (exclusive && flavour == kSmkVec) ? exclusive_reserve(ds) : 0;
    CopyGroup g = copy_group(ds, total, k);
    if (group) *group = g;
    return copy_sm_launch(t, k, 0, g, flavour, reserve, l2_stream, s, ds.status, ctas);
}

// The rest of a split SM collective: `rest` more CTAs of group `g`, numbered
// from `first`, exclusive like the first part, on stream `s2`.  Launched after
// the GEMM, so its CTAs start only on SMs the GEMM has left: the collective
// widens to them once the GEMM's CTAs finish (a CTA that finds no work left
// exits at once).  `dependent`: s2 is the GEMM's stream and this launch
// directly follows the GEMM there, as its programmatic dependent.
static int launch_coll_rest(DeviceState& ds, const CollPlan& cp, int sm_kernel, int l2_stream, int first, int rest,
                            const CopyGroup& g, cudaStream_t s2, int* ctas, unsigned gemm_ctas,
                            bool dependent = false) {
    if (ctas) *ctas = 0;
    const SegTable& t = cp.seg;
    if (rest <= 0) return 0;
    if (cp.has_rs)
        return allreduce_sm_launch(cp.rs, rest, first, g, exclusive_reserve(ds), l2_stream, s2, ds.status, ctas,
                                   gemm_ctas, dependent);
    if (t.nseg == 0 || t.seg_bytes == 0) return 0;
    const int flavour = pick_flavour(t, sm_kernel, true);
    const int reserve = flavour == kSmkVec ? exclusive_reserve(ds) : 0;
    return copy_sm_launch(t, rest, first, g, flavour, reserve, l2_stream, s2, ds.status, ctas, gemm_ctas, dependent);
}

// A split group whose second part could not be launched would never count to
// its total, so its work counter would stay dirty: clear it behind the first
// part, on the first part's stream.
static void abandon_group(const CopyGroup& g, cudaStream_t s) {
    if (g.work) cudaMemsetAsync(g.work, 0, 2 * sizeof(unsigned int), s);
}

static int wait_event(cudaEvent_t ev, double limit_s) {
    auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return C3_OK;
        if (e != cudaErrorNotReady) return set_cuda_error(e, "waiting for a run");
        double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
        if (el > limit_s) return set_error(C3_ETIMEOUT, "host wait for the run exceeded its limit");
        std::this_thread::yield();
    }
}

static double elapsed_s(cudaEvent_t a, cudaEvent_t b) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return -1.0;
    return (double)ms * 1e-3;
}

static int popcount8(const unsigned int* m) {
    int n = 0;
    for (int i = 0; i < 8; ++i) n += __builtin_popcount(m[i]);
    return n;
}

// SMs on which a GEMM CTA and a collective CTA were resident at the same
// time (their %globaltimer windows intersect), from the residency records.
static int coresident_sms(const DevStatus& h, int* shared_any) {
    unsigned int both_time[8] = {0}, both_any[8] = {0};
    for (int g = 0; g < kCtaRecs; ++g) {
        const CtaRec& a = h.gemm_rec[g];
        if (!a.used) continue;
        for (int c = 0; c < kCtaRecs; ++c) {
            const CtaRec& b = h.comm_rec[c];
            if (!b.used || a.smid != b.smid || a.smid >= 256) continue;
            both_any[a.smid >> 5] |= 1u << (a.smid & 31);
            if (a.t0 < b.t1 && b.t0 < a.t1) both_time[a.smid >> 5] |= 1u << (a.smid & 31);
        }
    }
    *shared_any = popcount8(both_any);
    return popcount8(both_time);
}

// Reads the status block into `out` (device windows, SM facts) and returns
// the device error word.
static int read_status(DeviceState& ds, c3_timing* out) {
    static DevStatus h;  // 12+ KiB: not on the stack
    cudaError_t e = cudaMemcpy(&h, ds.status, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e, "reading the status block");
    if (out) {
        out->t_gemm_dev = (h.gemm_t1 > h.gemm_t0) ? (double)(h.gemm_t1 - h.gemm_t0) * 1e-9 : 0.0;
        out->t_comm_dev = (h.comm_t1 > h.comm_t0) ? (double)(h.comm_t1 - h.comm_t0) * 1e-9 : 0.0;
        out->gemm_sms = popcount8(h.smid_gemm);
        out->comm_sms = popcount8(h.smid_comm);
        out->smid_overlap = coresident_sms(h, &out->sms_shared_any);
    }
    if (h.error) {
        // a launch that gave up may have left its tile-scheduler or copy work slot non-zero
        gemm_sched_reset(ds.status);
        cudaMemset(ds.status->coll_sched, 0, sizeof ds.status->coll_sched);
        char buf[128];
        std::snprintf(buf, sizeof buf, "device wait gave up (site %d)", h.where);
        return set_error(h.error, buf);
    }
    return C3_OK;
}

static int check_problem(const c3_problem* p, CollPlan* cp) {
    if (!p) return set_error(C3_EINVAL, "problem is NULL");
    int rc = check_gemm(p->A, p->B, p->C, p->M, p->N, p->K);
    if (rc) return rc;
    SegTable* t = &cp->seg;
    cp->has_rs = false;
    if (p->coll == C3_COLL_ALLGATHER)
        rc = build_allgather(p->shards, p->recv, p->unit_bytes, p->nranks, t);
    else if (p->coll == C3_COLL_ALLTOALL)
        rc = build_alltoall(p->send, p->recv, p->unit_bytes, p->nranks, t);
    else if (p->coll == C3_COLL_ALLREDUCE) {
        if (p->unit_bytes % sizeof(float)) return set_error(C3_EALIGN, "all-reduce unit_bytes must hold whole floats");
        rc = build_allreduce(p->shards, p->recv, p->unit_bytes / sizeof(float), p->nranks, cp);
    } else
        return set_error(C3_EINVAL, "unknown collective");
    if (rc) return rc;
    if (p->sm_kernel < C3_SMK_AUTO || p->sm_kernel > C3_SMK_BULK) return set_error(C3_EINVAL, "bad sm_kernel");
    if (p->coll_l2 != C3_L2_NORMAL && p->coll_l2 != C3_L2_EVICT_FIRST) return set_error(C3_EINVAL, "bad coll_l2");
    if (p->ce_variant < C3_CE_PER_SEGMENT || p->ce_variant > C3_CE_HOST_STAGED)
        return set_error(C3_EINVAL, "bad ce_variant");
    if (p->comm_sms < 0) return set_error(C3_EINVAL, "negative comm_sms");
    if (p->settle_us < 0 || p->settle_us > 1000000) return set_error(C3_EINVAL, "settle_us must be 0 .. 1000000");
    // each rate: 0 (unknown) or a positive finite number (NaN fails every comparison)
    for (double v : {p->peak_flops, p->peak_bytes_per_s, p->coll_plateau_sm, p->coll_plateau_ce})
        if (!(v >= 0.0 && v <= 1e300)) return set_error(C3_EINVAL, "peaks and plateaus must be >= 0 and finite");
    if (p->flush_buf && !aligned16(p->flush_buf)) return set_error(C3_EALIGN, "flush_buf must be 16-byte aligned");
    const size_t cb = p->coll == C3_COLL_ALLREDUCE ? p->unit_bytes * (size_t)p->nranks
                                                   : t->seg_bytes * (size_t)t->nseg;
    if (overlaps(p->C, (size_t)p->M * (size_t)p->N * 4, p->recv, cb))
        return set_error(C3_EINVAL, "C overlaps the collective's output");
    cp->stage = nullptr;
    if (p->ce_variant == C3_CE_HOST_STAGED) {
        // the copies move nseg * seg_bytes bytes (an all-reduce: its all-gather half, cb)
        if (!p->ce_stage) return set_error(C3_EINVAL, "C3_CE_HOST_STAGED needs a bounce buffer (ce_stage)");
        if (!aligned16(p->ce_stage)) return set_error(C3_EALIGN, "ce_stage must be 16-byte aligned");
        if (p->ce_stage_bytes < t->seg_bytes * (size_t)t->nseg)
            return set_error(C3_EINVAL, "ce_stage is smaller than the collective's copies");
        cp->stage = static_cast<uint8_t*>(p->ce_stage);
    }
    return C3_OK;
}

// The bounce buffer of the host-staged copy-engine variant must be page-locked
// host memory (both of its hops are then DMA), and the collective's sources
// device memory (page-locked host sources are DMA already, without a bounce).
static int locate_stage(const CollPlan& cp) {
    if (!cp.stage) return C3_OK;
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, cp.stage);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaPointerGetAttributes (ce_stage)");
    if (a.type != cudaMemoryTypeHost) return set_error(C3_EINVAL, "ce_stage must be page-locked host memory");
    if (cp.seg.host_src) return set_error(C3_EUNSUP, "C3_CE_HOST_STAGED needs device sources");
    return C3_OK;
}

// One run of `mode` on already-checked arguments; fills t_conc, the event
// times and the device facts.
// NVTX range around one timed phase, so that a profiler can select or filter
// the kernels each phase launches (ncu --nvtx, nsys); free when no tool is attached.
struct PhaseRange {
    explicit PhaseRange(const char* name) { nvtxRangePushA(name); }
    ~PhaseRange() { nvtxRangePop(); }
    PhaseRange(const PhaseRange&) = delete;
    PhaseRange& operator=(const PhaseRange&) = delete;
};

static const char* mode_range_name(int mode, int sm_split, int priority) {
    switch (mode) {
        case C3_MODE_SERIAL_SM: return "c3/serial (SM collective)";
        case C3_MODE_SERIAL_CE: return "c3/serial (memcpy collective)";
        case C3_MODE_CONCURRENT_CE: return sm_split ? "c3/concurrent memcpy, GEMM capped" : "c3/concurrent memcpy";
        case C3_MODE_CONCURRENT_SM_RECLAIM: return "c3/concurrent SM, partition with reclaim";
        default:
            if (sm_split) return priority ? "c3/concurrent SM, prioritised + partitioned" : "c3/concurrent SM, partitioned";
            return priority ? "c3/concurrent SM, prioritised" : "c3/concurrent SM, baseline";
    }
}

static int run_once(DeviceState& ds, const c3_problem* p, const CollPlan& t, int mode, int sm_split,
                    int priority, c3_timing* out) {
    PhaseRange range(mode_range_name(mode, sm_split, priority));
    cudaStream_t s0 = static_cast<cudaStream_t>(p->stream);
    cudaEvent_t ev0 = ds.ev[0], ev_g = ds.ev[1], ev_c = ds.ev[2], ev_end = ds.ev[3];
    const bool reclaim_mode = (mode == C3_MODE_CONCURRENT_SM_RECLAIM);
    int rc = 0;
    cudaError_t e;
    // With reclaim the GEMM is launched on every SM, so the collective's first
    // part must reach the hardware first or the GEMM takes every SM.  The
    // queue that records the start event is the one that proceeds first once
    // earlier work (an L2 flush) drains -- another stream has to notice the
    // event -- so in this mode the status reset, the start event and the
    // collective's first part all go on the collective's stream, and the
    // caller's stream waits for the start event before the GEMM.
    cudaStream_t sc_first = nullptr;
    if (reclaim_mode) {
        sc_first = ds.s_comm_hi;
        if ((e = cudaEventRecord(ds.ev[4], s0)) != cudaSuccess) return set_cuda_error(e, "event record");
        if ((e = cudaStreamWaitEvent(sc_first, ds.ev[4], 0)) != cudaSuccess) return set_cuda_error(e, "fork");
        if ((rc = status_reset_launch(ds.status, sc_first))) return rc;
    } else if ((rc = status_reset_launch(ds.status, s0))) {
        return rc;
    }
    int gctas = 0, cctas = 0;
    const bool serial = (mode == C3_MODE_SERIAL_SM || mode == C3_MODE_SERIAL_CE);
    const int engine = (mode == C3_MODE_CONCURRENT_CE || mode == C3_MODE_SERIAL_CE) ? C3_ENGINE_CE : C3_ENGINE_SM;
    // Host-side GEMM planning (tile choice, tensor maps) happens before the
    // start event: only device work and launch calls are timed.
    // A partition caps the GEMM at SM count - sm_split.  With reclaim its tiles are
    // planned for those SMs too, the ones it starts on, but it is launched on up to
    // every SM: CTAs that find their SM held start late, as the collective's SMs
    // free up, and take whatever tiles are left.  A GEMM whose tiles fit one wave
    // on the SMs it starts on then leaves none for a late second wave.  Every tile,
    // the first included, is claimed from the counter.
    const int gemm_cap = (!serial && sm_split > 0) ? ds.sm_count - sm_split : 0;
    GemmLaunch gl;
    if ((rc = gemm_prepare(p->A, p->B, p->C, p->M, p->N, p->K, gemm_cap, &gl))) return rc;
    if (reclaim_mode && gl.kind == 2) {
        gl.static_first = 0;
        const int64_t tiles = gl.num_m * gl.num_n;
        gl.grid = (int)(tiles < ds.sm_count ? tiles : ds.sm_count);
    }
    if ((e = cudaEventRecord(ev0, reclaim_mode ? sc_first : s0)) != cudaSuccess)
        return set_cuda_error(e, "event record");
    if (serial) {
        rc = gemm_enqueue(gl, s0, ds.status, &gctas);
        if (rc) return rc;
        if ((e = cudaEventRecord(ev_g, s0)) != cudaSuccess) return set_cuda_error(e, "event record");
        rc = launch_coll(ds, t, engine, p->sm_kernel, p->coll_l2, p->ce_variant, p->comm_sms, false, s0, &cctas);
        if (rc) return rc;
        if ((e = cudaEventRecord(ev_c, s0)) != cudaSuccess) return set_cuda_error(e, "event record");
    } else {
        if (sm_split < 0 || sm_split >= ds.sm_count)
            return set_error(C3_EINVAL, "sm_split must be 0 .. SM count - 1");
        // The GEMM runs on the caller's stream and only the collective is
        // forked onto a stream of its own: one cross-stream dependency on
        // the way in and one on the way out, instead of two each.
        cudaStream_t sg = s0;
        const bool reclaim = (mode == C3_MODE_CONCURRENT_SM_RECLAIM);
        // With reclaim the GEMM is launched on every SM, so the partition exists only
        // if the collective's CTAs are dispatched first: its stream takes the highest
        // priority, and the hardware hands pending CTAs of a higher-priority stream
        // the free SMs first.
        cudaStream_t sc = (priority || reclaim) ? ds.s_comm_hi : ds.s_comm;
        if (reclaim) {
            // sc already follows the start event in order; the GEMM's stream waits for it
            if ((e = cudaStreamWaitEvent(s0, ev0, 0)) != cudaSuccess) return set_cuda_error(e, "fork");
        } else if ((e = cudaStreamWaitEvent(sc, ev0, 0)) != cudaSuccess) {
            return set_cuda_error(e, "fork");
        }
        if (reclaim && sm_split < 1) return set_error(C3_EINVAL, "the reclaim mode needs sm_split >= 1");
        // Partitioning (sm_split > 0 on SMs): the collective starts on sm_split
        // SMs it holds alone and the GEMM on the others (capped at SM count -
        // sm_split, or, with reclaim, launched on every SM so that its CTAs
        // that find no free SM start as the collective's SMs free up).  The
        // collective is one launch group of SM-count CTAs in two parts: the
        // first sm_split CTAs, and the rest launched after the GEMM on a
        // second stream, whose CTAs start only on SMs the GEMM leaves and
        // claim whatever work is left -- so a collective that outlasts the
        // GEMM widens onto its SMs, and one that finishes first leaves nothing
        // for them but an immediate exit.
        //
        // The second part goes out right behind the GEMM on the GEMM's stream,
        // as its programmatic dependent: the hardware schedules it once every
        // GEMM CTA has started (each signals griddepcontrol.launch_dependents
        // on entry), so it can only take SMs the GEMM leaves, and it does not
        // wait for the GEMM to finish.  The first part, which creates the
        // launch group, therefore goes out before the GEMM, and the GEMM's
        // completion event follows the second part: t_gemm_ev then covers
        // the GEMM's stream (GEMM and the collective's second part).  The
        // all-reduce's one-pass kernel waits for nothing either, so it is
        // split the same way.
        const bool part = (engine == C3_ENGINE_SM && sm_split > 0);
        const int comm_budget = part ? sm_split : p->comm_sms;
        CopyGroup grp;
        int cctas2 = 0;
        bool comm_launched = false, rest_launched = false;
        // Each completion event is recorded right after its own launch(es), before
        // anything else is submitted.
        auto go_gemm = [&] {
            int r = gemm_enqueue(gl, sg, ds.status, &gctas);
            if (r == C3_OK && part) {
                r = launch_coll_rest(ds, t, p->sm_kernel, p->coll_l2, comm_budget, ds.sm_count - comm_budget, grp, sg,
                                     &cctas2, (unsigned)gctas, true);
                rest_launched = (r == C3_OK);
            }
            if (r == C3_OK && (e = cudaEventRecord(ev_g, sg)) != cudaSuccess) r = set_cuda_error(e, "event record");
            return r;
        };
        auto go_comm = [&] {
            int r = launch_coll(ds, t, engine, p->sm_kernel, p->coll_l2, p->ce_variant, comm_budget, part, sc, &cctas,
                                part ? ds.sm_count : 0, &grp);
            comm_launched = (r == C3_OK);
            if (r == C3_OK && (e = cudaEventRecord(ev_c, sc)) != cudaSuccess) r = set_cuda_error(e, "event record");
            return r;
        };
        // A failure after the collective went out still orders the caller's
        // stream after it, so that the caller may reuse its buffers once its
        // own stream has drained; a split group missing its second part has
        // its work counter cleared behind the first.
        auto fail = [&](int code) {
            if (comm_launched) {
                if (part && !rest_launched) abandon_group(grp, sc);
                if (cudaEventRecord(ev_c, sc) == cudaSuccess) cudaStreamWaitEvent(s0, ev_c, 0);
            }
            return code;
        };
        if (priority || reclaim || part) {
            if ((rc = go_comm())) return fail(rc);
            if ((rc = go_gemm())) return fail(rc);
        } else {
            if ((rc = go_gemm())) return rc;
            if ((rc = go_comm())) return fail(rc);
        }
        if ((e = cudaStreamWaitEvent(s0, ev_c, 0)) != cudaSuccess) return set_cuda_error(e, "join");
        cctas += cctas2;
    }
    if ((e = cudaEventRecord(ev_end, s0)) != cudaSuccess) return set_cuda_error(e, "event record");
    if ((rc = wait_event(ev_end, 120.0))) return rc;
    out->t_gemm_ev = elapsed_s(ev0, ev_g);
    out->t_comm_ev = elapsed_s(ev0, ev_c);
    // From the start event to the later of the two completion events, each
    // recorded right after its kernel(s), as the isolated phases are timed;
    // the join that orders the caller's stream after both is not part of it.
    out->t_conc = out->t_gemm_ev > out->t_comm_ev ? out->t_gemm_ev : out->t_comm_ev;
    out->gemm_ctas = gctas;
    out->comm_ctas = cctas;
    return read_status(ds, out);
}

// The settle period before a timed phase (c3_problem.settle_us): the previous
// phase has completed (every phase ends with a host wait on its last event),
// so the GPU idles for this long and each phase starts from the same clock
// and power state.
static void settle(const c3_problem* p) {
    if (p->settle_us > 0) std::this_thread::sleep_for(std::chrono::microseconds(p->settle_us));
}

// Times one phase that runs entirely on `s0`: fn() enqueues it.
template <class F>
static int time_phase(DeviceState& ds, cudaStream_t s0, const c3_problem* p, const char* name, double* t_out, F fn) {
    PhaseRange range(name);
    settle(p);
    int rc;
    if (p->flush_buf && p->flush_bytes && (rc = l2_flush_launch(p->flush_buf, p->flush_bytes, s0))) return rc;
    cudaError_t e;
    if ((e = cudaEventRecord(ds.ev[4], s0)) != cudaSuccess) return set_cuda_error(e, "event record");
    if ((rc = fn())) return rc;
    if ((e = cudaEventRecord(ds.ev[5], s0)) != cudaSuccess) return set_cuda_error(e, "event record");
    if ((rc = wait_event(ds.ev[5], 120.0))) return rc;
    *t_out = elapsed_s(ds.ev[4], ds.ev[5]);
    return C3_OK;
}

// Output bytes of the problem's collective (what its rate is counted in).
static double coll_out_bytes(const c3_problem* p, const CollPlan& t) {
    if (p->coll == C3_COLL_ALLREDUCE) return (double)p->unit_bytes * (double)p->nranks;
    return (double)t.seg.seg_bytes * (double)t.seg.nseg;
}

// The taxonomy's other two axes (c3_gemm_bound, c3_coll_bound in c3_api.h):
// the GEMM against the roofline ridge, the collective's isolated rate against
// half the plateau of its engine's size sweep.  Both compared cross-multiplied.
static void fill_bounds(c3_timing* r, const c3_problem* p, const CollPlan& t, int engine) {
    const double M = (double)p->M, N = (double)p->N, K = (double)p->K;
    const double flops = 2.0 * M * N * K;
    const double bytes = 2.0 * M * K + 2.0 * N * K + 4.0 * M * N;
    r->gemm_bound = C3_BOUND_UNKNOWN;
    if (p->peak_flops > 0.0 && p->peak_bytes_per_s > 0.0 && flops > 0.0 && bytes > 0.0)
        r->gemm_bound = (flops * p->peak_bytes_per_s < bytes * p->peak_flops) ? C3_GEMM_MEMORY : C3_GEMM_COMPUTE;
    const double plateau = engine == C3_ENGINE_CE ? p->coll_plateau_ce : p->coll_plateau_sm;
    const double cb = coll_out_bytes(p, t);
    r->coll_bound = C3_BOUND_UNKNOWN;
    if (plateau > 0.0 && cb > 0.0 && r->t_comm_iso > 0.0)
        r->coll_bound = (2.0 * cb >= plateau * r->t_comm_iso) ? C3_COLL_BANDWIDTH : C3_COLL_LATENCY;
}

static void fill_metrics(c3_timing* r) {
    r->t_serial = r->t_gemm_iso + r->t_comm_iso;
    r->t_ideal = r->t_gemm_iso > r->t_comm_iso ? r->t_gemm_iso : r->t_comm_iso;
    r->s_ideal = r->t_ideal > 0 ? r->t_serial / r->t_ideal : 0.0;
    r->s_real = r->t_conc > 0 ? r->t_serial / r->t_conc : 0.0;
    r->pct_ideal_gain = r->s_ideal > 1.0 ? (r->s_real - 1.0) / (r->s_ideal - 1.0) : 0.0;
    r->pct_ideal_ratio = r->s_ideal > 0 ? r->s_real / r->s_ideal : 0.0;
    if (r->t_gemm_iso >= 1.15 * r->t_comm_iso)
        r->cls = C3_CLASS_G_LONG;
    else if (r->t_comm_iso >= 1.15 * r->t_gemm_iso)
        r->cls = C3_CLASS_C_LONG;
    else
        r->cls = C3_CLASS_GC_EQUAL;
}

}  // namespace c3

using namespace c3;

extern "C" {

const char* c3_strerror(int status) {
    switch (status) {
        case C3_OK: return "ok";
        case C3_EINVAL: return "invalid argument";
        case C3_EALIGN: return "misaligned pointer or size";
        case C3_ECUDA: return "CUDA error";
        case C3_ETIMEOUT: return "bounded wait timed out";
        case C3_EUNSUP: return "unsupported";
        default: return "unknown status";
    }
}

const char* c3_last_error(void) { return g_err; }

uint64_t c3_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int c3_get_device_info(c3_device_info* out) {
    if (!out) return set_error(C3_EINVAL, "out is NULL");
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    out->device = ds->device;
    out->sm_count = ds->sm_count;
    out->l2_bytes = ds->l2_bytes;
    out->smem_per_sm = ds->smem_per_sm;
    out->smem_per_block = ds->smem_per_block;
    out->cc_major = ds->cc_major;
    out->cc_minor = ds->cc_minor;
    out->gemm_smem_bytes = gemm_smem_bytes();
    out->comm_default_sms = default_comm_sms(*ds);
    return C3_OK;
}

int c3_status_check(c3_stream s) {
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return set_cuda_error(e, "stream synchronize");
    int rc = read_status(*ds, nullptr);
    e = cudaMemset(ds->status, 0, kStatusBytes);
    if (e != cudaSuccess) return set_cuda_error(e, "clearing the status block");
    return rc;
}

int c3_shutdown(void) {
    for (auto& ds : g_dev)
        if (ds.ready) {
            int cur = 0;
            cudaGetDevice(&cur);
            cudaSetDevice(ds.device);
            cudaDeviceSynchronize();
            release_device(ds);
            cudaSetDevice(cur);
        }
    return C3_OK;
}

int c3_gemm(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int sm_budget,
            c3_stream s) {
    int rc = check_gemm(A, B, C, M, N, K);
    if (rc) return rc;
    if (sm_budget < 0) return set_error(C3_EINVAL, "negative sm_budget");
    if (M == 0 || N == 0) return C3_OK;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    return gemm_launch(A, B, C, M, N, K, sm_budget, static_cast<cudaStream_t>(s), ds->status, nullptr);
}

int c3_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_budget, int* bn, int* msub, int* ctas) {
    if (!bn || !msub || !ctas) return set_error(C3_EINVAL, "output pointer is NULL");
    if (M <= 0 || N <= 0 || K <= 0 || sm_budget < 0) return set_error(C3_EINVAL, "need M, N, K > 0, sm_budget >= 0");
    int cap = sm_budget;
    if (cap == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&cap, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return set_cuda_error(e, "SM count");
    }
    return gemm_describe(M, N, K, cap, bn, msub, ctas);
}

int c3_allgather(const void* const* shards, void* out, size_t shard_bytes, int nranks, int engine,
                 int sm_budget, c3_stream s) {
    if (engine != C3_ENGINE_SM && engine != C3_ENGINE_CE) return set_error(C3_EINVAL, "unknown engine");
    if (sm_budget < 0) return set_error(C3_EINVAL, "negative sm_budget");
    CollPlan t;
    int rc = build_allgather(shards, out, shard_bytes, nranks, &t.seg);
    if (rc) return rc;
    if (shard_bytes == 0) return C3_OK;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    if ((rc = locate_plan(*ds, &t))) return rc;
    return launch_coll(*ds, t, engine, C3_SMK_AUTO, 0, kCeGraph, sm_budget, false, static_cast<cudaStream_t>(s), nullptr);
}

int c3_alltoall(const void* in, void* out, size_t block_bytes, int nranks, int engine, int sm_budget,
                c3_stream s) {
    if (engine != C3_ENGINE_SM && engine != C3_ENGINE_CE) return set_error(C3_EINVAL, "unknown engine");
    if (sm_budget < 0) return set_error(C3_EINVAL, "negative sm_budget");
    CollPlan t;
    int rc = build_alltoall(in, out, block_bytes, nranks, &t.seg);
    if (rc) return rc;
    if (block_bytes == 0) return C3_OK;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    if ((rc = locate_plan(*ds, &t))) return rc;
    return launch_coll(*ds, t, engine, C3_SMK_AUTO, 0, kCeGraph, sm_budget, false, static_cast<cudaStream_t>(s), nullptr);
}

int c3_cta_windows(int kernel, c3_cta_window* out, int max, int* n) {
    if (kernel != 0 && kernel != 1) return set_error(C3_EINVAL, "kernel must be 0 (GEMM) or 1 (SM collective)");
    if (!out || !n || max < 0) return set_error(C3_EINVAL, "out, n and max >= 0 are required");
    *n = 0;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return set_cuda_error(e, "device synchronize");
    static DevStatus h;  // 12+ KiB: not on the stack
    e = cudaMemcpy(&h, ds->status, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return set_cuda_error(e, "reading the status block");
    const CtaRec* recs = kernel == 0 ? h.gemm_rec : h.comm_rec;
    unsigned long long t0 = ~0ull;
    for (int i = 0; i < kCtaRecs; ++i)
        if (recs[i].used && recs[i].t0 < t0) t0 = recs[i].t0;
    int k = 0;
    for (int i = 0; i < kCtaRecs && k < max; ++i) {
        if (!recs[i].used) continue;
        out[k].cta = i;
        out[k].smid = (int)recs[i].smid;
        out[k].t_start = (double)(recs[i].t0 - t0) * 1e-9;
        out[k].t_end = (double)(recs[i].t1 - t0) * 1e-9;
        ++k;
    }
    *n = k;
    return C3_OK;
}

int c3_inject_fault(int site) {
    if (site < C3_FAULT_NONE || site > C3_FAULT_DEVICE_INIT) return set_error(C3_EINVAL, "unknown fault site");
    g_fault.store(site);
    return C3_OK;
}

int c3_selftest_wait(uint64_t limit_ns, int arrive, c3_stream s) {
    if (limit_ns == 0 || limit_ns > 5000000000ull) return set_error(C3_EINVAL, "limit_ns must be 1 ns .. 5 s");
    if (arrive != 0 && arrive != 1) return set_error(C3_EINVAL, "arrive must be 0 or 1");
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(s);
    int rc = status_reset_launch(ds->status, st);
    if (rc) return rc;
    if ((rc = selftest_wait_launch(ds->status, limit_ns, arrive, st))) return rc;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_cuda_error(e, "stream synchronize");
    const int status = read_status(*ds, nullptr);
    // leave a clean status block behind, so later checks do not see this test
    if ((rc = status_reset_launch(ds->status, st))) return rc;
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_cuda_error(e, "stream synchronize");
    return status;
}

int c3_allreduce(const float* const* inputs, float* out, size_t count, int nranks, int engine, int sm_budget,
                 c3_stream s) {
    if (engine != C3_ENGINE_SM && engine != C3_ENGINE_CE) return set_error(C3_EINVAL, "unknown engine");
    if (sm_budget < 0) return set_error(C3_EINVAL, "negative sm_budget");
    CollPlan t;
    int rc = build_allreduce(reinterpret_cast<const void* const*>(inputs), out, count, nranks, &t);
    if (rc) return rc;
    if (count == 0) return C3_OK;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    if ((rc = locate_plan(*ds, &t))) return rc;
    return launch_coll(*ds, t, engine, C3_SMK_AUTO, 0, kCeGraph, sm_budget, false, static_cast<cudaStream_t>(s),
                       nullptr);
}

int c3_l2_flush(void* buf, size_t bytes, c3_stream s) {
    if (!buf && bytes) return set_error(C3_EINVAL, "buf is NULL");
    if (!aligned16(buf)) return set_error(C3_EALIGN, "buf must be 16-byte aligned");
    return l2_flush_launch(buf, bytes, static_cast<cudaStream_t>(s));
}

int c3_run(const c3_problem* p, int mode, int sm_split, int priority, c3_timing* out) {
    if (!out) return set_error(C3_EINVAL, "out is NULL");
    std::memset(out, 0, sizeof *out);
    if (mode < C3_MODE_SERIAL_SM || mode > C3_MODE_CONCURRENT_SM_RECLAIM) return set_error(C3_EINVAL, "unknown mode");
    if (priority != 0 && priority != 1) return set_error(C3_EINVAL, "priority must be 0 or 1");
    CollPlan t;
    int rc = check_problem(p, &t);
    if (rc) return rc;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    if (sm_split < 0 || sm_split >= ds->sm_count) return set_error(C3_EINVAL, "sm_split must be 0 .. SM count - 1");
    if ((rc = locate_plan(*ds, &t))) return rc;
    if ((rc = locate_stage(t))) return rc;
    if (t.seg.host_src && p->sm_kernel == C3_SMK_BULK)
        return set_error(C3_EUNSUP, "the bulk copy kernel reads device memory only");
    out->mode = mode;
    out->sm_split = sm_split;
    out->priority = priority;
    rc = run_once(*ds, p, t, mode, sm_split, priority, out);
    out->status = rc;
    return rc;
}

int c3_time(const c3_problem* p, int mode, int sm_split, int priority, int warmup, int reps,
            c3_timing* per_rep) {
    if (!per_rep || reps < 1 || warmup < 0) return set_error(C3_EINVAL, "need reps >= 1, warmup >= 0, per_rep");
    if (mode < C3_MODE_SERIAL_SM || mode > C3_MODE_CONCURRENT_SM_RECLAIM) return set_error(C3_EINVAL, "unknown mode");
    if (priority != 0 && priority != 1) return set_error(C3_EINVAL, "priority must be 0 or 1");
    CollPlan t;
    int rc = check_problem(p, &t);
    if (rc) return rc;
    DeviceState* ds = device_state();
    if (!ds) return C3_ECUDA;
    if (sm_split < 0 || sm_split >= ds->sm_count) return set_error(C3_EINVAL, "sm_split must be 0 .. SM count - 1");
    if ((rc = locate_plan(*ds, &t))) return rc;
    if ((rc = locate_stage(t))) return rc;
    if (t.seg.host_src && p->sm_kernel == C3_SMK_BULK)
        return set_error(C3_EUNSUP, "the bulk copy kernel reads device memory only");
    cudaStream_t s0 = static_cast<cudaStream_t>(p->stream);
    const int engine = (mode == C3_MODE_CONCURRENT_CE || mode == C3_MODE_SERIAL_CE) ? C3_ENGINE_CE : C3_ENGINE_SM;
    if (p->settle_us > 0) {
        // the first settle period must start from an idle stream too
        cudaError_t e = cudaStreamSynchronize(s0);
        if (e != cudaSuccess) return set_cuda_error(e, "stream synchronize");
    }
    for (int it = 0; it < warmup + reps; ++it) {
        c3_timing r;
        std::memset(&r, 0, sizeof r);
        GemmLaunch gl;
        if ((rc = gemm_prepare(p->A, p->B, p->C, p->M, p->N, p->K, 0, &gl))) return rc;
        rc = time_phase(*ds, s0, p, "c3/GEMM alone", &r.t_gemm_iso,
                        [&] { return gemm_enqueue(gl, s0, ds->status, nullptr); });
        if (rc) return rc;
        rc = time_phase(*ds, s0, p, "c3/collective alone", &r.t_comm_iso, [&] {
            return launch_coll(*ds, t, engine, p->sm_kernel, p->coll_l2, p->ce_variant, p->comm_sms, false, s0, nullptr);
        });
        if (rc) return rc;
        rc = time_phase(*ds, s0, p, "c3/GEMM then collective", &r.t_serial_meas, [&] {
            int r1 = gemm_enqueue(gl, s0, ds->status, nullptr);
            return r1 ? r1 : launch_coll(*ds, t, engine, p->sm_kernel, p->coll_l2, p->ce_variant, p->comm_sms, false, s0, nullptr);
        });
        if (rc) return rc;
        settle(p);
        if (p->flush_buf && p->flush_bytes && (rc = l2_flush_launch(p->flush_buf, p->flush_bytes, s0))) return rc;
        r.mode = mode;
        r.sm_split = sm_split;
        r.priority = priority;
        rc = run_once(*ds, p, t, mode, sm_split, priority, &r);
        r.status = rc;
        if (rc) return rc;
        fill_metrics(&r);
        fill_bounds(&r, p, t, engine);
        if (it >= warmup) per_rep[it - warmup] = r;
    }
    return C3_OK;
}

}  // extern "C"
