// c3_internal.h -- declarations shared by the translation units of libc3.so
// (host side).  Not installed; the public boundary is include/c3_api.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace c3 {

// One CTA's residency: the SM it ran on and its %globaltimer window.
struct CtaRec {
    unsigned int smid;
    unsigned int used;             // 1 once written
    unsigned long long t0, t1;
};

constexpr int kCtaRecs = 256;      // CTAs recorded per kernel (the first 256)
constexpr int kSchedSlots = 64;    // GEMM tile-scheduler counters, used round-robin by launches
constexpr int kMaxRanksAr = 8;     // ranks of an all-reduce

// Device status block (library-owned, reset before each timed run).
struct DevStatus {
    int error;                     // 0, or a negative c3_status (first writer wins)
    int where;                     // code of the wait that gave up
    unsigned int gemm_started;     // GEMM CTAs that have started since the last reset
    int pad1;
    unsigned long long gemm_t0;    // min CTA start of the GEMM (%globaltimer, ns)
    unsigned long long gemm_t1;    // max CTA end
    unsigned long long comm_t0;    // same for the SM collective
    unsigned long long comm_t1;
    unsigned int smid_gemm[8];     // bitmap of SMs that ran a GEMM CTA (256 SMs max)
    unsigned int smid_comm[8];     // bitmap of SMs that ran a collective CTA
    CtaRec gemm_rec[kCtaRecs];     // per-CTA residency, indexed by blockIdx.x
    CtaRec comm_rec[kCtaRecs];
    // Dynamic tile scheduler of the persistent GEMM: per slot, the next tile
    // to hand out and the number of CTAs done.  A launch takes one slot; its
    // last CTA puts both back to zero.  Zeroed when the block is created;
    // the per-run reset leaves them alone (a GEMM of another stream may be
    // using a slot).
    unsigned int sched[kSchedSlots][2];
    // Work counters of the SM collective kernels, the same way: per slot, the
    // next work unit and the number of CTAs done.  One slot serves a launch
    // group -- one launch, or several on different streams that share the
    // collective's work -- and its last CTA puts the slot back to zero.
    unsigned int coll_sched[kSchedSlots][2];
};

constexpr size_t kStatusBytes = 16384;
static_assert(sizeof(DevStatus) <= kStatusBytes, "status block too small");

constexpr int kMaxSegs = 64;

// A collective as a list of equal-size byte segments src[i] -> dst[i].
enum { kSegAllGather = 0, kSegAllToAll = 1, kSegAllReduce = 2 };

// The reduce-scatter half of an all-reduce of nranks fp32 vectors of `count`
// elements: chunk c (count / nranks elements) of the rank-order sum goes to
// row c of `out` (nranks rows of `count` floats).
struct RsTable {
    const float* in[kMaxRanksAr];
    float* out;
    uint64_t count;
    uint64_t chunk;
    int nranks;
    int pad;
};

struct SegTable {
    const uint8_t* src[kMaxSegs];
    uint8_t* dst[kMaxSegs];
    int nseg;
    int kind;       // kSegAllGather or kSegAllToAll
    uint64_t seg_bytes;
    int nranks;
    int host_src;   // 1: at least one source is page-locked host memory (src[] holds its device address)
};

enum { kCePerSegment = 0, kCeStrided = 1, kCeGraph = 2, kCeGraphParallel = 3, kCeHostStaged = 4 };

// A collective as launched: an optional reduce-scatter pass on SMs (all-reduce
// only) followed by the segment copies on the chosen engine.
struct CollPlan {
    SegTable seg;
    RsTable rs;
    bool has_rs = false;
    uint8_t* stage = nullptr;  // page-locked host bounce buffer of the host-staged copy-engine variant
};

enum { kSmkVec = 1, kSmkBulk = 2 };

// Per-device state owned by the library.
struct DeviceState {
    int device = -1;
    int sm_count = 0;
    int l2_bytes = 0;
    int smem_per_sm = 0;
    int smem_per_block = 0;
    int cc_major = 0, cc_minor = 0;
    cudaStream_t s_comm = nullptr;     // the forked collective, default priority
    cudaStream_t s_comm_hi = nullptr;  // highest priority
    cudaStream_t s_capture = nullptr;  // private stream for capturing copy-engine graphs
    cudaEvent_t ev[8] = {};
    DevStatus* status = nullptr;       // device status block
    unsigned int next_sched = 0;       // round-robin scheduler slot
    unsigned int next_coll_sched = 0;  // round-robin copy work-counter slot
    bool ready = false;
};

// Returns the state of the current device, initialising it on first use.
// nullptr on failure (error text recorded).
DeviceState* device_state();

// Host-side count of kernels launched (c3_kernel_launches).
void count_launch();

// Error plumbing (thread-local text for c3_last_error).
int set_cuda_error(cudaError_t e, const char* what);
int set_error(int code, const char* what);

// Kernels' host launchers.  Return 0 or a negative c3_status.
int gemm_launch(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                int sm_budget, cudaStream_t s, DevStatus* st, int* ctas_out);

// A GEMM planned on the host (tile configuration, grid, tensor maps), ready to
// enqueue: the timed paths prepare before their start event so that host-side
// planning is not counted as device time.
struct GemmLaunch {
    int kind = 0;  // 0: nothing to do, 1: zero fill (K == 0), 2: the kernel
    float* C = nullptr;
    int64_t M = 0, N = 0, K = 0;
    int ci = 0, grid = 0, num_kb = 0;
    int64_t num_m = 0, num_n = 0;
    int has_mc = 0;  // mc (the fp32 output as a TMA store target) is valid: N % 4 == 0
    int static_first = 1;  // CTA b starts on tile b; 0 when CTAs may start late (reclaim)
    CUtensorMap ma, mb, mc;
};
int gemm_prepare(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K, int sm_budget,
                 GemmLaunch* g);
int gemm_enqueue(const GemmLaunch& g, cudaStream_t s, DevStatus* st, int* ctas_out);
void gemm_sched_reset(DevStatus* st);  // zero every scheduler slot (host; after an aborted launch)
int gemm_describe(int64_t M, int64_t N, int64_t K, int cap, int* bn, int* msub, int* grid);
int gemm_smem_bytes();  // dynamic shared memory of the largest GEMM tile configuration
int gemm_init_device();  // function attributes; once per device

// A group of SM copy launches sharing one work counter: `total_ctas` CTAs over
// every launch of the group; each launch numbers its CTAs from `cta_base`.
// The first part (CTAs 0 .. static_ctas-1, launched first) starts on fixed
// work units; every later unit is claimed from the counter.
struct CopyGroup {
    unsigned int* work = nullptr;  // DevStatus::coll_sched slot
    int total_ctas = 0;
    int static_ctas = 0;
};
// Picks the next work-counter slot of the device (round robin) for a group of
// total_ctas CTAs whose first launch part has first_ctas CTAs.
CopyGroup copy_group(DeviceState& ds, int total_ctas, int first_ctas);
// gate_need > 0: each CTA of this launch first reads st->gemm_started and, if
// fewer than gate_need GEMM CTAs have started, leaves at once without work (it
// was dispatched before a GEMM whose CTAs still wait for SMs).
// dependent: launched with programmatic stream serialization, right after the
// GEMM on the GEMM's stream, so that the hardware schedules it only once every
// GEMM CTA has started (the GEMM signals griddepcontrol.launch_dependents on
// entry); the launch does not wait for the GEMM to finish.
int copy_sm_launch(const SegTable& t, int ctas, int cta_base, const CopyGroup& g, int flavour, int smem_reserve,
                   int l2_stream, cudaStream_t s, DevStatus* st, int* ctas_out, unsigned gate_need = 0,
                   bool dependent = false);
// Largest number of work units (64 KiB rounds / 32 KiB chunks) a collective may
// have: the 32-bit counters stay far from wrapping.
bool copy_units_fit(const SegTable& t);
int copy_init_device(int max_reserve);
int reduce_scatter_launch(const RsTable& t, int ctas, int smem_reserve, cudaStream_t s, DevStatus* st,
                          int* ctas_out);
// The whole all-reduce `r` on SMs in one pass (each sum computed once and
// stored into every rank's row), as one launch of a launch group, the group's
// counter as for copy_sm_launch: `ctas` CTAs numbered from cta_base;
// gate_need and dependent as for copy_sm_launch.
int allreduce_sm_launch(const RsTable& r, int ctas, int cta_base, const CopyGroup& g, int smem_reserve,
                        int l2_stream, cudaStream_t s, DevStatus* st, int* ctas_out, unsigned gate_need = 0,
                        bool dependent = false);
int bulk_copy_smem_bytes();

// `stage`: the page-locked host bounce buffer of kCeHostStaged (at least
// nseg * seg_bytes bytes), ignored by the other variants.
int copy_ce_launch(const SegTable& t, int variant, cudaStream_t s, cudaStream_t capture_stream,
                   uint8_t* stage = nullptr);

// One-shot host-side failure injection (c3_inject_fault): true, and disarmed,
// when `site` is the armed site.  Site values are those of c3_fault_site.
enum { kFaultGemmLaunch = 1, kFaultSmCollLaunch = 2, kFaultMemcpy = 3, kFaultDeviceInit = 4 };
bool take_fault(int site);
void ce_release_graphs(int device);

int status_reset_launch(DevStatus* st, cudaStream_t s);
int selftest_wait_launch(DevStatus* st, unsigned long long limit_ns, int arrive, cudaStream_t s);
int zero_fill_launch(void* buf, size_t bytes, cudaStream_t s);
int l2_flush_launch(void* buf, size_t bytes, cudaStream_t s);

}  // namespace c3
