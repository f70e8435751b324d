/*
 * c3_api.h -- C ABI of libc3.so: concurrent computation and communication (C3)
 * on one GB300 (sm_103a).
 *
 * The operation follows "Optimizing ML Concurrent Computation and
 * Communication with GPU DMA Engines" (ConCCL, arXiv 2412.14335) as its review
 * pages describe it: a GEMM runs at the same time as a bulk collective data
 * movement (an all-gather or an all-to-all), and the quality of the overlap is
 * measured against the ideal speedup (T_gemm + T_comm) / max(T_gemm, T_comm)
 * taken from isolated runs (pith.science paper page: abstract, "The reading",
 * referee report summary).  Four ways of running the pair are offered: the
 * plain concurrent baseline, schedule prioritisation (collective first on a
 * high-priority stream), SM partitioning (disjoint SM budgets) and copy-engine
 * offload (the collective as driver memcpy transfers issued from the host,
 * with no kernel of this library), with the option of taking SMs away from
 * the GEMM while offloading (the paper's ConCCL_rp).
 *
 * The collective is emulated inside one device's memory: the buffers of
 * `nranks` virtual ranks are separate device allocations of this GPU.  The
 * sources of an all-gather or all-to-all may instead be page-locked host
 * memory, which puts the "remote" ranks across the CPU-GPU link.
 *
 * Which hardware moves the "copy-engine" bytes is the driver's choice.  On
 * GB300 with driver 580, a memcpy between two buffers of the same GPU runs
 * as driver-internal SM work (measured with range counters: SM instructions
 * and L1/TEX reads equal to the collective's bytes), while a memcpy from
 * page-locked host memory is host-to-device DMA.
 *
 * Conventions for every entry point
 *   - The caller owns all device memory and all streams passed in.  Device
 *     pointers are plain CUDA device addresses of the current device; host
 *     pointers are marked as such.  Nothing is freed or retained after return
 *     except where stated.
 *   - Streams are `cudaStream_t` values passed as `c3_stream` (void *); NULL
 *     means the legacy default stream.
 *   - The library owns a few internal objects per device, created on first use
 *     with that device current and released by c3_shutdown(): three CUDA
 *     streams (the forked collective's, the same at the highest priority, and
 *     a private stream for capturing memcpy graphs), CUDA events, up to 16
 *     cached memcpy graphs, a 16 KiB device status block
 *     (error word, %globaltimer stamps, per-CTA %smid residency records) and
 *     the kernels' function attributes.
 *   - Return value: C3_OK (0) or a negative c3_status.  On an argument error
 *     nothing is launched.  C3_ECUDA carries the CUDA error text in
 *     c3_last_error().  A device-side wait that gives up (a bounded spin on an
 *     mbarrier, about two seconds) is reported as C3_ETIMEOUT by the next
 *     synchronising call (c3_run, c3_time, c3_status_check).
 *   - Not thread-safe: one host thread drives one device at a time.
 */
#ifndef C3_API_H
#define C3_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *c3_stream; /* a cudaStream_t */

typedef enum {
    C3_OK = 0,
    C3_EINVAL = -1,   /* bad argument: null pointer, negative size, unknown enum */
    C3_EALIGN = -2,   /* pointer not 16-byte aligned, or size not a multiple of 16 bytes */
    C3_ECUDA = -3,    /* a CUDA runtime/driver call failed; text in c3_last_error() */
    C3_ETIMEOUT = -4, /* a bounded device wait gave up; results of that launch are void */
    C3_EUNSUP = -5    /* valid request this build does not support (e.g. nranks != 8 on the CE 2-D path) */
} c3_status;

typedef enum { C3_ENGINE_SM = 0, C3_ENGINE_CE = 1 } c3_engine;
typedef enum { C3_COLL_ALLGATHER = 0, C3_COLL_ALLTOALL = 1, C3_COLL_ALLREDUCE = 2 } c3_coll;

/* How the GEMM and the collective are run (see c3_run). */
typedef enum {
    C3_MODE_SERIAL_SM = 0,     /* GEMM, then the collective on SMs, one stream */
    C3_MODE_CONCURRENT_SM = 1, /* GEMM || collective on SMs (baseline / prioritised / partitioned) */
    C3_MODE_CONCURRENT_CE = 2, /* GEMM || collective as driver memcpy (ConCCL, ConCCL_rp) */
    C3_MODE_SERIAL_CE = 3,     /* GEMM, then the collective as driver memcpy, one stream */
    C3_MODE_CONCURRENT_SM_RECLAIM = 4 /* SM partitioning with reclaim (see c3_run) */
} c3_mode;

/* SM copy kernel flavour.  VEC: 16-byte vector loads/stores, no shared memory,
 * may share SMs with the GEMM.  BULK: cp.async.bulk global->shared->global
 * through a shared-memory ring, one CTA per SM; device-memory sources only
 * (C3_EUNSUP with a host source; AUTO then takes VEC). */
typedef enum { C3_SMK_AUTO = 0, C3_SMK_VEC = 1, C3_SMK_BULK = 2 } c3_sm_kernel;

/* L2 treatment of the SM collective's loads and stores.  NORMAL: default
 * caching.  EVICT_FIRST: no L1 allocation and an L2 evict-first policy, so the
 * bytes the collective touches once do not displace a concurrent GEMM's
 * operands -- the software counterpart of the pages' point that DMA transfers
 * bypass the caches ("What carries the argument"; Sections II-A, VI-A).
 * The memcpy path ignores it. */
typedef enum { C3_L2_NORMAL = 0, C3_L2_EVICT_FIRST = 1 } c3_l2_policy;

/* How the copy-engine path issues its transfers.  PER_SEGMENT: one
 * cudaMemcpyAsync (cudaMemcpyDefault) per segment (8 for the all-gather, R^2 for
 * the all-to-all).  STRIDED: the all-to-all as R cudaMemcpy2DAsync calls, one
 * per source rank (all-gathers as PER_SEGMENT).  GRAPH: the STRIDED calls
 * captured once into a CUDA graph, cached by buffer addresses and size (up to
 * 16 graphs, released by c3_shutdown), replayed with one launch.
 * GRAPH_PARALLEL: a cached CUDA graph of independent copy nodes (the 2-D
 * copies for the all-to-all; 1-D pieces of >= 8 MiB of each segment
 * otherwise, at most 64 nodes) that the driver may run at the same time.
 * Measured on GB300: alone it moves a >= 128 MiB all-gather as fast
 * as the SM kernel (5.8 TB/s at 256 MiB), but a GEMM running beside it slows
 * far more than beside the other variants, and later concurrent runs in the
 * same process do too -- opt-in only.  The pages' DMA collectives lose to the
 * compute-unit library below 32 MB on launch and synchronisation cost (Figure
 * 9); STRIDED and GRAPH cut the number of host calls per collective.
 * HOST_STAGED: every segment goes device -> page-locked host -> device as
 * two transfers per piece of at most 16 MiB (c3_problem.ce_stage holds the
 * pieces in between), replayed from a cached CUDA graph: the device-to-host
 * pieces form one chain, the host-to-device pieces another, and each piece's
 * second transfer waits for its first, so the two directions run at the same
 * time one piece apart.  Both hops are copy-engine DMA; no SM runs any part
 * of the collective.  It costs twice the CPU-GPU link traffic of the
 * collective's bytes and runs at the link's rate (on GB300 about 3.8 ms for
 * 1 GiB, against 0.16 ms for the SM kernel), so it pays only where a GEMM is
 * long enough to hide it.  Needs device sources (C3_EUNSUP for page-locked
 * host sources, which the other variants already reach by DMA). */
typedef enum {
    C3_CE_PER_SEGMENT = 0,
    C3_CE_STRIDED = 1,
    C3_CE_GRAPH = 2,
    C3_CE_GRAPH_PARALLEL = 3,
    C3_CE_HOST_STAGED = 4
} c3_ce_variant;

/* The taxonomy class of a C3 pair (paper Section III, 115% / 15% thresholds). */
typedef enum { C3_CLASS_G_LONG = 0, C3_CLASS_GC_EQUAL = 1, C3_CLASS_C_LONG = 2 } c3_class;

/* The taxonomy's other two axes (the pith.science verdict's summary of the
 * paper's taxonomy: compute- versus memory-bound GEMMs, latency- versus
 * bandwidth-bound collectives; Section III).
 *   GEMM: memory-bound when its arithmetic intensity 2MNK / (2MK + 2NK + 4MN)
 *     lies below the roofline ridge peak_flops / peak_bytes_per_s (compared
 *     cross-multiplied), compute-bound otherwise.
 *   Collective: bandwidth-bound when its isolated rate (output bytes /
 *     t_comm_iso) reaches half the plateau rate of the same engine's size
 *     sweep, latency-bound below -- the plateau threshold the referee's minor
 *     comment on Section III asks for in place of "latency does not grow with
 *     size".
 * UNKNOWN when the problem carries no peaks / no plateau for that engine. */
typedef enum { C3_BOUND_UNKNOWN = -1, C3_GEMM_COMPUTE = 0, C3_GEMM_MEMORY = 1 } c3_gemm_bound;
typedef enum { C3_COLL_LATENCY = 0, C3_COLL_BANDWIDTH = 1 } c3_coll_bound;

typedef struct {
    int device;           /* CUDA ordinal */
    int sm_count;         /* streaming multiprocessors */
    int l2_bytes;         /* L2 size */
    int smem_per_sm;      /* shared memory per SM, bytes */
    int smem_per_block;   /* opt-in maximum per CTA, bytes */
    int cc_major, cc_minor;
    int gemm_smem_bytes;  /* dynamic shared memory one GEMM CTA takes (largest tile) */
    int comm_default_sms; /* SM budget of the SM collective when none is given */
} c3_device_info;

/* Library version and device facts (initialises the current device). */
int c3_get_device_info(c3_device_info *out);
/* Message for a status code (static string; never NULL). */
const char *c3_strerror(int status);
/* Detail of the most recent C3_ECUDA / C3_ETIMEOUT on this host thread. */
const char *c3_last_error(void);
/* Synchronises `s`, then reads and clears the device status word: C3_OK, or
 * C3_ETIMEOUT if a kernel launched since the last check gave up a wait. */
int c3_status_check(c3_stream s);
/* Releases the library's per-device objects (streams, events, status block). */
int c3_shutdown(void);
/* Number of kernels this library has launched in this process (all devices),
 * counted on the host at each successful launch.  Memcpy transfers are not
 * counted, whatever hardware the driver runs them on. */
uint64_t c3_kernel_launches(void);

/*
 * GEMM:  C[m][n] = sum_k A[m][k] * B[n][k]            (the computation half of C3)
 *   A  device, bf16, M x K row-major (K contiguous), 16-byte aligned
 *   B  device, bf16, N x K row-major (the weight as an all-gather delivers it), 16-byte aligned
 *   C  device, fp32, M x N row-major, written in full (no accumulation into C)
 *   M, N >= 0 any value (ragged edges are masked); K >= 0 and K % 8 == 0
 *      (the TMA row pitch must be a multiple of 16 bytes; else C3_EALIGN);
 *      K == 0 writes zeros.  M*N == 0 launches nothing.
 *   sm_budget  number of persistent CTAs, one per SM (0 = every SM); values
 *      above the SM count are clamped.  The CTAs claim output tiles one at a
 *      time from a counter in the library's status block, so a CTA that is
 *      slowed or starts late does less of the work.
 * bf16 products are accumulated in fp32 on the tensor cores (tcgen05).
 * Asynchronous on `s`.
 */
int c3_gemm(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
            int sm_budget, c3_stream s);

/*
 * The launch c3_gemm would make for this shape and budget, without launching:
 * the tile width BN, the number of 128-row sub-tiles per CTA (1 or 2) and the
 * number of persistent CTAs.  Host only (reads the SM count of the current
 * device when sm_budget is 0).
 */
int c3_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_budget, int *bn, int *msub, int *ctas);

/*
 * All-gather over `nranks` virtual ranks of one device:
 *   out[r * shard_bytes + i] = shards[r][i]   for r < nranks, i < shard_bytes
 * (every rank's initial buffer concatenated in rank order: the check the
 * pith.science verdict's skeptic critique asks for, "concrete_test").
 *   shards  HOST array of nranks pointers (read during the call only), each to
 *           device memory of the current device or to page-locked host memory
 *           (cudaHostAlloc / cudaHostRegister); pageable or another device's
 *           memory is C3_EINVAL
 *   out     device, nranks * shard_bytes bytes; must not overlap any shard
 *   shard_bytes  multiple of 16 (else C3_EALIGN); 0 launches nothing
 *   nranks  1..64
 *   engine  C3_ENGINE_SM: an SM copy kernel on `sm_budget` SMs (0 = default
 *           budget; host shards are read with plain loads over the CPU-GPU
 *           link); C3_ENGINE_CE: the driver memcpy path, one transfer per
 *           shard replayed from a cached CUDA graph (C3_CE_GRAPH), sm_budget
 *           ignored.
 * Bit-exact byte copy.  Asynchronous on `s`.
 */
int c3_allgather(const void *const *shards, void *out, size_t shard_bytes, int nranks,
                 int engine, int sm_budget, c3_stream s);

/*
 * All-to-all over an nranks x nranks grid of equal blocks:
 *   out[(j * nranks + i) * block_bytes + b] = in[(i * nranks + j) * block_bytes + b]
 * rank i's send buffer is in[i*nranks*block_bytes ...), its block j goes to
 * receive slot i of rank j (the all-to-all the pages pair with the GEMM).
 *   in, out  nranks^2 * block_bytes bytes each, not overlapping; out is device
 *            memory, in is device or page-locked host memory (as for shards)
 *   block_bytes multiple of 16 (else C3_EALIGN); 0 launches nothing
 *   nranks  1..8 (the SM kernel's segment table holds 64 blocks)
 *   engine  as for c3_allgather (CE: one strided 2-D transfer per source rank,
 *           replayed from a cached CUDA graph)
 * Bit-exact.  Asynchronous on `s`.
 */
int c3_alltoall(const void *in, void *out, size_t block_bytes, int nranks, int engine,
                int sm_budget, c3_stream s);

/*
 * All-reduce of `nranks` fp32 vectors of `count` elements.
 *   engine C3_ENGINE_CE: decomposed the way the pages propose for DMA offload,
 *     a reduce-scatter, which needs arithmetic and runs on SMs, then an
 *     all-gather of the reduced chunks as driver memcpy (synthesis page,
 *     "Attack 1"; pith.science paper page, "Reading between the lines": a DMA
 *     engine has no arithmetic);
 *   engine C3_ENGINE_SM: one pass on SMs.  Each 16-byte vector of the sum is
 *     computed once and stored into every rank's row, so every input byte is
 *     read once and every output byte written once (2 * nranks * count * 4
 *     bytes; the reduce-scatter and copies of the copy-engine form move
 *     (3 * nranks - 1) * count * 4).
 *   inputs  HOST array of nranks device pointers, count floats each, 16-byte aligned
 *   out     device, nranks * count floats: row r (out + r*count) is rank r's result
 *   count   multiple of 4 * nranks (16-byte chunks; else C3_EALIGN); 0 launches nothing
 *   nranks  1..8
 * Every row ends as out[r][i] = ((0 + in_0[i]) + in_1[i]) + ... + in_{R-1}[i]
 * in fp32, rank order -- the same on every row, on either engine, and
 * bit-reproducible.  The SM work (the one pass, or the reduce-scatter) uses
 * sm_budget SMs (0 = default).  Asynchronous on `s`.
 */
int c3_allreduce(const float *const *inputs, float *out, size_t count, int nranks, int engine,
                 int sm_budget, c3_stream s);

/* One C3 problem: a GEMM and one collective, both on caller-owned buffers. */
typedef struct {
    /* GEMM (as c3_gemm) */
    const void *A;
    const void *B;
    float *C;
    int64_t M, N, K;
    /* collective */
    int coll;                  /* c3_coll */
    const void *const *shards; /* all-gather: HOST array of nranks pointers, each device or
                                  page-locked host memory (all-reduce: its nranks fp32 input
                                  vectors, device memory) */
    const void *send;          /* all-to-all: send buffer, device or page-locked host memory */
    void *recv;                /* output of the collective */
    size_t unit_bytes;         /* shard bytes (all-gather), block bytes (all-to-all) or bytes of one
                                  rank's fp32 vector (all-reduce; recv holds nranks of them) */
    int nranks;
    int comm_sms;              /* SM budget of the un-partitioned SM collective (0 = default) */
    int sm_kernel;             /* c3_sm_kernel */
    int coll_l2;               /* c3_l2_policy of the SM collective */
    int ce_variant;            /* c3_ce_variant of the copy-engine collective */
    /* optional L2 flush (c3_l2_flush) before each phase of c3_time
     * (caller-owned scratch, at least 2 x L2; NULL = no flush) */
    void *flush_buf;
    size_t flush_bytes;
    c3_stream stream;          /* runs fork from and join back to this stream */
    /* Timer options (c3_time).  Zero leaves each one off. */
    int settle_us;             /* idle time before each timed phase: the host sleeps this long after
                                  the previous phase completed (0..1000000 us).  A GB300 at its power
                                  limit runs a phase that follows an idle period at higher clocks than
                                  one that follows seconds of load, so without a common idle period
                                  the isolated and concurrent phases are timed in different power
                                  states. */
    double peak_flops;         /* dense bf16 tensor peak, FLOP/s: with peak_bytes_per_s, classifies
                                  the GEMM as compute- or memory-bound (0 = unknown) */
    double peak_bytes_per_s;   /* memory bandwidth peak, bytes/s (0 = unknown) */
    double coll_plateau_sm;    /* plateau rate of the SM collective over a size sweep, output bytes
                                  per second: classifies the collective as latency- or
                                  bandwidth-bound (0 = unknown) */
    double coll_plateau_ce;    /* the same for the copy-engine (memcpy) collective */
    /* Bounce buffer of C3_CE_HOST_STAGED: page-locked host memory (cudaHostAlloc or
     * cudaHostRegister), caller-owned, 16-byte aligned, at least the bytes the collective's
     * copies move (all-gather and all-to-all: the output's size; all-reduce: the output's
     * size, its all-gather half).  Read only when ce_variant is C3_CE_HOST_STAGED; NULL, too
     * small, misaligned or not page-locked is then C3_EINVAL (C3_EALIGN for alignment).  Its
     * contents are scratch. */
    void *ce_stage;
    size_t ce_stage_bytes;
} c3_problem;

/* Times in seconds. */
typedef struct {
    double t_gemm_iso;     /* GEMM alone, every SM                                  (c3_time) */
    double t_comm_iso;     /* collective alone on the engine the mode uses           (c3_time) */
    double t_serial;       /* t_gemm_iso + t_comm_iso: the serial time               (c3_time) */
    double t_serial_meas;  /* GEMM then collective on one stream, measured           (c3_time) */
    double t_conc;         /* start event to the later of the GEMM's and the collective's
                              completion events (events recorded right after each)  (c3_run)  */
    double t_ideal;        /* max(t_gemm_iso, t_comm_iso)                            (c3_time) */
    double s_ideal;        /* t_serial / t_ideal                                     (c3_time) */
    double s_real;         /* t_serial / t_conc                                      (c3_time) */
    double pct_ideal_gain; /* (s_real - 1) / (s_ideal - 1): share of the ideal gain  (c3_time) */
    double pct_ideal_ratio;/* s_real / s_ideal                                       (c3_time) */
    double t_gemm_dev;     /* GEMM kernel window by %globaltimer (first CTA start to last CTA end) */
    double t_comm_dev;     /* SM collective kernel window by %globaltimer (0 for CE) */
    double t_gemm_ev;      /* fork to GEMM completion, CUDA events (partitioned SM modes: to the
                              completion of the GEMM's stream, which also carries the
                              collective's second part) */
    double t_comm_ev;      /* fork to collective completion, CUDA events */
    int cls;               /* c3_class of (t_gemm_iso, t_comm_iso)                   (c3_time) */
    int mode, sm_split, priority;
    int gemm_ctas;         /* persistent GEMM CTAs launched */
    int comm_ctas;         /* SM collective CTAs launched (0 for CE) */
    int gemm_sms;          /* distinct SMs the GEMM CTAs ran on (%smid) */
    int comm_sms;          /* distinct SMs the collective CTAs ran on */
    int smid_overlap;      /* SMs on which a GEMM CTA and a collective CTA were resident at the
                              same time, by their %globaltimer windows (0 = the partition held) */
    int sms_shared_any;    /* SMs that ran CTAs of both kernels at any time during the run */
    int status;            /* C3_OK or the run's device status */
    int gemm_bound;        /* c3_gemm_bound of the problem's GEMM                     (c3_time) */
    int coll_bound;        /* c3_coll_bound of t_comm_iso on the mode's engine          (c3_time) */
} c3_timing;

/*
 * One C3 execution of `p` in `mode`, synchronised, timed.
 *   mode C3_MODE_CONCURRENT_SM:
 *     sm_split == 0: baseline -- the GEMM on every SM and the collective with
 *                    its default budget, free to share SMs;
 *     sm_split  > 0: SM partitioning -- the collective on sm_split SMs it holds
 *                    alone (its CTAs reserve enough shared memory that no GEMM
 *                    CTA fits beside them) and the GEMM on the others.
 *     priority == 1: schedule prioritisation -- the collective is launched
 *                    first, on the library's highest-priority stream; 0: the
 *                    collective's stream has default priority and the GEMM is
 *                    launched first (with sm_split > 0 the collective's first
 *                    part still goes first, see below).  (Pages: c3_sp, c3_rp
 *                    and their combination.)
 *   In every concurrent mode the GEMM runs on p->stream and the collective on
 *   a library stream forked from it by an event and joined back by another.
 *   mode C3_MODE_CONCURRENT_CE: the collective as driver memcpy transfers on
 *     its own stream (ConCCL); sm_split > 0 removes that many SMs from the GEMM
 *     (ConCCL_rp).  priority as above.  (Device-to-device copies run on SMs
 *     inside the driver on GB300; copies from page-locked host sources are DMA.)
 *   mode C3_MODE_CONCURRENT_SM_RECLAIM (sm_split >= 1): SM partitioning with
 *     reclaim -- the collective is launched first on sm_split SMs it holds
 *     alone, on the library's highest-priority stream so that its CTAs are
 *     dispatched before the GEMM's.  The GEMM's tiles are planned for the SM
 *     count - sm_split SMs it starts on, and it is launched on up to every
 *     SM: the GEMM CTAs that find no free SM start as soon as the
 *     collective's SMs free up and, since the GEMM claims its tiles
 *     dynamically, take only the tiles still left (none, when the tiles fit
 *     one wave on the SMs it started on).  The partition lasts as long as the
 *     collective, not as long as the GEMM.
 *     priority has no further effect in this mode.
 *   In both partitioned modes the collective is one launch group of SM-count
 *   CTAs: its first sm_split CTAs, launched before the GEMM, and the rest,
 *   launched right behind the GEMM on the GEMM's stream as its programmatic
 *   dependent (cudaLaunchAttributeProgrammaticStreamSerialization): every GEMM
 *   CTA signals on entry, so the hardware schedules the rest only once no GEMM
 *   CTA waits for an SM, and they run only on SMs the GEMM has left -- a
 *   collective that outlasts the GEMM widens onto them.  t_gemm_ev then times
 *   the GEMM's stream, the GEMM and that second part.  An all-reduce on the
 *   SM engine is such a group too: its one-pass kernel (see c3_allreduce)
 *   waits for nothing, so the whole all-reduce widens.
 *   mode C3_MODE_SERIAL_SM / _CE: GEMM then collective on one stream.
 * Fills t_conc, the device windows, CTA counts and %smid facts of `out`; the
 * fields marked (c3_time) are left 0.  Returns C3_OK, an argument error
 * (nothing launched) or the device status of the run.  If a launch fails after
 * the collective went out (prioritised and partitioned modes launch it first), the
 * call returns C3_ECUDA with p->stream still ordered after the collective, so
 * the caller may reuse the buffers once that stream has drained.
 */
int c3_run(const c3_problem *p, int mode, int sm_split, int priority, c3_timing *out);

/*
 * The C3 timer: `warmup` untimed repetitions, then `reps` timed repetitions,
 * each made of: GEMM alone (every SM), collective alone (the mode's engine,
 * default budget), serial (GEMM then collective), and the requested mode.
 * When p->settle_us is set, the host waits that long before each phase (after
 * synchronising p->stream once at entry); when p->flush_buf is set, L2 is then
 * flushed before each phase, outside its timed interval.  per_rep[r] (reps
 * entries, host memory) receives every field, with the speedups of repetition
 * r computed from that repetition's own isolated times, and the taxonomy
 * class and bounds of the pair.
 */
int c3_time(const c3_problem *p, int mode, int sm_split, int priority, int warmup, int reps,
            c3_timing *per_rep);

/*
 * The GEMM of c3_gemm for callers that cannot allocate device memory: code
 * that runs where cudaMalloc is unavailable or forbidden (a host framework
 * with its own fixed memory pool, a plugin called while a caller holds every
 * byte of the device, real-time code that may not enter the allocator).  The
 * pages have no counterpart of this entry point; it exists for those callers.
 *
 * Same arguments, result and ragged-edge handling as c3_gemm.  It allocates
 * nothing: it does not touch the library's per-device state (no streams,
 * events or status block are created), and calls no cudaMalloc, cudaFree or
 * allocating library routine.  The scratch the GEMM kernel writes (error
 * word, %globaltimer window, per-CTA SM records) is one file-scope device
 * array of 16 KiB, present on every GPU that loads libc3.so until the process
 * exits.  It records at most 256 CTAs: a launch that would need more (a GPU
 * with more than 256 SMs and sm_budget 0 or above 256) is refused with
 * C3_EUNSUP before anything is launched.
 *
 * The first call on each device does a one-time set-up with that device
 * current (looks up the array's device address, reads the SM count, sets the
 * kernels' shared-memory attribute); make that first call before any stream
 * capture.  Each call clears the scratch on `s` before the GEMM (the status
 * words and the tile-scheduler slot it takes), since the array keeps the
 * previous call's contents, also after a call whose wait gave up.  All calls
 * share the one array:
 * calls whose executions overlap on the GPU (different streams, no ordering)
 * race on it, and a caller must order them.
 *   check  0: asynchronous on `s` (like c3_gemm); device wait timeouts are
 *             then not reported.  Non-zero: synchronises `s` and returns
 *             C3_ETIMEOUT if a bounded device wait of this GEMM gave up.
 * K == 0 zero-fills C with cudaMemsetAsync.
 */
int c3_gemm_noalloc(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                    int sm_budget, c3_stream s, int check);

/*
 * Self-test of the library's failure detection: launches one kernel whose
 * single thread waits on an mbarrier phase with the same bounded wait the
 * GEMM and the bulk copy use, limited to `limit_ns` (1 ns .. 5 s, else
 * C3_EINVAL).  arrive = 1: the phase is completed first, the wait succeeds,
 * C3_OK.  arrive = 0: nothing completes the phase, the wait gives up after
 * the limit and the call returns C3_ETIMEOUT -- with the CUDA context intact.
 * Synchronises `s`.  The pages have no counterpart (failure handling is this
 * library's own).
 */
int c3_selftest_wait(uint64_t limit_ns, int arrive, c3_stream s);

/*
 * Host-side failure injection, so that a caller's error paths (and this
 * library's own recovery) can be tested without faulting a GPU.  Arms a
 * one-shot failure of the next call, on any thread, that reaches `site`:
 *   C3_FAULT_GEMM_LAUNCH     the GEMM kernel launch
 *   C3_FAULT_SM_COLL_LAUNCH  an SM collective kernel launch (copy or reduce-scatter)
 *   C3_FAULT_MEMCPY          the memcpy path's transfer calls
 *   C3_FAULT_DEVICE_INIT     the per-device initialisation (as if allocating the
 *                            status block were refused; takes effect on the next
 *                            initialisation, i.e. after c3_shutdown)
 * That step then launches nothing and returns C3_ECUDA, with c3_last_error()
 * naming the injection; work enqueued before it in the same call stays
 * enqueued.  C3_FAULT_NONE disarms.  Returns C3_OK, or C3_EINVAL for an
 * unknown site.  The pages have no counterpart.
 */
typedef enum {
    C3_FAULT_NONE = 0,
    C3_FAULT_GEMM_LAUNCH = 1,
    C3_FAULT_SM_COLL_LAUNCH = 2,
    C3_FAULT_MEMCPY = 3,
    C3_FAULT_DEVICE_INIT = 4
} c3_fault_site;
int c3_inject_fault(int site);

/*
 * Runtime heuristics of the pages (Section V-C).
 *
 * c3_sp_predict: schedule prioritisation -- returns 1 when the collective
 * should be launched first (it has fewer CTAs than the GEMM), else 0; the
 * pages' rule is to launch the lower-workgroup-count kernel first.
 *
 * c3_rp_predict: resource partitioning from a one-time slowdown table (the
 * pages' Figure 5) and a roofline at 70% efficiency.  Entry i of the table
 * says: with sms[i] SMs given to the collective, a compute-bound GEMM runs
 * gemm_compute[i] times slower than on every SM, a memory-bound GEMM
 * gemm_memory[i] times slower, and the collective coll[i] times slower than
 * on every SM.  The isolated times are taken from the roofline (GEMM:
 * max(flops / (0.7 * peak_flops), bytes / (0.7 * peak_bw)); collective:
 * 2 * coll_bytes / (0.7 * peak_bw)); the prediction for entry i is the larger
 * of the two scaled times; the entry with the smallest prediction wins.
 * Returns its SM count in *best_sms and its predicted time (s) in
 * *t_pred_best; t_pred_each (may be NULL) receives all n predictions.  Host
 * only; C3_EINVAL on empty tables, non-positive entries or sizes.
 *
 * c3_rp_predict_elastic: the same, for this library's partitions, which
 * dissolve when the GEMM ends (c3_run: the collective's second part widens
 * onto the SMs the GEMM leaves).  Where the collective would outlast the
 * GEMM (T_comm * coll[i] > T_gemm * slowdown_gemm[i]), it has moved the share
 * T_gemm * slowdown_gemm[i] / (T_comm * coll[i]) of its bytes by the time the
 * GEMM ends and moves the rest at the every-SM rate, so the prediction is
 *     T_comm + T_gemm * slowdown_gemm[i] * (1 - 1 / coll[i]);
 * otherwise it is the GEMM's scaled time, as in c3_rp_predict.  Same
 * arguments, outputs and errors.
 */
#define C3_RP_MAX 16
typedef struct {
    int n;
    int sms[C3_RP_MAX];
    double gemm_compute[C3_RP_MAX];
    double gemm_memory[C3_RP_MAX];
    double coll[C3_RP_MAX];
} c3_rp_table;

int c3_sp_predict(int gemm_ctas, int coll_ctas);
int c3_rp_predict(const c3_rp_table *t, double gemm_flops, double gemm_bytes, double coll_bytes,
                  double peak_flops, double peak_bytes_per_s, int *best_sms, double *t_pred_best,
                  double *t_pred_each);
int c3_rp_predict_elastic(const c3_rp_table *t, double gemm_flops, double gemm_bytes, double coll_bytes,
                          double peak_flops, double peak_bytes_per_s, int *best_sms, double *t_pred_best,
                          double *t_pred_each);

/*
 * Per-CTA windows of the last run (diagnostics; the pages have no
 * counterpart).  Every CTA of the GEMM kernel and of the SM collective
 * records the SM it ran on and its %globaltimer start and end in the
 * library's status block; c3_run (and the concurrent phase ending each
 * c3_time repetition) clears the block first, so after a c3_run these are
 * that run's kernels.  A c3_run in a serial mode gives the GEMM's CTAs timed
 * alone.  Collective CTAs that found no work left record nothing.
 *   kernel  0: the GEMM's CTAs; 1: the SM collective's CTAs
 *   out     host array of `max` entries, filled in CTA order (the first 256
 *           CTAs of a launch are recorded); times in seconds from the
 *           earliest start among the recorded CTAs of that kernel
 *   *n      receives the number of entries written
 * Synchronises the device.  C3_EINVAL on a bad kernel index or NULL output.
 */
typedef struct {
    int cta;          /* CTA index within its launch group */
    int smid;         /* %smid of the SM it ran on */
    double t_start;   /* seconds from the kernel's first recorded CTA start */
    double t_end;
} c3_cta_window;
int c3_cta_windows(int kernel, c3_cta_window *out, int max, int *n);

/* The L2 flush used between timed phases: writes `bytes` of zeros over `buf`
 * (device), then reads back its first half, so that L2 ends up holding clean
 * lines (a write-only flush would leave L2 full of dirty lines whose
 * write-back the next timed kernel pays for).  A complete flush needs
 * bytes >= 2 x L2.  Two SM kernels, asynchronous on `s`. */
int c3_l2_flush(void *buf, size_t bytes, c3_stream s);

#ifdef __cplusplus
}
#endif
#endif /* C3_API_H */
