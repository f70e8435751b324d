// ce_offload.cpp -- the collective as driver memcpy transfers (the DMA-offload mode).
//
// ConCCL breaks each collective into individual transfers and hands them to
// the GPU's DMA engines from the CPU, so that no compute unit and no L1/L2
// capacity is spent on the data movement ("Optimizing ML Concurrent
// Computation and Communication with GPU DMA Engines", pith.science paper
// page, "What carries the argument"; Sections VI-A/VI-B).  CUDA exposes no
// per-engine queue.  This file issues the transfers through cudaMemcpyAsync
// and its 2-D and graph forms on a dedicated stream, and lets the driver pick
// the engine (cudaMemcpyDefault, so a source may also be page-locked host
// memory).
//
// Which engine the driver picks is measured, not assumed.  On GB300 with
// driver 580 a copy between two device buffers of the same GPU runs as
// driver-internal SM work: its profiled range executes SM instructions and
// reads the collective's bytes through L1/TEX, in every form below.  A copy
// whose source is page-locked host memory is host-to-device DMA.
//
// The ways to issue the transfers (the pages' DMA path is 4x slower than the
// CU-based library below 32 MB because of launch and synchronisation cost,
// Figure 9; the variants below attack that cost):
//   PER_SEGMENT  one cudaMemcpyAsync per segment (8 for an all-gather, R^2 for
//                an all-to-all) -- the direct algorithm;
//   STRIDED      the all-to-all as R cudaMemcpy2DAsync calls, one per source
//                rank (its R blocks land R blocks apart); all-gathers as above;
//   GRAPH        the STRIDED calls captured once into a CUDA graph (cached by
//                buffer addresses and size) and replayed with one launch.
//   GRAPH_PARALLEL  a CUDA graph of independent copy nodes (strided 2-D nodes
//                for the all-to-all, 1-D pieces otherwise), which the driver
//                may run at the same time.  Measured on GB300: as fast as the
//                SM kernel alone for all-gathers of >= 128 MiB, but a
//                concurrent GEMM runs much slower beside it, and so do later
//                concurrent runs in the same process.  Opt-in.
//   HOST_STAGED  each segment device -> page-locked host -> device, two DMA
//                transfers per piece, as a cached graph (build_graph_staged).
//                The one way on this driver to move a collective between two
//                device buffers with copy engines and no SM: the pages' DMA
//                offload, paid for with two crossings of the CPU-GPU link.
#include "c3_internal.h"

#include <cstring>

namespace c3 {

static int ce_per_segment(const SegTable& t, cudaStream_t s) {
    for (int i = 0; i < t.nseg; ++i) {
        cudaError_t e = cudaMemcpyAsync(t.dst[i], t.src[i], (size_t)t.seg_bytes, cudaMemcpyDefault, s);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync (collective segment)");
    }
    return 0;
}

static int ce_strided(const SegTable& t, cudaStream_t s) {
    if (t.kind != kSegAllToAll || t.nranks < 1) return ce_per_segment(t, s);
    const int R = t.nranks;
    const size_t B = (size_t)t.seg_bytes;
    for (int i = 0; i < R; ++i) {
        // source rank i: blocks j = 0..R-1 contiguous at src[i*R]; block j goes to
        // dst[i*R + j] = out + (j*R + i)*B, i.e. R*B apart starting at dst[i*R].
        cudaError_t e = cudaMemcpy2DAsync(t.dst[i * R], (size_t)R * B, t.src[i * R], B, B, (size_t)R,
                                          cudaMemcpyDefault, s);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpy2DAsync (collective rank)");
    }
    return 0;
}

// Small cache of instantiated graphs, keyed by the exact segment table.
struct GraphEntry {
    bool used = false;
    int variant = kCeGraph;  // kCeGraph, kCeGraphParallel or kCeHostStaged
    int device = -1;
    uint8_t* stage = nullptr;
    SegTable key;
    cudaGraphExec_t exec = nullptr;
    unsigned long long stamp = 0;
};
constexpr int kGraphCache = 16;
static GraphEntry g_graphs[kGraphCache];
static unsigned long long g_graph_clock = 0;

// The whole table is the key: the layout (kind, ranks) decides how the
// captured graph issues the copies, and the source's memory type how the
// driver carries them.
static bool same_table(const SegTable& a, const SegTable& b) {
    if (a.nseg != b.nseg || a.seg_bytes != b.seg_bytes || a.kind != b.kind || a.nranks != b.nranks ||
        a.host_src != b.host_src)
        return false;
    for (int i = 0; i < a.nseg; ++i)
        if (a.src[i] != b.src[i] || a.dst[i] != b.dst[i]) return false;
    return true;
}

// Builds a graph directly, with no edges between the copy nodes, so that the
// driver may run them at the same time (a stream-captured graph would chain
// them in issue order).  The all-to-all uses one strided 2-D node
// per source rank; other collectives one 1-D node per segment, each segment
// cut into pieces of at least kPieceBytes when there is room (at most 64
// nodes), so that large transfers can proceed in parallel.
constexpr uint64_t kPieceBytes = 8ull << 20;

static int build_graph_parallel(const SegTable& t, cudaGraphExec_t* exec) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphCreate");
    auto fail = [&](cudaError_t err, const char* what) {
        cudaGraphDestroy(graph);
        return set_cuda_error(err, what);
    };
    cudaGraphNode_t node;
    if (t.kind == kSegAllToAll && t.nranks >= 1) {
        const int R = t.nranks;
        const size_t B = (size_t)t.seg_bytes;
        for (int i = 0; i < R; ++i) {
            cudaMemcpy3DParms prm = {};
            prm.srcPtr = make_cudaPitchedPtr(const_cast<uint8_t*>(t.src[i * R]), B, B, (size_t)R);
            prm.dstPtr = make_cudaPitchedPtr(t.dst[i * R], (size_t)R * B, B, (size_t)R);
            prm.extent = make_cudaExtent(B, (size_t)R, 1);
            prm.kind = cudaMemcpyDefault;
            e = cudaGraphAddMemcpyNode(&node, graph, nullptr, 0, &prm);
            if (e != cudaSuccess) return fail(e, "cudaGraphAddMemcpyNode (2-D)");
        }
    } else {
        uint64_t pieces = t.seg_bytes / kPieceBytes;
        const uint64_t max_pieces = (uint64_t)(64 / (t.nseg > 0 ? t.nseg : 1));
        if (pieces > max_pieces) pieces = max_pieces;
        if (pieces < 1) pieces = 1;
        const uint64_t step = ((t.seg_bytes / pieces) + 15) & ~15ull;
        for (int i = 0; i < t.nseg; ++i)
            for (uint64_t off = 0; off < t.seg_bytes; off += step) {
                const uint64_t n = (t.seg_bytes - off) < step ? (t.seg_bytes - off) : step;
                e = cudaGraphAddMemcpyNode1D(&node, graph, nullptr, 0, t.dst[i] + off, t.src[i] + off, (size_t)n,
                                             cudaMemcpyDefault);
                if (e != cudaSuccess) return fail(e, "cudaGraphAddMemcpyNode1D");
            }
    }
    e = cudaGraphInstantiate(exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphInstantiate");
    return 0;
}

// The STRIDED calls captured from one stream: the copy nodes form a chain in
// issue order, exactly like the stream-issued variants.
static int build_graph_captured(const SegTable& t, cudaStream_t capture_stream, cudaGraphExec_t* exec) {
    cudaError_t e = cudaStreamBeginCapture(capture_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamBeginCapture");
    int rc = ce_strided(t, capture_stream);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(capture_stream, &graph);
    if (rc) {
        if (graph) cudaGraphDestroy(graph);
        return rc;
    }
    if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphInstantiate");
    return 0;
}

// HOST_STAGED: piece k of segment i (at most kStagePiece bytes, at offset
// off) is two nodes, src[i] + off -> stage + i * seg_bytes + off (device to
// host) and back to dst[i] + off (host to device).  The device-to-host nodes
// form one chain and the host-to-device nodes another, and each piece's
// second node also waits for its first: the two directions, which have
// engines of their own, run at the same time one piece apart.  Pieces grow
// past kStagePiece only to keep the graph within kStageMaxPieces pieces.
constexpr uint64_t kStagePiece = 16ull << 20;
constexpr uint64_t kStageMaxPieces = 512;

static int build_graph_staged(const SegTable& t, uint8_t* stage, cudaGraphExec_t* exec) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphCreate");
    auto fail = [&](cudaError_t err, const char* what) {
        cudaGraphDestroy(graph);
        return set_cuda_error(err, what);
    };
    const uint64_t total = t.seg_bytes * (uint64_t)t.nseg;
    uint64_t piece = kStagePiece;
    if (total / piece + (uint64_t)t.nseg > kStageMaxPieces) piece = total / (kStageMaxPieces - (uint64_t)t.nseg) + 1;
    piece = (piece + 15) & ~15ull;
    cudaGraphNode_t prev_d2h = nullptr, prev_h2d = nullptr;
    for (int i = 0; i < t.nseg; ++i)
        for (uint64_t off = 0; off < t.seg_bytes; off += piece) {
            const uint64_t n = (t.seg_bytes - off) < piece ? (t.seg_bytes - off) : piece;
            uint8_t* host = stage + (uint64_t)i * t.seg_bytes + off;
            cudaGraphNode_t d2h = nullptr, h2d = nullptr;
            e = cudaGraphAddMemcpyNode1D(&d2h, graph, prev_d2h ? &prev_d2h : nullptr, prev_d2h ? 1 : 0, host,
                                         t.src[i] + off, (size_t)n, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return fail(e, "cudaGraphAddMemcpyNode1D (device to host)");
            cudaGraphNode_t deps[2] = {d2h, prev_h2d};
            e = cudaGraphAddMemcpyNode1D(&h2d, graph, deps, prev_h2d ? 2 : 1, t.dst[i] + off, host, (size_t)n,
                                         cudaMemcpyHostToDevice);
            if (e != cudaSuccess) return fail(e, "cudaGraphAddMemcpyNode1D (host to device)");
            prev_d2h = d2h;
            prev_h2d = h2d;
        }
    e = cudaGraphInstantiate(exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphInstantiate");
    return 0;
}

static int ce_graph(const SegTable& t, int variant, cudaStream_t s, cudaStream_t capture_stream,
                    uint8_t* stage = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
    GraphEntry* hit = nullptr;
    for (auto& g : g_graphs)
        if (g.used && g.device == dev && g.variant == variant && g.stage == stage && same_table(g.key, t)) hit = &g;
    if (!hit) {
        GraphEntry* victim = &g_graphs[0];
        for (auto& g : g_graphs) {
            if (!g.used) {
                victim = &g;
                break;
            }
            if (g.stamp < victim->stamp) victim = &g;
        }
        if (victim->used && victim->exec) cudaGraphExecDestroy(victim->exec);
        *victim = GraphEntry();
        int rc = variant == kCeGraphParallel ? build_graph_parallel(t, &victim->exec)
                 : variant == kCeHostStaged  ? build_graph_staged(t, stage, &victim->exec)
                                             : build_graph_captured(t, capture_stream, &victim->exec);
        if (rc) return rc;
        victim->used = true;
        victim->variant = variant;
        victim->stage = stage;
        victim->device = dev;
        victim->key = t;
        hit = victim;
    }
    hit->stamp = ++g_graph_clock;
    e = cudaGraphLaunch(hit->exec, s);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphLaunch");
    return 0;
}

int copy_ce_launch(const SegTable& t, int variant, cudaStream_t s, cudaStream_t capture_stream, uint8_t* stage) {
    if (t.nseg <= 0 || t.seg_bytes == 0) return 0;
    if (take_fault(kFaultMemcpy)) return set_error(-3, "injected failure: memcpy transfer");
    if (variant == kCeStrided) return ce_strided(t, s);
    if (variant == kCeGraph || variant == kCeGraphParallel) return ce_graph(t, variant, s, capture_stream);
    if (variant == kCeHostStaged) {
        if (!stage) return set_error(-1, "host-staged copies need a bounce buffer");
        return ce_graph(t, variant, s, capture_stream, stage);
    }
    return ce_per_segment(t, s);
}

void ce_release_graphs(int device) {
    for (auto& g : g_graphs)
        if (g.used && g.device == device) {
            if (g.exec) cudaGraphExecDestroy(g.exec);
            g = GraphEntry();
        }
}

}  // namespace c3
