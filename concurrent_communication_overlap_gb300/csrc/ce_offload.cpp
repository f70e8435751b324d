// ce_offload.cpp -- the collective as copy-engine transfers (the DMA offload).
//
// ConCCL breaks each collective into individual transfers and hands them to
// the GPU's DMA engines from the CPU, so that no compute unit and no L1/L2
// capacity is spent on the data movement ("Optimizing ML Concurrent
// Computation and Communication with GPU DMA Engines", pith.science paper
// page, "What carries the argument"; Sections VI-A/VI-B).  CUDA exposes no
// per-engine queue; the portable equivalent is device-to-device
// cudaMemcpyAsync on a dedicated stream, which the driver gives to a copy
// engine.  Whether any SM kernel ran for these transfers is checked by
// profiling (kernel launch list) rather than assumed.
//
// Three ways to issue them (the pages' DMA path is 4x slower than the
// CU-based library below 32 MB because of launch and synchronisation cost,
// Figure 9; the variants below attack that cost):
//   PER_SEGMENT  one cudaMemcpyAsync per segment (8 for an all-gather, R^2 for
//                an all-to-all) -- the direct algorithm;
//   STRIDED      the all-to-all as R cudaMemcpy2DAsync calls, one per source
//                rank (its R blocks land R blocks apart); all-gathers as above;
//   GRAPH        the STRIDED calls captured once into a CUDA graph (cached by
//                buffer addresses and size) and replayed with one launch.
#include "c3_internal.h"

#include <cstring>

namespace c3 {

static int ce_per_segment(const SegTable& t, cudaStream_t s) {
    for (int i = 0; i < t.nseg; ++i) {
        cudaError_t e = cudaMemcpyAsync(t.dst[i], t.src[i], (size_t)t.seg_bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync (copy engine)");
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
                                          cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpy2DAsync (copy engine)");
    }
    return 0;
}

// Small cache of instantiated graphs, keyed by the exact segment table.
struct GraphEntry {
    bool used = false;
    int device = -1;
    SegTable key;
    cudaGraphExec_t exec = nullptr;
    unsigned long long stamp = 0;
};
constexpr int kGraphCache = 16;
static GraphEntry g_graphs[kGraphCache];
static unsigned long long g_graph_clock = 0;

static bool same_table(const SegTable& a, const SegTable& b) {
    if (a.nseg != b.nseg || a.seg_bytes != b.seg_bytes) return false;
    for (int i = 0; i < a.nseg; ++i)
        if (a.src[i] != b.src[i] || a.dst[i] != b.dst[i]) return false;
    return true;
}

static int ce_graph(const SegTable& t, cudaStream_t s, cudaStream_t capture_stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
    GraphEntry* hit = nullptr;
    for (auto& g : g_graphs)
        if (g.used && g.device == dev && same_table(g.key, t)) hit = &g;
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
        e = cudaStreamBeginCapture(capture_stream, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamBeginCapture");
        int rc = ce_strided(t, capture_stream);
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(capture_stream, &graph);
        if (rc) {
            if (graph) cudaGraphDestroy(graph);
            return rc;
        }
        if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamEndCapture");
        e = cudaGraphInstantiate(&victim->exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphInstantiate");
        victim->used = true;
        victim->device = dev;
        victim->key = t;
        hit = victim;
    }
    hit->stamp = ++g_graph_clock;
    e = cudaGraphLaunch(hit->exec, s);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaGraphLaunch");
    return 0;
}

int copy_ce_launch(const SegTable& t, int variant, cudaStream_t s, cudaStream_t capture_stream) {
    if (t.nseg <= 0 || t.seg_bytes == 0) return 0;
    if (variant == kCeStrided) return ce_strided(t, s);
    if (variant == kCeGraph) return ce_graph(t, s, capture_stream);
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
