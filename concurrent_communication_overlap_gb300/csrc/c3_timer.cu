// c3_timer.cu -- device side of the C3 timer and small utility kernels.
//
// The C3 timer reports isolated, serial, concurrent and ideal times (the
// paper's Section IV-B3 ideal speedup needs isolated GEMM and collective
// times; its concurrent runs need the time from fork to join).  Host-side CUDA
// events give those intervals; the kernels themselves add device evidence:
// each CTA of the GEMM and of the SM collective stamps %globaltimer at start
// (atomicMin) and end (atomicMax) and sets its SM's bit (%smid) in the
// device status block.  This file holds the kernels that reset that block
// and the zero-fill kernel (L2 flush between timed phases, K == 0 GEMMs).
#include "c3_device.cuh"
#include "c3_internal.h"

namespace c3 {

__global__ void status_reset_kernel(DevStatus* st) {
    const int i = threadIdx.x;
    if (i == 0) {
        st->error = 0;
        st->where = 0;
        st->gemm_t0 = ~0ull;
        st->gemm_t1 = 0;
        st->comm_t0 = ~0ull;
        st->comm_t1 = 0;
    }
    if (i < 8) {
        st->smid_gemm[i] = 0;
        st->smid_comm[i] = 0;
    }
    if (i < kCtaRecs) {
        st->gemm_rec[i] = CtaRec{0, 0, 0, 0};
        st->comm_rec[i] = CtaRec{0, 0, 0, 0};
    }
}

// Writes zeros with 16-byte stores, grid-stride; a byte tail (< 16) by thread 0.
__global__ void zero_fill_kernel(uint8_t* buf, size_t bytes) {
    const size_t nvec = bytes >> 4;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    uint4 z = make_uint4(0, 0, 0, 0);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride)
        reinterpret_cast<uint4*>(buf)[i] = z;
    if (blockIdx.x == 0 && threadIdx.x == 0)
        for (size_t b = nvec << 4; b < bytes; ++b) buf[b] = 0;
}

int status_reset_launch(DevStatus* st, cudaStream_t s) {
    status_reset_kernel<<<1, kCtaRecs, 0, s>>>(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "status reset launch");
    count_launch();
    return 0;
}

int zero_fill_launch(void* buf, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return 0;
    if (((uintptr_t)buf & 15u) != 0) return set_error(-2, "zero fill needs a 16-byte aligned buffer");
    DeviceState* ds = device_state();
    if (!ds) return -3;
    size_t nvec = bytes >> 4;
    size_t want = (nvec + 255) / 256;
    int grid = (int)(want < (size_t)ds->sm_count * 4 ? (want ? want : 1) : (size_t)ds->sm_count * 4);
    zero_fill_kernel<<<grid, 256, 0, s>>>(static_cast<uint8_t*>(buf), bytes);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_cuda_error(e, "zero fill launch");
    count_launch();
    return 0;
}

}  // namespace c3
