// copy.cu -- byte copy by the SMs between any two device-accessible buffers:
// device memory, or page-locked host memory, which on GB300 the SMs address
// directly over NVLink-C2C (unified addressing). For the few hundred KB a
// decode step moves between host and device this avoids the copy engines'
// set-up latency, and as a programmatic dependent the copy of a step's
// result is launched while the kernel that wrote it is still running (and
// waits for it); the grid after the copy starts only once the copy is done.
//
// Each thread moves 16-byte words (both pointers 16-byte aligned) or single
// bytes; the grid covers the buffer in one pass up to four CTAs per SM,
// then loops.
#include <algorithm>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) copy_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src,
                                                        int64_t bytes, int vec16) {
    // The source may be written by the preceding grid. No early trigger: the
    // next grid (a decode reads its block tables and seq_lens before its own
    // wait) starts only once this copy has finished.
    grid_dep_wait();
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t nth = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t done = 0;
    if (vec16) {
        const int64_t n16 = bytes >> 4;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        for (int64_t i = tid; i < n16; i += nth) d4[i] = s4[i];
        done = n16 << 4;
    }
    for (int64_t i = done + tid; i < bytes; i += nth) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
    if (bytes == 0) return cudaSuccess;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int vec16 = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
    const int64_t items = vec16 ? (bytes + 15) / 16 : bytes;
    const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>((items + kThreads - 1) / kThreads, 4 * sms));
    return launch_dependent(copy_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kThreads), 0, s,
                            static_cast<uint8_t*>(dst), static_cast<const uint8_t*>(src), bytes, vec16);
}

}  // namespace pkv
