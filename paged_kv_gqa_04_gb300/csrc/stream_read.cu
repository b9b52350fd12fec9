// stream_read.cu -- streaming-read ceiling of one launch.
//
// mainarch, decode-attention section: a pure device-memory streaming read
// is measured first and is the ceiling every decode kernel is held to. This
// kernel reads `bytes` of device memory once with 16-byte non-caching loads
// (each CTA strides over the buffer, eight independent loads in flight per
// thread per iteration) and folds them into one word per CTA, so that the
// time of one launch of a given size can be set beside the decode kernel's
// time for the same number of bytes.
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kThreads) stream_read_kernel(const uint4* __restrict__ buf, int64_t n16,
                                                               uint32_t* __restrict__ sink) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    uint32_t acc = 0;
    for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(buf + i + u * stride);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = ld_stream(buf + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ uint32_t red[kThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < kThreads / 32; ++w) r ^= red[w];
        sink[blockIdx.x] = r;
    }
}

}  // namespace

cudaError_t launch_stream_read(const void* buf, int64_t bytes, uint32_t* sink, int ctas, cudaStream_t s) {
    if (bytes <= 0) return cudaSuccess;
    stream_read_kernel<<<ctas, kThreads, 0, s>>>(static_cast<const uint4*>(buf), bytes / 16, sink);
    return cudaGetLastError();
}

}  // namespace pkv
