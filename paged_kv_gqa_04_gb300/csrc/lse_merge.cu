// lse_merge.cu -- log-sum-exp merge of split-K decode partials.
//
// mainarch, decode-attention section: the split-KV partials are combined by
// their log-sum-exp weights; Loom Kernels, "Attention" row: local
// split-K/LSE merge.
//
// One warp per (sequence, query head) row. The warp reads the row's S LSE
// values, forms M = max and the weights w_s = exp(lse_s - M), then each lane
// accumulates D/32 consecutive output columns over the S partial rows with
// 8- or 16-byte loads (a partial row of D floats is one fully coalesced
// 256/512-byte read), divides by sum w_s and writes bf16 (round to nearest
// even) plus lse = M + ln sum w_s. The kernel is latency-bound (the partials
// are a few MB): partial rows are loaded in batches of sixteen, the first
// together with the LSE values and each next one while the previous batch is
// summed, and the CTAs are two warps so the rows spread over many SMs.
#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 2;  // small CTAs: the rows spread over more SMs

template <int V>
struct Vec;
template <>
struct Vec<4> {
    using T = float4;
    static __device__ __forceinline__ void fma(float* acc, float w, const T& x) {
        acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    }
};
template <>
struct Vec<2> {
    using T = float2;
    static __device__ __forceinline__ void fma(float* acc, float w, const T& x) {
        acc[0] += w * x.x; acc[1] += w * x.y;
    }
};

constexpr int kBatch = 16;  // partial rows in flight per lane

template <int D>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const MergeArgs a) {
    constexpr int V = D / 32;  // columns per lane
    using VT = typename Vec<V>::T;
    grid_dep_wait();  // the partials come from the preceding decode grid
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= static_cast<int64_t>(a.B) * a.Hq) return;
    const int b = static_cast<int>(row / a.Hq);
    const int h = static_cast<int>(row % a.Hq);
    const float* lse = a.lse_partial + b * a.lp_s0 + h;
    const float* op = a.out_partial + b * a.op_s0 + h * a.op_s2 + lane * V;
    const int S = a.S;

    // All loads of a batch are issued before any is used: the first batch of
    // up to 16 partial rows goes out together with the LSE values, and each
    // later batch is requested before the previous one is accumulated.
    float lv = (lane < S) ? __ldg(lse + lane * a.lp_s1) : -INFINITY;
    VT x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
        if (j < S) x[j] = __ldg(reinterpret_cast<const VT*>(op + j * a.op_s1));
    float m = lv;
    for (int s = 32 + lane; s < S; s += 32) m = fmaxf(m, __ldg(lse + s * a.lp_s1));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
        float w_mine = (lane < S) ? __expf(lv - m) : 0.f;
        wsum = w_mine;
        for (int s0 = 0; s0 < S; s0 += kBatch) {
            VT y[kBatch];
            const int s1 = s0 + kBatch;
            if (s1 < S) {  // next batch in flight while this one is summed
#pragma unroll
                for (int j = 0; j < kBatch; ++j)
                    if (s1 + j < S) y[j] = __ldg(reinterpret_cast<const VT*>(op + (s1 + j) * a.op_s1));
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int s = s0 + j;
                if ((s & 31) == 0 && s > 0) {  // weights of splits s .. s+31
                    w_mine = (s + lane < S) ? __expf(__ldg(lse + (s + lane) * a.lp_s1) - m) : 0.f;
                    wsum += w_mine;
                }
                const float w = __shfl_sync(0xffffffffu, w_mine, s & 31);
                if (s < S) Vec<V>::fma(acc, w, x[j]);
            }
            if (s1 < S) {
#pragma unroll
                for (int j = 0; j < kBatch; ++j) x[j] = y[j];
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        const float inv = 1.f / wsum;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] *= inv;
    }
    uint16_t* dst = a.out + b * a.o_s0 + h * a.o_s1 + lane * V;
    if constexpr (V == 4) {
        uint2 w;
        w.x = pack_bf16(acc[0], acc[1]);
        w.y = pack_bf16(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(dst) = w;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
    }
    if (a.lse_out && lane == 0)
        a.lse_out[b * a.lo_s0 + h * a.lo_s1] = (m == -INFINITY) ? -INFINITY : m + __logf(wsum);
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s) {
    const int64_t rows = static_cast<int64_t>(a.B) * a.Hq;
    if (rows == 0) return cudaSuccess;
    const int64_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kWarps * 32);
    if (a.D == 128) return launch_dependent(lse_merge_kernel<128>, grid, block, 0, s, a);
    if (a.D == 64) return launch_dependent(lse_merge_kernel<64>, grid, block, 0, s, a);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
