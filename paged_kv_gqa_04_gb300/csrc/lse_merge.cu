// lse_merge.cu -- log-sum-exp merge of split-K decode partials.
//
// mainarch, decode-attention section: the split-KV partials are combined by
// their log-sum-exp weights; Loom Kernels, "Attention" row: local
// split-K/LSE merge.
//
// A warp merges a run of splits of one (sequence, query head) row: it reads
// their LSE values, forms their max M and the weights w_s = exp(lse_s - M),
// and each lane accumulates D/32 consecutive output columns over the partial
// rows with 8- or 16-byte loads (a partial row of D floats is one coalesced
// 256/512-byte read). With up to 32 splits one warp does the whole row and
// writes bf16 (round to nearest even) out = sum w_s o_s / sum w_s and
// lse = M + ln sum w_s. With more, the row is a two-level tree (mainarch,
// decode-attention section: a parallel tree combine rather than one
// workgroup grinding through the partials): the 32 warps of one CTA each
// merge a contiguous run of splits of a 64-column slice in parallel and
// their results are merged again by their own LSE weights. The kernel is
// latency-bound (the partials are a few MB): partial rows are loaded in
// batches (4 or 16 for one warp per row, by the call's record count;
// eight in the tree: one batch per warp up to 256 splits), the first
// together with the LSE values and each next one while the previous batch
// is summed. Rows wider than 128 columns
// (the 512-value latent output of MLA decode) are cut into slices (128
// columns for one warp per row, 64 in the tree), each merged with the same
// LSE weights.
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

// One warp's share of a row: splits [s_lo, s_hi). Returns the warp's LSE
// maximum m (-inf when every split in the range is empty), the weight sum
// l = sum_s exp(lse_s - m) (warp-reduced, every lane holds it) and, per
// lane, acc = sum_s exp(lse_s - m) * out_partial_s over the lane's V columns.
// All loads of a batch of 16 partial rows are issued before any is used: the
// first batch goes out with the first 32 LSE values, each later batch while
// the previous one is summed. (16 rows per batch for a warp that merges a
// whole row, 8 in the tree kernel, whose 32 warps share the register file.)
template <int V, int kBatch, bool kSingle = false>
__device__ __forceinline__ void warp_merge(const float* lse, int64_t lp_s1, const float* op, int64_t op_s1, int s_lo,
                                           int s_hi, float& m, float& l, float (&acc)[V]) {
    if constexpr (kSingle) {
        // At most kBatch splits (the caller guarantees it; used for up to 4):
        // every lane reads the same few LSE values (one broadcast
        // transaction each) and forms the weights itself, no cross-lane
        // step; one batch of partial rows.
        using VT = typename Vec<V>::T;
        const int n = s_hi - s_lo;
        lse += s_lo * lp_s1;
        op += s_lo * op_s1;
        float lj[kBatch];
        VT x[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            lj[j] = (j < n) ? __ldg(lse + j * lp_s1) : -INFINITY;
            if (j < n) x[j] = __ldg(reinterpret_cast<const VT*>(op + j * op_s1));
        }
        m = lj[0];
#pragma unroll
        for (int j = 1; j < kBatch; ++j) m = fmaxf(m, lj[j]);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        l = 0.f;
        if (m == -INFINITY) return;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < n) {
                const float w = __expf(lj[j] - m);
                l += w;
                Vec<V>::fma(acc, w, x[j]);
            }
        }
        return;
    }
    using VT = typename Vec<V>::T;
    const int lane = threadIdx.x & 31;
    const int n = s_hi - s_lo;
    lse += s_lo * lp_s1;
    op += s_lo * op_s1;
    float lv = (lane < n) ? __ldg(lse + lane * lp_s1) : -INFINITY;
    VT x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
        if (j < n) x[j] = __ldg(reinterpret_cast<const VT*>(op + j * op_s1));
    m = lv;
    for (int s = 32 + lane; s < n; s += 32) m = fmaxf(m, __ldg(lse + s * lp_s1));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    l = 0.f;
    if (m == -INFINITY) return;
    float w_mine = (lane < n) ? __expf(lv - m) : 0.f;
    float wsum = w_mine;
    for (int s0 = 0; s0 < n; s0 += kBatch) {
        VT y[kBatch];
        const int s1 = s0 + kBatch;
        if (s1 < n) {  // next batch in flight while this one is summed
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (s1 + j < n) y[j] = __ldg(reinterpret_cast<const VT*>(op + (s1 + j) * op_s1));
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int s = s0 + j;
            if ((s & 31) == 0 && s > 0) {  // weights of splits s .. s+31
                w_mine = (s + lane < n) ? __expf(__ldg(lse + (s + lane) * lp_s1) - m) : 0.f;
                wsum += w_mine;
            }
            const float w = __shfl_sync(0xffffffffu, w_mine, s & 31);
            if (s < n) Vec<V>::fma(acc, w, x[j]);
        }
        if (s1 < n) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) x[j] = y[j];
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    l = wsum;
}

template <int V>
__device__ __forceinline__ void store_row(uint16_t* dst, const float (&o)[V]) {
    if constexpr (V == 4) {
        uint2 w;
        w.x = pack_bf16(o[0], o[1]);
        w.y = pack_bf16(o[2], o[3]);
        *reinterpret_cast<uint2*>(dst) = w;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16(o[0], o[1]);
    }
}

// The records merged for sequence b: its own split count under a split plan
// (clamped to [1, S]; out-of-range counts were flagged by the decode), else
// all S.
__device__ __forceinline__ int records_of(const MergeArgs& a, int b) {
    if (a.splits_per_seq == nullptr) return a.S;
    return min(max(__ldg(a.splits_per_seq + b), 1), a.S);
}

// Columns of a row one warp merges, and the slices a row is cut into.
template <int D>
struct Slice {
    static constexpr int DW = D > 128 ? 128 : D;
    static constexpr int N = D / DW;
    static constexpr int V = DW / 32;  // columns per lane
};

// Few splits (S <= 32): one warp per row slice, two slices per CTA.
template <int D, int kBatch, bool kSingle>
__global__ void __launch_bounds__(kWarps * 32) lse_merge_kernel(const MergeArgs a) {
    using SL = Slice<D>;
    constexpr int V = SL::V;
    const int lane = threadIdx.x & 31;
    const int64_t vrow = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (vrow >= static_cast<int64_t>(a.B) * a.Hq * SL::N) {
        grid_dep_wait();
        return;
    }
    const int64_t row = vrow / SL::N;
    const int c0 = static_cast<int>(vrow % SL::N) * SL::DW + lane * V;
    const int b = static_cast<int>(row / a.Hq);
    const int h = static_cast<int>(row % a.Hq);
    // The record count is an index input of the step (never written by the
    // decode): read it while the decode may still run; the partials come
    // from that decode grid, so they are read only after the wait.
    const int S = records_of(a, b);
    grid_dep_wait();
    float m, l, acc[V];
    warp_merge<V, kBatch, kSingle>(a.lse_partial + b * a.lp_s0 + h, a.lp_s1,
                                   a.out_partial + b * a.op_s0 + h * a.op_s2 + c0, a.op_s1, 0, S, m, l, acc);
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] *= inv;
    store_row<V>(a.out + b * a.o_s0 + h * a.o_s1 + c0, acc);
    if (a.lse_out && c0 == 0)
        a.lse_out[b * a.lo_s0 + h * a.lo_s1] = (m == -INFINITY) ? -INFINITY : m + __logf(l);
}

// Many splits: a two-level tree. One CTA per 64-column slice of a row; each
// of its 32 warps merges a contiguous run of at most ceil(S / 32) splits
// (one batch of loads up to S = 256), then the warp results are combined
// through shared memory by their own LSE weights, each computed once.
constexpr int kTreeWarps = 32;
constexpr int kTreeCols = 64;

template <int D>
__global__ void __launch_bounds__(kTreeWarps * 32) lse_merge_tree_kernel(const MergeArgs a) {
    constexpr int DW = kTreeCols;
    constexpr int NS = D / DW;  // slices per row
    constexpr int V = DW / 32;  // columns per lane
    constexpr int W = kTreeWarps;
    // W * DW partial sums, then W maxima, W weight sums, W weights
    extern __shared__ float tree_smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t row = blockIdx.x / NS;
    const int c0 = static_cast<int>(blockIdx.x % NS) * DW;  // first column of this CTA's slice
    const int b = static_cast<int>(row / a.Hq);
    const int h = static_cast<int>(row % a.Hq);
    const int S = records_of(a, b);  // an index input: read before the wait, as above
    grid_dep_wait();
    const int chunk = (S + W - 1) / W;
    const int s_lo = min(S, warp * chunk), s_hi = min(S, s_lo + chunk);
    float m, l, acc[V];
    warp_merge<V, 8>(a.lse_partial + b * a.lp_s0 + h, a.lp_s1,
                     a.out_partial + b * a.op_s0 + h * a.op_s2 + c0 + lane * V, a.op_s1, s_lo, s_hi, m, l, acc);
    float* sacc = tree_smem;
    float* sm = tree_smem + W * DW;
    float* sl = sm + W;
    float* sw = sl + W;
#pragma unroll
    for (int i = 0; i < V; ++i) sacc[warp * DW + lane * V + i] = acc[i];
    if (lane == 0) {
        sm[warp] = m;
        sl[warp] = l;
    }
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < W; ++w) M = fmaxf(M, sm[w]);
    if (threadIdx.x < W) sw[threadIdx.x] = (sm[threadIdx.x] == -INFINITY) ? 0.f : __expf(sm[threadIdx.x] - M);
    __syncthreads();
    float L = 0.f;
    for (int w = 0; w < W; ++w) L += sw[w] * sl[w];
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    for (int d2 = threadIdx.x; d2 < DW / 2; d2 += blockDim.x) {
        float o0 = 0.f, o1 = 0.f;
        for (int w = 0; w < W; ++w) {  // an empty run's weight is 0 and its sums are 0
            o0 += sw[w] * sacc[w * DW + 2 * d2];
            o1 += sw[w] * sacc[w * DW + 2 * d2 + 1];
        }
        *reinterpret_cast<uint32_t*>(a.out + b * a.o_s0 + h * a.o_s1 + c0 + 2 * d2) = pack_bf16(o0 * inv, o1 * inv);
    }
    if (a.lse_out && c0 == 0 && threadIdx.x == 0)
        a.lse_out[b * a.lo_s0 + h * a.lo_s1] = (M == -INFINITY) ? -INFINITY : M + __logf(L);
}

// One warp per row slice. Up to four records, a batch of four rows read
// with the LSE values by every lane (44 registers: the 8,192 rows of up to 4
// records of the ragged workload fit one wave of warps; with the 16-row
// batch, 164 registers per thread, they ran in about five waves, 11.0 us
// per launch in ncu, caches cold). More records: the 16-row batch with the
// weights shared by shuffles (measured faster there: one LSE load per lane
// instead of one broadcast load per record).
template <int D, int kBatch, bool kSingle>
cudaError_t launch_rows(const MergeArgs& a, int64_t rows, cudaStream_t s) {
    const int64_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    return launch_dependent(lse_merge_kernel<D, kBatch, kSingle>, dim3(static_cast<unsigned>(blocks)),
                            dim3(kWarps * 32), 0, s, a);
}

template <int D>
cudaError_t launch_d(const MergeArgs& a, cudaStream_t s) {
    using SL = Slice<D>;
    const int64_t rows = static_cast<int64_t>(a.B) * a.Hq * SL::N;  // row slices
    if (a.S <= 32) {
        if (a.S <= 4) return launch_rows<D, 4, true>(a, rows, s);
        return launch_rows<D, 16, false>(a, rows, s);
    }
    const int64_t trows = static_cast<int64_t>(a.B) * a.Hq * (D / kTreeCols);  // 64-column row slices
    if (trows > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const size_t smem = static_cast<size_t>(kTreeWarps) * (kTreeCols + 3) * sizeof(float);
    return launch_dependent(lse_merge_tree_kernel<D>, dim3(static_cast<unsigned>(trows)), dim3(kTreeWarps * 32), smem,
                            s, a);
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s) {
    if (static_cast<int64_t>(a.B) * a.Hq == 0) return cudaSuccess;
    switch (a.D) {
        case 64: return launch_d<64>(a, s);
        case 128: return launch_d<128>(a, s);
        case 512: return launch_d<512>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
