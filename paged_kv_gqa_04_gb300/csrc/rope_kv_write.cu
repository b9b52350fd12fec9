// rope_kv_write.cu -- fused RoPE + paged-KV cache write.
//
// Loom Kernels, "Supported operator paths" table, row "Position and KV":
// NeoX or interleaved RoPE of q and k, then k (rotated) and v written into
// NHD/HND page views as bf16 or static-scale FP8 E4M3 bytes, from packed or
// separate q/k/v. microLLM-rocm, optimisation checkpoints: split-half RoPE
// reading the projection layout and writing the attention layout directly.
//
// Mapping: every (token, row) -- a q head, a k head or a v head -- is handled
// by D/16 threads; thread c of a row owns the 8-element chunk starting at 8c
// and the chunk starting at D/2 + 8c. Under NeoX these two chunks are exactly
// the partners of one another's rotation pairs (i, i + D/2); under the
// interleaved style each chunk holds four whole pairs (2i, 2i+1). Every
// thread therefore reads and writes two 16-byte chunks of its row with
// 16-byte loads and stores, so a row is read and written in full 128-byte
// segments by D/16 consecutive lanes.
//
// Arithmetic: y1 = x1*c - x2*s and y2 = x2*c + x1*s with every product and
// the sum/difference rounded separately (__fmul_rn/__fsub_rn/__fadd_rn are
// never contracted into FMA), then bf16 round-to-nearest-even, or for FP8
// the correctly rounded quotient y / scale (__fdiv_rn) followed by the
// hardware's saturating round-to-nearest-even E4M3 conversion.
#include <cuda_fp8.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

struct Chunk8 {
    float v[8];
};

__device__ __forceinline__ Chunk8 unpack_bf16x8(uint4 w) {
    Chunk8 c;
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        c.v[2 * i] = bf16_lo(u[i]);
        c.v[2 * i + 1] = bf16_hi(u[i]);
    }
    return c;
}

__device__ __forceinline__ uint4 pack_bf16x8(const Chunk8& c) {
    uint4 w;
    w.x = pack_bf16(c.v[0], c.v[1]);
    w.y = pack_bf16(c.v[2], c.v[3]);
    w.z = pack_bf16(c.v[4], c.v[5]);
    w.w = pack_bf16(c.v[6], c.v[7]);
    return w;
}

__device__ __forceinline__ uint2 pack_e4m3x8(const Chunk8& c, float scale) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t b = 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float2 z = make_float2(__fdiv_rn(c.v[4 * h + 2 * i], scale), __fdiv_rn(c.v[4 * h + 2 * i + 1], scale));
            __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(z, __NV_SATFINITE, __NV_E4M3);
            b |= static_cast<uint32_t>(p) << (16 * i);
        }
        w[h] = b;
    }
    return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void rot(float x1, float x2, float c, float s, float& y1, float& y2) {
    y1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
    y2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
}

template <int D, bool INTER>
__device__ __forceinline__ void rotate_row(Chunk8& lo, Chunk8& hi, const float* cs, int c) {
    if constexpr (!INTER) {
        // pairs (8c + j, D/2 + 8c + j), frequency index 8c + j
        const float4 c0 = *reinterpret_cast<const float4*>(cs + 8 * c);
        const float4 c1 = *reinterpret_cast<const float4*>(cs + 8 * c + 4);
        const float4 s0 = *reinterpret_cast<const float4*>(cs + D / 2 + 8 * c);
        const float4 s1 = *reinterpret_cast<const float4*>(cs + D / 2 + 8 * c + 4);
        const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float y1, y2;
            rot(lo.v[j], hi.v[j], cv[j], sv[j], y1, y2);
            lo.v[j] = y1;
            hi.v[j] = y2;
        }
    } else {
        // chunk 8c holds pairs of frequency 4c..4c+3; chunk D/2 + 8c holds
        // pairs of frequency D/4 + 4c .. D/4 + 4c + 3
        const float4 cl = *reinterpret_cast<const float4*>(cs + 4 * c);
        const float4 sl = *reinterpret_cast<const float4*>(cs + D / 2 + 4 * c);
        const float4 ch = *reinterpret_cast<const float4*>(cs + D / 4 + 4 * c);
        const float4 sh = *reinterpret_cast<const float4*>(cs + D / 2 + D / 4 + 4 * c);
        const float clv[4] = {cl.x, cl.y, cl.z, cl.w}, slv[4] = {sl.x, sl.y, sl.z, sl.w};
        const float chv[4] = {ch.x, ch.y, ch.z, ch.w}, shv[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float y1, y2;
            rot(lo.v[2 * m], lo.v[2 * m + 1], clv[m], slv[m], y1, y2);
            lo.v[2 * m] = y1;
            lo.v[2 * m + 1] = y2;
            rot(hi.v[2 * m], hi.v[2 * m + 1], chv[m], shv[m], y1, y2);
            hi.v[2 * m] = y1;
            hi.v[2 * m + 1] = y2;
        }
    }
}

template <int D, bool INTER, bool FP8>
__global__ void __launch_bounds__(256) rope_kv_write_kernel(const RopeArgs a, const int64_t total) {
    constexpr int TPR = D / 16;  // threads per row
    // The decode kernel that usually follows may start its prologue now; it
    // waits for this grid's writes before it reads q or the cache.
    grid_dep_launch();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int rows = a.Hq + 2 * a.Hkv;
    const int64_t per_tok = static_cast<int64_t>(rows) * TPR;
    const int64_t t = idx / per_tok;
    const int r = static_cast<int>(idx - t * per_tok);
    const int row = r / TPR;
    const int c = r % TPR;

    // slot, position and the row's two chunks do not depend on one another:
    // all four loads are issued before any of them is checked (reading the
    // row of a skipped token stays inside the [T, heads, D] input).
    const bool is_q = row < a.Hq;
    const bool is_k = !is_q && row < a.Hq + a.Hkv;
    const int h = is_q ? row : (is_k ? row - a.Hq : row - a.Hq - a.Hkv);
    const uint16_t* src = is_q ? a.q + t * a.q_s0 + h * a.q_s1
                               : (is_k ? a.k + t * a.k_s0 + h * a.k_s1 : a.v + t * a.v_s0 + h * a.v_s1);
    const int32_t slot = __ldg(a.slots + t);
    const int32_t pos = __ldg(a.positions + t);
    const uint4 wlo = *reinterpret_cast<const uint4*>(src + 8 * c);
    const uint4 whi = *reinterpret_cast<const uint4*>(src + D / 2 + 8 * c);
    if (slot < 0) return;
    const int64_t num_slots = a.num_pages * a.page_size;
    if (slot >= num_slots) {
        if (r == 0) flag_error(a.err, PKV_FLAG_SLOT_RANGE);
        return;
    }
    if (pos < 0 || pos >= a.max_pos) {
        if (r == 0) flag_error(a.err, PKV_FLAG_POSITION_RANGE);
        return;
    }
    const float* cs = a.cos_sin + pos * a.cs_s0;
    Chunk8 lo = unpack_bf16x8(wlo);
    Chunk8 hi = unpack_bf16x8(whi);

    if (is_q) {  // q head: rotate in place
        rotate_row<D, INTER>(lo, hi, cs, c);
        uint16_t* p = a.q + t * a.q_s0 + h * a.q_s1;
        *reinterpret_cast<uint4*>(p + 8 * c) = pack_bf16x8(lo);
        *reinterpret_cast<uint4*>(p + D / 2 + 8 * c) = pack_bf16x8(hi);
        return;
    }
    if (is_k) rotate_row<D, INTER>(lo, hi, cs, c);

    const int64_t page = slot / a.page_size;
    const int off = static_cast<int>(slot - page * a.page_size);
    const int64_t* st = is_k ? a.kc_s : a.vc_s;
    const int64_t e = (a.layout == PKV_HND) ? page * st[0] + h * st[1] + off * st[2]
                                            : page * st[0] + off * st[1] + h * st[2];
    if constexpr (FP8) {
        const float* sp = is_k ? a.k_scale : a.v_scale;
        const float scale = __ldg(sp + (a.n_scale == 1 ? 0 : h));
        uint8_t* dst = static_cast<uint8_t*>(is_k ? a.k_cache : a.v_cache) + e;
        *reinterpret_cast<uint2*>(dst + 8 * c) = pack_e4m3x8(lo, scale);
        *reinterpret_cast<uint2*>(dst + D / 2 + 8 * c) = pack_e4m3x8(hi, scale);
    } else {
        uint16_t* dst = static_cast<uint16_t*>(is_k ? a.k_cache : a.v_cache) + e;
        *reinterpret_cast<uint4*>(dst + 8 * c) = pack_bf16x8(lo);
        *reinterpret_cast<uint4*>(dst + D / 2 + 8 * c) = pack_bf16x8(hi);
    }
}

template <int D, bool INTER, bool FP8>
cudaError_t launch_t(const RopeArgs& a, cudaStream_t s) {
    const int64_t total = a.T * static_cast<int64_t>(a.Hq + 2 * a.Hkv) * (D / 16);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    rope_kv_write_kernel<D, INTER, FP8><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a, total);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const RopeArgs& a, cudaStream_t s) {
    if (a.interleaved) return a.fp8 ? launch_t<D, true, true>(a, s) : launch_t<D, true, false>(a, s);
    return a.fp8 ? launch_t<D, false, true>(a, s) : launch_t<D, false, false>(a, s);
}

}  // namespace

cudaError_t launch_rope_kv_write(const RopeArgs& a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_d<64>(a, s);
        case 128: return launch_d<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
