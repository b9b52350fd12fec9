// rope_kv_write.cu -- fused RoPE + paged-KV cache write.
//
// Loom Kernels, "Supported operator paths" table, row "Position and KV":
// NeoX or interleaved RoPE of q and k, then k (rotated) and v written into
// NHD/HND page views as bf16 or static-scale FP8 E4M3 bytes, from packed or
// separate q/k/v. microLLM-rocm, optimisation checkpoints: split-half RoPE
// reading the projection layout and writing the attention layout directly.
//
// Mapping: a CTA takes `toks` tokens at a time (U groups of them per thread).
// Its threads are ordered by the kind of row first -- the q heads of all its
// tokens, then their k heads, then their v heads -- and within a kind by
// token, head and chunk, so a warp holds one kind of row only (the rotation
// and the cos/sin loads of k rows are not spread over warps that also hold
// v rows). Every (token, row) -- a q head, a k head or a v head -- is
// handled by D/16 threads; thread c of a row owns the 8-element chunk starting at 8c
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
// the E4M3 byte of the correctly rounded quotient y / scale (from a
// reciprocal product when that provably gives the same byte, else from the
// IEEE division), with the hardware's saturating round-to-nearest-even
// E4M3 conversion.
//
// NVFP4 caches (mainarch, decode-attention section: 4-bit E2M1 KV with block
// scales; NVFP4 form): a 16-value block of a row is the two 8-value chunks of
// a lane pair (chunk c and c^1 are adjacent lanes), so the block's largest
// magnitude takes one shuffle. Its E4M3 scale is the saturating RNE byte of
// amax / (6 g), g the head's static scale; each value is the E2M1 code of the
// correctly rounded quotient y / (g s), again from a reciprocal product unless
// a value lies near an E2M1 rounding boundary. The lane with the even chunk
// stores the scale of the low-half block, the odd lane that of the high half.
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

// Packed float32 product (sm_100+ f32x2 arithmetic): each lane is rounded
// exactly as the scalar product would be, in one issue slot for two values.
// Where a sum follows (the rotation), the sum is a scalar operation with
// explicit rounding, which is never contracted with the product.
__device__ __forceinline__ void mul_rn_x2(float a0, float a1, float b0, float b1, float& d0, float& d1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// Four E4M3 bytes (a -> byte 0 .. d -> byte 3), saturating round-to-nearest-even.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 l, h;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
        "mov.b32 %0, {l, h};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// Per-scale constants of the FP8 quantiser: the reciprocal of the scale
// nudged down and up by 2^-20 (relative), each rounded to float32.
struct E4m3Rcp {
    float lo, hi;
    bool exact_only;  // a scale whose reciprocal could leave float32's normal range
};
__device__ __forceinline__ E4m3Rcp e4m3_rcp(float scale) {
    E4m3Rcp r;
    r.exact_only = !(scale >= 0x1p-100f && scale <= 0x1p100f);
    const float rcp = __frcp_rn(scale);
    r.lo = __fmul_rn(rcp, 1.0f - 0x1p-20f);
    r.hi = __fmul_rn(rcp, 1.0f + 0x1p-20f);
    return r;
}

// E4M3 bytes (low byte first) of the correctly rounded float32 quotients
// Q = RN(y / scale), saturating, for the 8 values of a chunk, without a
// division in the common case. With r = RN(1/scale), r_lo = RN(r (1 - 2^-20))
// and r_hi = RN(r (1 + 2^-20)), the products z_lo = RN(y r_lo) and
// z_hi = RN(y r_hi) differ from y / scale by factors within
// (1 - 2^-20)(1 +- 2^-24)^3 and (1 + 2^-20)(1 +- 2^-24)^3, while Q differs from
// it by a factor within 1 +- 2^-24; so Q lies between z_lo and z_hi (values
// so small that float32 rounds them absolutely are far below E4M3's smallest
// step, where every one of the three gives the zero byte of the right
// sign). E4M3 rounding is monotone, so when z_lo and z_hi give the same byte,
// Q gives it too. When they differ -- Q is within about 2^-19 (relative) of
// an E4M3 rounding boundary, about one value in 2^15 -- the chunk is
// quantised from the IEEE divisions.
__device__ __forceinline__ uint2 pack_e4m3x8(const Chunk8& c, float scale, const E4m3Rcp& r) {
    float zl[8], zh[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        mul_rn_x2(c.v[j], c.v[j + 1], r.lo, r.lo, zl[j], zl[j + 1]);
        mul_rn_x2(c.v[j], c.v[j + 1], r.hi, r.hi, zh[j], zh[j + 1]);
    }
    uint32_t w0 = e4m3x4(zl[0], zl[1], zl[2], zl[3]);
    uint32_t w1 = e4m3x4(zl[4], zl[5], zl[6], zl[7]);
    const uint32_t h0 = e4m3x4(zh[0], zh[1], zh[2], zh[3]);
    const uint32_t h1 = e4m3x4(zh[4], zh[5], zh[6], zh[7]);
    if ((w0 != h0) | (w1 != h1) | r.exact_only) {
        float z[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) z[j] = __fdiv_rn(c.v[j], scale);
        w0 = e4m3x4(z[0], z[1], z[2], z[3]);
        w1 = e4m3x4(z[4], z[5], z[6], z[7]);
    }
    return make_uint2(w0, w1);
}

__device__ __forceinline__ float amax8(const Chunk8& c) {
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(c.v[j]));
    return m;
}

// Bracketing reciprocals of a divisor d: RN(RN(1/d) (1 -+ 2^-20)). For any y,
// RN(y * lo) and RN(y * hi) enclose the correctly rounded quotient RN(y / d)
// (the argument of pack_e4m3x8), so a monotone rounding that gives both the
// same code gives the quotient that code too. Divisors whose reciprocal could
// leave float32's normal range are marked for the division path.
__device__ __forceinline__ E4m3Rcp bracket_rcp(float d) { return e4m3_rcp(d); }

// The same brackets from the hardware's approximate reciprocal r ~ 1/d
// (rcp.approx.f32, documented within one unit in the last place; measured on
// GB300 over every float32 in [2^-30, 2^30): relative error at most
// 2^-23.27). With
// |r d - 1| < 2^-22 the products RN(y RN(r (1 -+ 2^-20))) still differ from
// y / d by factors within (1 -+ 2^-20)(1 +- 2^-22)(1 +- 2^-24)^2, i.e.
// strictly beyond the 1 +- 2^-24 of RN(y / d) on each side, so they still
// enclose it. Used for the per-block divisors of the NVFP4 quantiser.
__device__ __forceinline__ E4m3Rcp bracket_rcp_approx(float d) {
    E4m3Rcp r;
    r.exact_only = !(d >= 0x1p-100f && d <= 0x1p100f);
    float rcp;
    asm("rcp.approx.f32 %0, %1;" : "=f"(rcp) : "f"(d));
    r.lo = __fmul_rn(rcp, 1.0f - 0x1p-20f);
    r.hi = __fmul_rn(rcp, 1.0f + 0x1p-20f);
    return r;
}

// One 8-value half of an NVFP4 block whose largest magnitude is `amax`,
// under the static scale g (six_g = RN(6 g), r6 = bracket_rcp(six_g)):
// returns the four bytes of E2M1 pairs and the block's E4M3 scale byte,
// which are those of the correctly rounded quotients amax / six_g and
// y / RN(g s). Each is taken from the bracketing products when both
// products give the same code, else (rarely) from the IEEE divisions.
__device__ __forceinline__ uint32_t nvfp4_half(const Chunk8& c, float amax, float g, float six_g,
                                               const E4m3Rcp& r6, uint32_t& sbyte) {
    uint32_t sb;
    {
        uint16_t bl, bh;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(bl) : "f"(__fmul_rn(amax, r6.hi)), "f"(__fmul_rn(amax, r6.lo)));
        bh = static_cast<uint16_t>(bl >> 8);
        bl = static_cast<uint16_t>(bl & 0xFF);
        sb = bl;
        if (bl != bh || r6.exact_only)
            sb = __nv_cvt_float_to_fp8(__fdiv_rn(amax, six_g), __NV_SATFINITE, __NV_E4M3);
    }
    sbyte = sb;
    const float s = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(sb), __NV_E4M3)));
    if (s == 0.f) return 0u;
    const float denom = __fmul_rn(g, s);
    const E4m3Rcp r = bracket_rcp_approx(denom);
    float zl[8], zh[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
        mul_rn_x2(c.v[j], c.v[j + 1], r.lo, r.lo, zl[j], zl[j + 1]);
        mul_rn_x2(c.v[j], c.v[j + 1], r.hi, r.hi, zh[j], zh[j + 1]);
    }
    const uint32_t wl = pack_e2m1x8(zl);
    if (wl == pack_e2m1x8(zh) && !r.exact_only) return wl;
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = __fdiv_rn(c.v[j], denom);
    return pack_e2m1x8(z);
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm("mov.u32 %0, %%laneid;" : "=r"(l));
    return l;
}

// The cos and sin a thread needs for its two chunks, loaded as four 16-byte
// vectors. NeoX: chunk 8c pairs with chunk D/2 + 8c at frequencies 8c..8c+7.
// Interleaved: chunk 8c holds the pairs of frequencies 4c..4c+3, chunk
// D/2 + 8c those of D/4 + 4c .. D/4 + 4c + 3.
template <int D, bool INTER>
__device__ __forceinline__ void load_cos_sin(const float* cs, int c, float (&cv)[8], float (&sv)[8]) {
    float4 a0, a1, b0, b1;
    if constexpr (!INTER) {
        a0 = *reinterpret_cast<const float4*>(cs + 8 * c);
        a1 = *reinterpret_cast<const float4*>(cs + 8 * c + 4);
        b0 = *reinterpret_cast<const float4*>(cs + D / 2 + 8 * c);
        b1 = *reinterpret_cast<const float4*>(cs + D / 2 + 8 * c + 4);
    } else {
        a0 = *reinterpret_cast<const float4*>(cs + 4 * c);
        a1 = *reinterpret_cast<const float4*>(cs + D / 4 + 4 * c);
        b0 = *reinterpret_cast<const float4*>(cs + D / 2 + 4 * c);
        b1 = *reinterpret_cast<const float4*>(cs + D / 2 + D / 4 + 4 * c);
    }
    cv[0] = a0.x; cv[1] = a0.y; cv[2] = a0.z; cv[3] = a0.w;
    cv[4] = a1.x; cv[5] = a1.y; cv[6] = a1.z; cv[7] = a1.w;
    sv[0] = b0.x; sv[1] = b0.y; sv[2] = b0.z; sv[3] = b0.w;
    sv[4] = b1.x; sv[5] = b1.y; sv[6] = b1.z; sv[7] = b1.w;
}

// y1 = x1 c - x2 s, y2 = x2 c + x1 s for every pair of the row's two chunks,
// each product and the sum / difference rounded on its own, never fused:
// the products are packed f32x2 multiplies (two per instruction, explicit
// round-to-nearest), the sums and differences scalar operations with
// explicit rounding. (A packed sum reading a packed product may be
// contracted into a fused multiply-add by the compiler, which changes the
// rounding; the scalar forms are not.)
template <bool INTER>
__device__ __forceinline__ void rotate_row(Chunk8& lo, Chunk8& hi, const float (&cv)[8], const float (&sv)[8]) {
    if constexpr (!INTER) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            float lc0, lc1, hs0, hs1, hc0, hc1, ls0, ls1;
            mul_rn_x2(lo.v[j], lo.v[j + 1], cv[j], cv[j + 1], lc0, lc1);
            mul_rn_x2(hi.v[j], hi.v[j + 1], sv[j], sv[j + 1], hs0, hs1);
            mul_rn_x2(hi.v[j], hi.v[j + 1], cv[j], cv[j + 1], hc0, hc1);
            mul_rn_x2(lo.v[j], lo.v[j + 1], sv[j], sv[j + 1], ls0, ls1);
            lo.v[j] = __fsub_rn(lc0, hs0);
            lo.v[j + 1] = __fsub_rn(lc1, hs1);
            hi.v[j] = __fadd_rn(hc0, ls0);
            hi.v[j + 1] = __fadd_rn(hc1, ls1);
        }
    } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float p0, p1, q0, q1;
            // lo pair (2m, 2m + 1) at frequency m
            mul_rn_x2(lo.v[2 * m], lo.v[2 * m + 1], cv[m], cv[m], p0, p1);
            mul_rn_x2(lo.v[2 * m + 1], lo.v[2 * m], sv[m], sv[m], q0, q1);
            lo.v[2 * m] = __fsub_rn(p0, q0);
            lo.v[2 * m + 1] = __fadd_rn(p1, q1);
            // hi pair at frequency 4 + m
            mul_rn_x2(hi.v[2 * m], hi.v[2 * m + 1], cv[4 + m], cv[4 + m], p0, p1);
            mul_rn_x2(hi.v[2 * m + 1], hi.v[2 * m], sv[4 + m], sv[4 + m], q0, q1);
            hi.v[2 * m] = __fsub_rn(p0, q0);
            hi.v[2 * m + 1] = __fadd_rn(p1, q1);
        }
    }
}

// U tokens per thread: all of their loads (slot, position, the row's two
// chunks, then the cos/sin rows) are issued before any token is processed,
// so a thread keeps U times as many bytes in flight.
#ifndef PKV_WRITE_FILL_MIN_CTAS
#define PKV_WRITE_FILL_MIN_CTAS 4  // resident CTAs per SM the multi-token form is register-budgeted for
#endif
template <int D, bool INTER, int KIND, int U>
__global__ void __launch_bounds__(U == 1 ? 1024 : 256, U == 1 ? 1 : (U == 2 ? PKV_WRITE_FILL_MIN_CTAS : 2))
    rope_kv_write_kernel(const RopeArgs a) {
    constexpr int TPR = D / 16;  // threads per row
    // Launched as a programmatic dependent: the inputs may come from the
    // preceding grid (a copy of the step's inputs), and a preceding decode
    // may still read the cache.
    grid_dep_wait();
    // The decode kernel that usually follows may start its prologue now; it
    // waits for this grid's writes before it reads q or the cache.
    grid_dep_launch();
    // threadIdx.x: [0, nq) the q rows of the CTA's `toks` tokens, then
    // [nq, nq + nk) their k rows, then their v rows; within a kind, token
    // tl, head h and chunk c (TPR threads per row, so a row's threads are
    // consecutive lanes of one warp). u and blockIdx.x: groups of tokens.
    const int toks = a.toks;
    const int L = threadIdx.x;
    const int nq = toks * a.Hq * TPR, nk = toks * a.Hkv * TPR;
    const bool is_q = L < nq;
    const bool is_k = !is_q && L < nq + nk;
    const int j = is_q ? L : (is_k ? L - nq : L - nq - nk);
    const int per = (is_q ? a.Hq : a.Hkv) * TPR;  // threads of one token's rows of this kind
    const int tl = j / per;
    const int h = (j - tl * per) / TPR;
    const int c = j % TPR;
    const bool lead = h == 0 && c == 0;  // flags a bad token once per kind
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * toks * U + tl;
    const int64_t num_slots = a.num_pages * a.page_size;

    // Reading the row of a skipped token stays inside the [T, heads, D] input.
    int32_t slot[U], pos[U];
    uint4 wlo[U], whi[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + static_cast<int64_t>(u) * toks;
        live[u] = t < a.T;
        if (!live[u]) continue;
        const uint16_t* src = is_q ? a.q + t * a.q_s0 + h * a.q_s1
                                   : (is_k ? a.k + t * a.k_s0 + h * a.k_s1 : a.v + t * a.v_s0 + h * a.v_s1);
        slot[u] = __ldg(a.slots + t);
        pos[u] = __ldg(a.positions + t);
        wlo[u] = *reinterpret_cast<const uint4*>(src + 8 * c);
        whi[u] = *reinterpret_cast<const uint4*>(src + D / 2 + 8 * c);
    }
    float cv[U][8], sv[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!live[u] || slot[u] < 0) {
            live[u] = false;
            continue;
        }
        if (slot[u] >= num_slots) {
            if (lead) flag_error(a.err, PKV_FLAG_SLOT_RANGE);
            live[u] = false;
            continue;
        }
        if (pos[u] < 0 || pos[u] >= a.max_pos) {
            if (lead) flag_error(a.err, PKV_FLAG_POSITION_RANGE);
            live[u] = false;
            continue;
        }
        if (is_q || is_k) load_cos_sin<D, INTER>(a.cos_sin + pos[u] * a.cs_s0, c, cv[u], sv[u]);
    }

    float scale = 1.f, six_g = 1.f;
    E4m3Rcp r8{1.f, 1.f, false};  // FP8: brackets of 1/scale; NVFP4: of 1/RN(6 g)
    if constexpr (KIND != kBf16) {
        if (!is_q) {
            scale = __ldg((is_k ? a.k_scale : a.v_scale) + (a.n_scale == 1 ? 0 : h));
            if constexpr (KIND == kFp8) {
                r8 = e4m3_rcp(scale);
            } else {
                six_g = __fmul_rn(6.f, scale);
                r8 = bracket_rcp(six_g);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!live[u]) continue;
        const int64_t t = t0 + static_cast<int64_t>(u) * toks;
        Chunk8 lo = unpack_bf16x8(wlo[u]);
        Chunk8 hi = unpack_bf16x8(whi[u]);
        if (is_q) {  // q head: rotate in place
            rotate_row<INTER>(lo, hi, cv[u], sv[u]);
            uint16_t* p = a.q + t * a.q_s0 + h * a.q_s1;
            *reinterpret_cast<uint4*>(p + 8 * c) = pack_bf16x8(lo);
            *reinterpret_cast<uint4*>(p + D / 2 + 8 * c) = pack_bf16x8(hi);
            continue;
        }
        if (is_k) rotate_row<INTER>(lo, hi, cv[u], sv[u]);
        int64_t page;
        int off;
        if (a.page_size == 16) {  // the decode kernel's page size: no division
            page = slot[u] >> 4;
            off = slot[u] & 15;
        } else {
            page = slot[u] / a.page_size;
            off = static_cast<int>(slot[u] - page * a.page_size);
        }
        const int64_t* st = is_k ? a.kc_s : a.vc_s;
        const int64_t e = (a.layout == PKV_HND) ? page * st[0] + h * st[1] + off * st[2]
                                                : page * st[0] + off * st[1] + h * st[2];
        if constexpr (KIND == kFp8) {
            uint8_t* dst = static_cast<uint8_t*>(is_k ? a.k_cache : a.v_cache) + e;
            *reinterpret_cast<uint2*>(dst + 8 * c) = pack_e4m3x8(lo, scale, r8);
            *reinterpret_cast<uint2*>(dst + D / 2 + 8 * c) = pack_e4m3x8(hi, scale, r8);
        } else if constexpr (KIND == kFp4) {
            // both lanes of the pair (chunks c, c^1 of this row) are here
            const unsigned pair = 3u << (lane_id() & 30u);
            float am_lo = amax8(lo), am_hi = amax8(hi);
            am_lo = fmaxf(am_lo, __shfl_xor_sync(pair, am_lo, 1));
            am_hi = fmaxf(am_hi, __shfl_xor_sync(pair, am_hi, 1));
            uint32_t s_lo, s_hi;
            const uint32_t w_lo = nvfp4_half(lo, am_lo, scale, six_g, r8, s_lo);
            const uint32_t w_hi = nvfp4_half(hi, am_hi, scale, six_g, r8, s_hi);
            uint8_t* dst = static_cast<uint8_t*>(is_k ? a.k_cache : a.v_cache) + e;
            *reinterpret_cast<uint32_t*>(dst + 4 * c) = w_lo;
            *reinterpret_cast<uint32_t*>(dst + D / 4 + 4 * c) = w_hi;
            const int64_t* bs = is_k ? a.kbs_s : a.vbs_s;
            const int64_t eb = (a.layout == PKV_HND) ? page * bs[0] + h * bs[1] + off * bs[2]
                                                     : page * bs[0] + off * bs[1] + h * bs[2];
            uint8_t* bdst = (is_k ? a.k_bs : a.v_bs) + eb;
            if (c & 1)
                bdst[D / 32 + c / 2] = static_cast<uint8_t>(s_hi);
            else
                bdst[c / 2] = static_cast<uint8_t>(s_lo);
        } else {
            uint16_t* dst = static_cast<uint16_t*>(is_k ? a.k_cache : a.v_cache) + e;
            *reinterpret_cast<uint4*>(dst + 8 * c) = pack_bf16x8(lo);
            *reinterpret_cast<uint4*>(dst + D / 2 + 8 * c) = pack_bf16x8(hi);
        }
    }
}

// Tokens per thread of a cache fill (measured on GB300; see the launcher).
#ifndef PKV_WRITE_FILL_TOKENS
#define PKV_WRITE_FILL_TOKENS 2
#endif

template <int D, bool INTER, int KIND>
cudaError_t launch_t(const RopeArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const int per_tok = (a.Hq + 2 * a.Hkv) * (D / 16);  // work items of one token
    if (per_tok > 1024) return cudaErrorInvalidConfiguration;
    const int toks = per_tok >= 256 ? 1 : 256 / per_tok;  // tokens per group of the CTA
    // Two tokens per thread when there are enough tokens to keep every SM
    // busy (cache fills of bf16 and FP8 caches: twice the bytes in flight per
    // thread), with registers budgeted for four CTAs per SM (a few bytes of
    // spill, but 32 warps to hide the loads: measured fills of the ragged,
    // longctx and fp8 workloads 7%, 8% and 2% faster than at three CTAs,
    // qwen 2% slower; three or four tokens per thread were slower); one for
    // a decode step's few tokens and for NVFP4 (measured no faster there:
    // its quantiser is bound by instruction issue).
    const bool two = KIND != kFp4 && a.T >= 8192 && per_tok * toks <= 256;
    constexpr int UF = PKV_WRITE_FILL_TOKENS;
    const int64_t per_cta = static_cast<int64_t>(toks) * (two ? UF : 1);
    const int64_t blocks = (a.T + per_cta - 1) / per_cta;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    RopeArgs b = a;
    b.toks = toks;
    const dim3 grid(static_cast<unsigned>(blocks)), block(per_tok * toks);
    if constexpr (KIND != kFp4) {
        if (two) return launch_dependent(rope_kv_write_kernel<D, INTER, KIND, UF>, grid, block, 0, s, b);
    }
    return launch_dependent(rope_kv_write_kernel<D, INTER, KIND, 1>, grid, block, 0, s, b);
}

template <int D, bool INTER>
cudaError_t launch_k(const RopeArgs& a, cudaStream_t s) {
    switch (a.kind) {
        case kBf16: return launch_t<D, INTER, kBf16>(a, s);
        case kFp8: return launch_t<D, INTER, kFp8>(a, s);
        case kFp4: return launch_t<D, INTER, kFp4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_d(const RopeArgs& a, cudaStream_t s) {
    return a.interleaved ? launch_k<D, true>(a, s) : launch_k<D, false>(a, s);
}

// MLA latent-cache write (mainarch, MLA decode section: FP8 E4M3 ckv beside
// BF16 kpe). threadIdx.x of a token: [0, 32) the 16-value chunks of ckv
// (E4M3 of the correctly rounded quotient by the scale, as the FP8 KV
// write; 32-byte loads, 16-byte stores); [32, 36) kpe, chunks c and 32 + c
// as a D = 64 RoPE row; then four threads per q_pe row, rotated in place.
// threadIdx.y and blockIdx.x: tokens; with U > 1 a thread takes U tokens
// blockDim.y apart, all of whose loads are issued before any is used.
template <bool INTER, int U>
__global__ void __launch_bounds__(U > 1 ? 256 : 1024) mla_cache_write_kernel(const MlaWriteArgs a) {
    grid_dep_wait();  // as rope_kv_write_kernel: a programmatic dependent
    grid_dep_launch();
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.y * U + threadIdx.y;
    const int x = threadIdx.x;
    const int r = x - kMlaDc / 16;  // kpe / q_pe threads: 0..3 kpe, 4.. q_pe rows
    const int c = r & 3;
    const int row = r >> 2;          // 0 = kpe, 1 + h = q_pe head h
    if (r >= 0 && row > a.H) return;
    const int64_t num_slots = a.num_pages * a.page_size;

    // every load of the thread's tokens first; a skipped token's row is
    // still inside the [T, ...] inputs
    int32_t slot[U], pos[U];
    uint4 w0[U], w1[U];
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.y;
        live[u] = t < a.T;
        if (!live[u]) continue;
        slot[u] = __ldg(a.slots + t);
        pos[u] = __ldg(a.positions + t);
        if (r < 0) {  // ckv values 16x .. 16x + 15
            const uint16_t* src = a.ckv + t * a.ckv_s0 + 16 * x;
            w0[u] = *reinterpret_cast<const uint4*>(src);
            w1[u] = *reinterpret_cast<const uint4*>(src + 8);
        } else {
            const uint16_t* src = row == 0 ? a.kpe + t * a.kpe_s0 : a.q_pe + t * a.qp_s0 + (row - 1) * a.qp_s1;
            w0[u] = *reinterpret_cast<const uint4*>(src + 8 * c);
            w1[u] = *reinterpret_cast<const uint4*>(src + kMlaDr / 2 + 8 * c);
        }
    }
    float scale = 1.f;
    E4m3Rcp r8{1.f, 1.f, false};
    if (r < 0) {
        scale = __ldg(a.ckv_scale);
        r8 = e4m3_rcp(scale);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!live[u] || slot[u] < 0) continue;
        if (slot[u] >= num_slots) {
            if (x == 0) flag_error(a.err, PKV_FLAG_SLOT_RANGE);
            continue;
        }
        if (pos[u] < 0 || pos[u] >= a.max_pos) {
            if (x == 0) flag_error(a.err, PKV_FLAG_POSITION_RANGE);
            continue;
        }
        const int64_t t = t0 + static_cast<int64_t>(u) * blockDim.y;
        int64_t page, off;
        if (a.page_shift >= 0) {  // no division for power-of-two page sizes
            page = slot[u] >> a.page_shift;
            off = slot[u] & ((1 << a.page_shift) - 1);
        } else {
            page = slot[u] / a.page_size;
            off = slot[u] - page * a.page_size;
        }
        if (r < 0) {
            const uint2 q0 = pack_e4m3x8(unpack_bf16x8(w0[u]), scale, r8);
            const uint2 q1 = pack_e4m3x8(unpack_bf16x8(w1[u]), scale, r8);
            *reinterpret_cast<uint4*>(a.ckv_cache + page * a.cc_s0 + off * a.cc_s1 + 16 * x) =
                make_uint4(q0.x, q0.y, q1.x, q1.y);
            continue;
        }
        Chunk8 lo = unpack_bf16x8(w0[u]);
        Chunk8 hi = unpack_bf16x8(w1[u]);
        float cv[8], sv[8];
        load_cos_sin<kMlaDr, INTER>(a.cos_sin + pos[u] * a.cs_s0, c, cv, sv);
        rotate_row<INTER>(lo, hi, cv, sv);
        uint16_t* dst = row == 0 ? a.kpe_cache + page * a.kc_s0 + off * a.kc_s1
                                 : a.q_pe + t * a.qp_s0 + (row - 1) * a.qp_s1;
        *reinterpret_cast<uint4*>(dst + 8 * c) = pack_bf16x8(lo);
        *reinterpret_cast<uint4*>(dst + kMlaDr / 2 + 8 * c) = pack_bf16x8(hi);
    }
}

// Tokens per thread of an MLA cache fill.
#ifndef PKV_MLA_FILL_TOKENS
#define PKV_MLA_FILL_TOKENS 2
#endif

}  // namespace

cudaError_t launch_mla_cache_write(const MlaWriteArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const int per_tok = kMlaDc / 16 + 4 * (1 + a.H);  // threads of one token
    if (per_tok > 1024) return cudaErrorInvalidConfiguration;
    const int toks = per_tok >= 256 ? 1 : 256 / per_tok;
    // Two tokens per thread for large fills (CTAs of at most 256 threads):
    // twice the bytes in flight per thread. Measured on GB300 against one:
    // a 319,783-token fill 5% faster, a 51,199-token fill 5% slower (fewer
    // CTAs to spread over the SMs); three or four were slower. One for a
    // decode step's few tokens.
    constexpr int UF = PKV_MLA_FILL_TOKENS;
    const bool many = UF > 1 && a.T >= 131072 && per_tok * toks <= 256;
    const int64_t per_cta = static_cast<int64_t>(toks) * (many ? UF : 1);
    const int64_t blocks = (a.T + per_cta - 1) / per_cta;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks)), block(per_tok, toks);
    if (many) {
        if (a.interleaved) return launch_dependent(mla_cache_write_kernel<true, UF>, grid, block, 0, s, a);
        return launch_dependent(mla_cache_write_kernel<false, UF>, grid, block, 0, s, a);
    }
    if (a.interleaved) return launch_dependent(mla_cache_write_kernel<true, 1>, grid, block, 0, s, a);
    return launch_dependent(mla_cache_write_kernel<false, 1>, grid, block, 0, s, a);
}

cudaError_t launch_rope_kv_write(const RopeArgs& a, cudaStream_t s) {
    switch (a.D) {
        case 64: return launch_d<64>(a, s);
        case 128: return launch_d<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
