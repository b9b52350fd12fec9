/*
 * oracle.c -- plain, slow, float64 CPU oracle for the paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h). Built with gcc -O2
 * -ffp-contract=off so that no multiply-add is fused; every rounding below is
 * written out.
 *
 * Rounding model. A product of two float32 values (or of a bf16 and a
 * float32) is exact in float64; converting a float64 to float32 with C's
 * (float) cast rounds to nearest-even. For +, -, * and / of two float32
 * operands, computing in float64 and then rounding to float32 gives the
 * correctly rounded float32 result, because 53 >= 2*24 + 2 (double rounding
 * is innocuous at that width). So f32(x*c) and f32((double)a - (double)b)
 * below equal IEEE float32 arithmetic with no fused multiply-add.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* float32 <-> bits                                                        */
/* ---------------------------------------------------------------------- */
static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

float orc_f32(double x) { return (float)x; }

/* ---------------------------------------------------------------------- */
/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. A     */
/* bf16 pattern is the high half of the float32 pattern of the same value.  */
/* ---------------------------------------------------------------------- */
double orc_bf16_to_f64(uint16_t b) { return (double)bits_f32((uint32_t)b << 16); }

/* Round-to-nearest, ties-to-even, from the definition: the two bf16
 * neighbours of x are the truncated pattern (same sign, magnitude <= |x|) and
 * the next pattern up in magnitude; pick the nearer, and on a tie the one
 * whose last mantissa bit is 0. Above the largest finite bf16 the next
 * pattern up is infinity, whose value for this comparison is 2^128 (the
 * value an unbounded exponent would give). NaN maps to the quiet NaN 0x7FC0
 * with the input's sign. */
uint16_t orc_bf16_rne(float x) {
    uint32_t u = f32_bits(x);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return (uint16_t)((sign >> 16) | 0x7FC0u);
    if (mag == 0x7F800000u) return (uint16_t)((sign | mag) >> 16);
    uint32_t lo = mag & 0xFFFF0000u;
    uint32_t hi = lo + 0x10000u;
    double ax = (double)bits_f32(mag);
    double vlo = (double)bits_f32(lo);
    double vhi = (hi >= 0x7F800000u) ? ldexp(1.0, 128) : (double)bits_f32(hi);
    double dlo = ax - vlo, dhi = vhi - ax;
    uint32_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;
    return (uint16_t)((sign | pick) >> 16);
}

void orc_bf16_rne_n(const float* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(x[i]);
}

/* ---------------------------------------------------------------------- */
/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3         */
/* mantissa bits; no infinities; S.1111.111 is NaN; the largest finite      */
/* magnitude is S.1111.110 = 1.75 * 2^8 = 448; exponent field 0 holds the   */
/* subnormals m * 2^-9. (mainarch: "FP8 here is OCP e4m3fn"; Loom Kernels:  */
/* vLLM-compatible E4M3 cache bytes.)                                       */
/* ---------------------------------------------------------------------- */
double orc_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Magnitudes of codes 0x00..0x7E, increasing. */
static double g_e4m3_mag[127];
static int g_e4m3_ready = 0;
static void e4m3_table(void) {
    if (g_e4m3_ready) return;
    for (int c = 0; c < 127; ++c) g_e4m3_mag[c] = orc_e4m3_to_f64((uint8_t)c);
    g_e4m3_ready = 1;
}

/* Saturating round-to-nearest-even: magnitudes at or above 448 give 448
 * (saturation to the largest finite value, never NaN); below, the nearer of
 * the two neighbouring codes, ties to the even code (last mantissa bit 0);
 * the sign bit is kept (so -0 and tiny negatives give 0x80); NaN gives 0x7F
 * with the input's sign. */
uint8_t orc_e4m3_sat_rne(float x) {
    e4m3_table();
    double dx = (double)x;
    uint8_t sign = (f32_bits(x) >> 24) & 0x80u;
    if (isnan(dx)) return (uint8_t)(sign | 0x7F);
    double ax = fabs(dx);
    if (ax >= 448.0) return (uint8_t)(sign | 0x7E);
    /* largest code c with mag[c] <= ax (binary search over the sorted table) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_e4m3_mag[mid] <= ax) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (g_e4m3_mag[c] != ax) {
        double dlo = ax - g_e4m3_mag[c], dhi = g_e4m3_mag[c + 1] - ax;
        if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;
    }
    return (uint8_t)(sign | c);
}

void orc_e4m3_sat_rne_n(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_sat_rne(x[i]);
}

/* ---------------------------------------------------------------------- */
/* E2M1 ("e2m1fn", the 4-bit element of NVFP4 and MXFP4): 1 sign bit, 2     */
/* exponent bits (bias 1), 1 mantissa bit; no infinities or NaN. Exponent   */
/* field 0 is the subnormal m * 0.5. Magnitudes of codes 0..7:              */
/* 0, 0.5, 1, 1.5, 2, 3, 4, 6. (mainarch, decode-attention section: FP4 is   */
/* E2M1 with block scales.)                                                 */
/* ---------------------------------------------------------------------- */
double orc_e2m1_to_f64(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Saturating round-to-nearest-even: magnitudes >= 6 give 6; below, the
 * nearer of the two neighbouring codes, ties to the even code; the sign bit
 * is kept (tiny negatives give 0x8). NaN is not an input of this path. */
uint8_t orc_e2m1_sat_rne(float x) {
    double dx = (double)x;
    uint8_t sign = (f32_bits(x) >> 31) ? 0x8 : 0x0;
    double ax = fabs(dx);
    if (ax >= 6.0) return (uint8_t)(sign | 7);
    int c = 0;
    while (c < 7 && orc_e2m1_to_f64((uint8_t)(c + 1)) <= ax) ++c;
    if (orc_e2m1_to_f64((uint8_t)c) != ax) {
        double dlo = ax - orc_e2m1_to_f64((uint8_t)c), dhi = orc_e2m1_to_f64((uint8_t)(c + 1)) - ax;
        if (dhi < dlo || (dhi == dlo && (c & 1))) c = c + 1;
    }
    return (uint8_t)(sign | c);
}

void orc_e2m1_sat_rne_n(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_sat_rne(x[i]);
}

/*
 * NVFP4 block of 16 values y (float32) under the static scale g:
 *   s = E4M3(f32(amax / f32(6 g)))        (saturating RNE, positive)
 *   nibble_i = E2M1(f32(y_i / f32(g * s)))  (0 for every value when s = 0)
 * packed[i] holds value 2i in its low nibble and value 2i+1 in its high
 * nibble. Dequantisation: y_i ~ g * s * E2M1(nibble_i). (The 16-element
 * block with an E4M3 scale is Blackwell's NVFP4 form of mainarch's "E2M1
 * KV with block scales"; the scale choice maps the block's largest
 * magnitude to E2M1's largest value, 6.)
 */
void orc_nvfp4_block(const float* y, float g, uint8_t* packed, uint8_t* scale_byte) {
    double amax = 0.0;
    for (int i = 0; i < 16; ++i) {
        double a = fabs((double)y[i]);
        if (a > amax) amax = a;
    }
    float six_g = orc_f32(6.0 * (double)g);
    uint8_t sb = orc_e4m3_sat_rne(orc_f32(amax / (double)six_g));
    double s = orc_e4m3_to_f64(sb);
    *scale_byte = sb;
    float denom = orc_f32((double)g * s);
    for (int i = 0; i < 8; ++i) {
        uint8_t lo = 0, hi = 0;
        if (s != 0.0) {
            lo = orc_e2m1_sat_rne(orc_f32((double)y[2 * i] / (double)denom));
            hi = orc_e2m1_sat_rne(orc_f32((double)y[2 * i + 1] / (double)denom));
        }
        packed[i] = (uint8_t)(lo | (hi << 4));
    }
}

/* ---------------------------------------------------------------------- */
/* RoPE                                                                    */
/* Pairs: NeoX rotates (i, i + D/2); interleaved rotates (2i, 2i+1); both   */
/* use frequency index i in [0, D/2). With (c, s) the cos and sin of the    */
/* angle: y1 = x1*c - x2*s, y2 = x2*c + x1*s.                               */
/* (Loom Kernels, "Position and KV" row: NeoX/interleaved RoPE;             */
/* microLLM-rocm: split-half RoPE.)                                         */
/* ---------------------------------------------------------------------- */
static void pair_index(int i, int D, int interleaved, int* j1, int* j2) {
    if (interleaved) { *j1 = 2 * i; *j2 = 2 * i + 1; }
    else { *j1 = i; *j2 = i + D / 2; }
}

void orc_rope_rotate_f64(const double* x, double* y, int D, double pos, double base, int interleaved) {
    for (int i = 0; i < D / 2; ++i) {
        double ang = pos * pow(base, -2.0 * i / D);
        double c = cos(ang), s = sin(ang);
        int j1, j2;
        pair_index(i, D, interleaved, &j1, &j2);
        y[j1] = x[j1] * c - x[j2] * s;
        y[j2] = x[j2] * c + x[j1] * s;
    }
}

/* Table row layout: cs_row[i] = cos, cs_row[D/2 + i] = sin, float32. Every
 * product and the sum/difference is rounded to float32; nothing is fused. */
void orc_rope_row_f32(const uint16_t* x, const float* cs_row, float* y, int D, int interleaved) {
    for (int i = 0; i < D / 2; ++i) {
        double c = (double)cs_row[i], s = (double)cs_row[D / 2 + i];
        int j1, j2;
        pair_index(i, D, interleaved, &j1, &j2);
        double x1 = orc_bf16_to_f64(x[j1]), x2 = orc_bf16_to_f64(x[j2]);
        float a = orc_f32(x1 * c);
        float b = orc_f32(x2 * s);
        float e = orc_f32(x2 * c);
        float f = orc_f32(x1 * s);
        y[j1] = orc_f32((double)a - (double)b);
        y[j2] = orc_f32((double)e + (double)f);
    }
}

/* ---------------------------------------------------------------------- */
/* Cache layout: NHD = [pages, P, Hkv, D], HND = [pages, Hkv, P, D].        */
/* slot = page * P + offset. (Loom Kernels, "Position and KV" row: NHD/HND  */
/* cache views; the slot encoding is the plainest reading of "paged-KV      */
/* write".)                                                                 */
/* ---------------------------------------------------------------------- */
static int64_t cache_index(int layout, int64_t page, int off, int h, int d, int Hkv, int P, int D) {
    if (layout == 1) return ((page * Hkv + h) * (int64_t)P + off) * D + d;
    return ((page * P + off) * (int64_t)Hkv + h) * D + d;
}

static float scale_of(const float* sc, int n_scale, int h) { return n_scale == 1 ? sc[0] : sc[h]; }

/* Encode one float32 value as a cache element. FP8: z = f32(y / scale), then
 * saturating round-to-nearest-even E4M3 (the quotient is the correctly
 * rounded float32 quotient; dequantisation is byte * scale). */
static void store_elem(void* cache, int64_t idx, float y, int fp8, float scale) {
    if (fp8) {
        float z = orc_f32((double)y / (double)scale);
        ((uint8_t*)cache)[idx] = orc_e4m3_sat_rne(z);
    } else {
        ((uint16_t*)cache)[idx] = orc_bf16_rne(y);
    }
}

int64_t orc_rope_kv_write(int64_t T, int Hq, int Hkv, int D, int page_size,
                          uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* positions, const float* cos_sin, int64_t max_pos,
                          void* k_cache, void* v_cache, int64_t num_pages, int layout,
                          int interleaved, int fp8, const float* k_scale, const float* v_scale,
                          int n_scale, const int32_t* slot_mapping) {
    int64_t bad = 0;
    float* y = (float*)malloc(sizeof(float) * (size_t)D);
    int64_t num_slots = num_pages * page_size;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t pos = positions[t];
        if (slot < 0) continue;
        if (slot >= num_slots || pos < 0 || pos >= max_pos) { ++bad; continue; }
        const float* cs = cos_sin + pos * D;
        int64_t page = slot / page_size;
        int off = (int)(slot % page_size);
        if (q) {
            for (int h = 0; h < Hq; ++h) {
                uint16_t* row = q + (t * Hq + h) * D;
                orc_rope_row_f32(row, cs, y, D, interleaved);
                for (int d = 0; d < D; ++d) row[d] = orc_bf16_rne(y[d]);
            }
        }
        for (int h = 0; h < Hkv; ++h) {
            const uint16_t* krow = k + (t * Hkv + h) * D;
            const uint16_t* vrow = v + (t * Hkv + h) * D;
            float ks = fp8 ? scale_of(k_scale, n_scale, h) : 1.0f;
            float vs = fp8 ? scale_of(v_scale, n_scale, h) : 1.0f;
            orc_rope_row_f32(krow, cs, y, D, interleaved);
            for (int d = 0; d < D; ++d)
                store_elem(k_cache, cache_index(layout, page, off, h, d, Hkv, page_size, D), y[d], fp8, ks);
            for (int d = 0; d < D; ++d)
                store_elem(v_cache, cache_index(layout, page, off, h, d, Hkv, page_size, D),
                           (float)orc_bf16_to_f64(vrow[d]), fp8, vs);
        }
    }
    free(y);
    return bad;
}

/*
 * NVFP4 cache write: as orc_rope_kv_write, but each (token, kv head) row of
 * rotated k / plain v is quantised in blocks of 16 (orc_nvfp4_block) with
 * the static scale of its head. Value caches hold packed E2M1 pairs,
 * NHD [pages, P, Hkv, D/2] or HND [pages, Hkv, P, D/2]; scale caches hold
 * one E4M3 byte per block, [pages, P, Hkv, D/16] or [pages, Hkv, P, D/16].
 */
int64_t orc_rope_kv_write_nvfp4(int64_t T, int Hq, int Hkv, int D, int page_size,
                                uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const int32_t* positions, const float* cos_sin, int64_t max_pos,
                                uint8_t* k_cache, uint8_t* v_cache, uint8_t* k_block_scale,
                                uint8_t* v_block_scale, int64_t num_pages, int layout, int interleaved,
                                const float* k_scale, const float* v_scale, int n_scale,
                                const int32_t* slot_mapping) {
    int64_t bad = 0;
    float* y = (float*)malloc(sizeof(float) * (size_t)D);
    int64_t num_slots = num_pages * page_size;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t pos = positions[t];
        if (slot < 0) continue;
        if (slot >= num_slots || pos < 0 || pos >= max_pos) { ++bad; continue; }
        const float* cs = cos_sin + pos * D;
        int64_t page = slot / page_size;
        int off = (int)(slot % page_size);
        if (q) {
            for (int h = 0; h < Hq; ++h) {
                uint16_t* row = q + (t * Hq + h) * D;
                orc_rope_row_f32(row, cs, y, D, interleaved);
                for (int d = 0; d < D; ++d) row[d] = orc_bf16_rne(y[d]);
            }
        }
        for (int h = 0; h < Hkv; ++h) {
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which == 0 ? k : v) + (t * Hkv + h) * D;
                float g = scale_of(which == 0 ? k_scale : v_scale, n_scale, h);
                if (which == 0) orc_rope_row_f32(src, cs, y, D, interleaved);
                else for (int d = 0; d < D; ++d) y[d] = (float)orc_bf16_to_f64(src[d]);
                uint8_t* vals = which == 0 ? k_cache : v_cache;
                uint8_t* scales = which == 0 ? k_block_scale : v_block_scale;
                for (int blk = 0; blk < D / 16; ++blk) {
                    uint8_t packed[8], sb;
                    orc_nvfp4_block(y + 16 * blk, g, packed, &sb);
                    int64_t vrow = cache_index(layout, page, off, h, 0, Hkv, page_size, D / 2);
                    for (int i = 0; i < 8; ++i) vals[vrow + 8 * blk + i] = packed[i];
                    scales[cache_index(layout, page, off, h, blk, Hkv, page_size, D / 16)] = sb;
                }
            }
        }
    }
    free(y);
    return bad;
}

/* ---------------------------------------------------------------------- */
/* Decode attention                                                        */
/* ---------------------------------------------------------------------- */
/* A cache as the decode reads it: bf16 bits (fmt 0), E4M3 bytes (fmt 1) or
 * NVFP4 packed E2M1 pairs with one E4M3 scale byte per 16 elements (fmt 2). */
typedef struct {
    const void* data;
    const uint8_t* block_scale;
    int fmt;
} cache_view;

static double cache_value(const cache_view* c, int layout, int64_t page, int off, int h, int d, int Hkv, int P,
                          int D) {
    if (c->fmt == 2) {
        int64_t e = cache_index(layout, page, off, h, d, Hkv, P, D);
        uint8_t byte = ((const uint8_t*)c->data)[e / 2];
        uint8_t nib = (e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
        uint8_t sb = c->block_scale[cache_index(layout, page, off, h, d / 16, Hkv, P, D / 16)];
        return orc_e2m1_to_f64(nib) * orc_e4m3_to_f64(sb);
    }
    int64_t idx = cache_index(layout, page, off, h, d, Hkv, P, D);
    if (c->fmt == 1) return orc_e4m3_to_f64(((const uint8_t*)c->data)[idx]);
    return orc_bf16_to_f64(((const uint16_t*)c->data)[idx]);
}

/*
 * The split count sequence b's pages are dealt into: splits_per_seq[b]
 * (reading: a count below 1 is taken as 1 and one above num_splits as
 * num_splits, the records the call has), or num_splits for every sequence
 * when splits_per_seq is NULL.
 */
static int seq_split_count(const int32_t* splits_per_seq, int b, int num_splits) {
    if (!splits_per_seq) return num_splits;
    int sb = splits_per_seq[b];
    if (sb < 1) sb = 1;
    if (sb > num_splits) sb = num_splits;
    return sb;
}

/*
 * One query head. Readings: query head h reads kv head floor(h / G) with
 * G = Hq / Hkv; the context is positions 0..L-1 (L = seq_lens[b], which
 * counts the new token); no mask, window, ALiBi or soft-cap. Split s covers
 * pages [s*pps, min((s+1)*pps, npages)) with npages = ceil(L/P) and
 * pps = ceil(npages / S_b), where S_b = seq_splits is the number of splits
 * this sequence's pages are dealt into (the call's num_splits, or a count of
 * its own per sequence, at most num_splits); records s >= S_b, and any
 * split past the last page, are empty. Each split is a plain two-pass softmax in float64:
 * m = max score, l = sum exp(score - m), o = sum exp(score - m) * v / l,
 * lse = m + ln l; an empty split gives o = 0, lse = -inf. Scores are
 * softmax_scale * sum_d q_d * k_d with k = cache value * k_scale (FP8) and
 * v likewise with v_scale. Pages whose block-table entry is outside
 * [0, num_pages) are left out of the sum.
 */
static void decode_head_impl(int b, int h, int Hq, int Hkv, int D, int page_size, const uint16_t* q_row,
                             const cache_view* kc, const cache_view* vc, int64_t num_pages, int layout,
                             const float* k_scale, const float* v_scale, int n_scale,
                             const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                             double softmax_scale, int num_splits, int seq_splits, double* out_partial,
                             double* lse_partial) {
    int fp8 = kc->fmt != 0;  /* the static per-tensor / per-head scales apply */
    int G = Hq / Hkv;
    int kvh = h / G;
    int64_t L = seq_lens[b];
    if (L < 0) L = 0;
    int64_t npages = (L + page_size - 1) / page_size;
    if (npages > max_pages) npages = max_pages;
    if (L > npages * page_size) L = npages * page_size;
    int64_t pps = (npages + seq_splits - 1) / seq_splits;
    double ks = fp8 ? (double)scale_of(k_scale, n_scale, kvh) : 1.0;
    double vs = fp8 ? (double)scale_of(v_scale, n_scale, kvh) : 1.0;
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) qd[d] = orc_bf16_to_f64(q_row[d]);
    int64_t cap = pps * page_size > 0 ? pps * page_size : 1;
    double* sc = (double*)malloc(sizeof(double) * (size_t)cap);
    int64_t* where = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);

    for (int s = 0; s < num_splits; ++s) {
        double* o = out_partial + (int64_t)s * D;
        int64_t p0 = (int64_t)s * pps, p1 = p0 + pps;
        if (p1 > npages) p1 = npages;
        int64_t n = 0;
        for (int64_t p = p0; p < p1; ++p) {
            int64_t page = block_tables[(int64_t)b * max_pages + p];
            if (page < 0 || page >= num_pages) continue;
            for (int off = 0; off < page_size; ++off) {
                int64_t t = p * page_size + off;
                if (t >= L) break;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += qd[d] * (cache_value(kc, layout, page, off, kvh, d, Hkv, page_size, D) * ks);
                sc[n] = softmax_scale * dot;
                where[n] = page * page_size + off;
                ++n;
            }
        }
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n == 0) { lse_partial[s] = -INFINITY; continue; }
        double m = sc[0];
        for (int64_t i = 1; i < n; ++i) if (sc[i] > m) m = sc[i];
        double l = 0.0;
        for (int64_t i = 0; i < n; ++i) l += exp(sc[i] - m);
        for (int64_t i = 0; i < n; ++i) {
            double p = exp(sc[i] - m) / l;
            int64_t page = where[i] / page_size;
            int off = (int)(where[i] % page_size);
            for (int d = 0; d < D; ++d)
                o[d] += p * (cache_value(vc, layout, page, off, kvh, d, Hkv, page_size, D) * vs);
        }
        lse_partial[s] = m + log(l);
    }
    free(where);
    free(sc);
    free(qd);
}

void orc_decode_head(int b, int h, int Hq, int Hkv, int D, int page_size,
                     const uint16_t* q_row, const void* k_cache, const void* v_cache,
                     int64_t num_pages, int layout, int fp8, const float* k_scale,
                     const float* v_scale, int n_scale, const int32_t* block_tables,
                     int max_pages, const int32_t* seq_lens, double softmax_scale,
                     int num_splits, double* out_partial, double* lse_partial) {
    cache_view kc = {k_cache, NULL, fp8 ? 1 : 0}, vc = {v_cache, NULL, fp8 ? 1 : 0};
    decode_head_impl(b, h, Hq, Hkv, D, page_size, q_row, &kc, &vc, num_pages, layout, k_scale, v_scale, n_scale,
                     block_tables, max_pages, seq_lens, softmax_scale, num_splits, num_splits, out_partial,
                     lse_partial);
}

/* NVFP4 caches: value k = g_k * s_block * E2M1 (and likewise v). */
void orc_decode_head_nvfp4(int b, int h, int Hq, int Hkv, int D, int page_size,
                           const uint16_t* q_row, const uint8_t* k_cache, const uint8_t* v_cache,
                           const uint8_t* k_block_scale, const uint8_t* v_block_scale, int64_t num_pages,
                           int layout, const float* k_scale, const float* v_scale, int n_scale,
                           const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                           double softmax_scale, int num_splits, double* out_partial, double* lse_partial) {
    cache_view kc = {k_cache, k_block_scale, 2}, vc = {v_cache, v_block_scale, 2};
    decode_head_impl(b, h, Hq, Hkv, D, page_size, q_row, &kc, &vc, num_pages, layout, k_scale, v_scale, n_scale,
                     block_tables, max_pages, seq_lens, softmax_scale, num_splits, num_splits, out_partial,
                     lse_partial);
}


static void paged_decode_all(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                             const cache_view* kc, const cache_view* vc, int64_t num_pages, int layout,
                             const float* k_scale, const float* v_scale, int n_scale,
                             const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                             double softmax_scale, int num_splits, const int32_t* splits_per_seq,
                             double* out_partial, double* lse_partial) {
    double* o = (double*)malloc(sizeof(double) * (size_t)num_splits * D);
    double* l = (double*)malloc(sizeof(double) * (size_t)num_splits);
    for (int b = 0; b < B; ++b) {
        int sb = seq_split_count(splits_per_seq, b, num_splits);
        for (int h = 0; h < Hq; ++h) {
            decode_head_impl(b, h, Hq, Hkv, D, page_size, q + ((int64_t)b * Hq + h) * D, kc, vc, num_pages, layout,
                             k_scale, v_scale, n_scale, block_tables, max_pages, seq_lens, softmax_scale, num_splits,
                             sb, o, l);
            for (int s = 0; s < num_splits; ++s) {
                int64_t r = ((int64_t)b * num_splits + s) * Hq + h;
                lse_partial[r] = l[s];
                for (int d = 0; d < D; ++d) out_partial[r * D + d] = o[(int64_t)s * D + d];
            }
        }
    }
    free(l);
    free(o);
}

void orc_paged_decode_nvfp4_splits(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                                   const uint8_t* k_cache, const uint8_t* v_cache, const uint8_t* k_block_scale,
                                   const uint8_t* v_block_scale, int64_t num_pages, int layout, const float* k_scale,
                                   const float* v_scale, int n_scale, const int32_t* block_tables, int max_pages,
                                   const int32_t* seq_lens, double softmax_scale, int num_splits,
                                   const int32_t* splits_per_seq, double* out_partial, double* lse_partial) {
    cache_view kc = {k_cache, k_block_scale, 2}, vc = {v_cache, v_block_scale, 2};
    paged_decode_all(B, Hq, Hkv, D, page_size, q, &kc, &vc, num_pages, layout, k_scale, v_scale, n_scale,
                     block_tables, max_pages, seq_lens, softmax_scale, num_splits, splits_per_seq, out_partial,
                     lse_partial);
}

void orc_paged_decode_nvfp4(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                            const uint8_t* k_cache, const uint8_t* v_cache, const uint8_t* k_block_scale,
                            const uint8_t* v_block_scale, int64_t num_pages, int layout, const float* k_scale,
                            const float* v_scale, int n_scale, const int32_t* block_tables, int max_pages,
                            const int32_t* seq_lens, double softmax_scale, int num_splits,
                            double* out_partial, double* lse_partial) {
    orc_paged_decode_nvfp4_splits(B, Hq, Hkv, D, page_size, q, k_cache, v_cache, k_block_scale, v_block_scale,
                                  num_pages, layout, k_scale, v_scale, n_scale, block_tables, max_pages, seq_lens,
                                  softmax_scale, num_splits, NULL, out_partial, lse_partial);
}

void orc_paged_decode_splits(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                             const void* k_cache, const void* v_cache, int64_t num_pages, int layout,
                             int fp8, const float* k_scale, const float* v_scale, int n_scale,
                             const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                             double softmax_scale, int num_splits, const int32_t* splits_per_seq,
                             double* out_partial, double* lse_partial) {
    cache_view kc = {k_cache, NULL, fp8 ? 1 : 0}, vc = {v_cache, NULL, fp8 ? 1 : 0};
    paged_decode_all(B, Hq, Hkv, D, page_size, q, &kc, &vc, num_pages, layout, k_scale, v_scale, n_scale,
                     block_tables, max_pages, seq_lens, softmax_scale, num_splits, splits_per_seq, out_partial,
                     lse_partial);
}

void orc_paged_decode(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                      const void* k_cache, const void* v_cache, int64_t num_pages, int layout,
                      int fp8, const float* k_scale, const float* v_scale, int n_scale,
                      const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                      double softmax_scale, int num_splits, double* out_partial,
                      double* lse_partial) {
    orc_paged_decode_splits(B, Hq, Hkv, D, page_size, q, k_cache, v_cache, num_pages, layout, fp8, k_scale,
                            v_scale, n_scale, block_tables, max_pages, seq_lens, softmax_scale, num_splits, NULL,
                            out_partial, lse_partial);
}

/* ---------------------------------------------------------------------- */
/* Multi-head latent attention (MLA), absorbed decode form.                */
/* mainarch, MLA decode section: the cache holds one compressed latent     */
/* per token -- ckv, 512 values, stored as FP8 E4M3 -- beside a 64-value   */
/* positional part kpe stored as BF16; the per-head projections are        */
/* applied to the query before the cache is read (q_lat = the query        */
/* already in latent space), so every head attends to the same cache rows: */
/* per-head dot scores over [ckv | kpe], a local softmax with an exported  */
/* LSE, softmax-weighted latent outputs (V = ckv), split-K over the        */
/* sequence and a stage-2 merge of the partial records (orc_lse_merge).    */
/* ---------------------------------------------------------------------- */

/*
 * MLA cache write. For every token t with slot_mapping[t] >= 0 (slot =
 * page * page_size + offset; ckv_cache [pages][P][Dc] bytes, kpe_cache
 * [pages][P][Dr] bf16 bits):
 *   ckv_cache[slot][d] = E4M3(f32(ckv[t][d] / ckv_scale))   saturating RNE,
 *                        the rule of the FP8 KV write;
 *   kpe_cache[slot]    = bf16(RoPE(kpe[t]))  RoPE of the Dr-value row with
 *                        cos_sin row positions[t] (orc_rope_row_f32);
 *   q_pe[t][h]         = bf16(RoPE(q_pe[t][h])) in place, when q_pe != NULL.
 * Tokens whose slot is >= num_pages*page_size or whose position is outside
 * [0, max_pos) are skipped (q_pe untouched) and counted in the return value.
 */
int64_t orc_mla_cache_write(int64_t T, int H, int Dc, int Dr, int page_size, uint16_t* q_pe,
                            const uint16_t* ckv, const uint16_t* kpe, const int32_t* positions,
                            const float* cos_sin, int64_t max_pos, uint8_t* ckv_cache, uint16_t* kpe_cache,
                            int64_t num_pages, int interleaved, float ckv_scale, const int32_t* slot_mapping) {
    int64_t bad = 0;
    float* y = (float*)malloc(sizeof(float) * (size_t)Dr);
    int64_t num_slots = num_pages * page_size;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t pos = positions[t];
        if (slot < 0) continue;
        if (slot >= num_slots || pos < 0 || pos >= max_pos) { ++bad; continue; }
        const float* cs = cos_sin + pos * Dr;
        if (q_pe) {
            for (int h = 0; h < H; ++h) {
                uint16_t* row = q_pe + (t * H + h) * Dr;
                orc_rope_row_f32(row, cs, y, Dr, interleaved);
                for (int r = 0; r < Dr; ++r) row[r] = orc_bf16_rne(y[r]);
            }
        }
        for (int d = 0; d < Dc; ++d) {
            float z = orc_f32(orc_bf16_to_f64(ckv[t * Dc + d]) / (double)ckv_scale);
            ckv_cache[slot * Dc + d] = orc_e4m3_sat_rne(z);
        }
        orc_rope_row_f32(kpe + t * Dr, cs, y, Dr, interleaved);
        for (int r = 0; r < Dr; ++r) kpe_cache[slot * Dr + r] = orc_bf16_rne(y[r]);
    }
    free(y);
    return bad;
}

/*
 * MLA decode. For sequence b with L = seq_lens[b] tokens, split s covers the
 * logical pages [s*pps, min((s+1)*pps, npages)), npages = ceil(L/P),
 * pps = ceil(npages / S). For head h, over the split's tokens t:
 *   score_t = softmax_scale * ( sum_d q_lat[b,h,d] * ckv_t[d]
 *                             + sum_r q_pe[b,h,r]  * kpe_t[r] )
 * with ckv_t[d] = E4M3 byte value * ckv_scale; then a plain two-pass softmax
 * in float64: out_partial[b,s,h,:] = sum_t e^(score_t - m) ckv_t / l,
 * lse_partial[b,s,h] = m + ln l (empty split: 0 and -inf). Pages whose
 * block-table entry is outside [0, num_pages) are left out.
 * q_lat [B][H][Dc], q_pe [B][H][Dr] bf16 bits; out_partial [B][S][H][Dc],
 * lse_partial [B][S][H].
 */
void orc_mla_decode(int B, int H, int Dc, int Dr, int page_size, const uint16_t* q_lat, const uint16_t* q_pe,
                    const uint8_t* ckv_cache, const uint16_t* kpe_cache, int64_t num_pages, float ckv_scale,
                    const int32_t* block_tables, int max_pages, const int32_t* seq_lens, double softmax_scale,
                    int num_splits, double* out_partial, double* lse_partial) {
    orc_mla_decode_splits(B, H, Dc, Dr, page_size, q_lat, q_pe, ckv_cache, kpe_cache, num_pages, ckv_scale,
                          block_tables, max_pages, seq_lens, softmax_scale, num_splits, NULL, out_partial,
                          lse_partial);
}

/* orc_mla_decode with a split count per sequence (reading: as for the GQA
 * decode, sequence b's pages are dealt into splits_per_seq[b] splits,
 * clamped to [1, num_splits], by the rule above; its records past that
 * count are empty). NULL = num_splits for every sequence. */
void orc_mla_decode_splits(int B, int H, int Dc, int Dr, int page_size, const uint16_t* q_lat, const uint16_t* q_pe,
                           const uint8_t* ckv_cache, const uint16_t* kpe_cache, int64_t num_pages, float ckv_scale,
                           const int32_t* block_tables, int max_pages, const int32_t* seq_lens, double softmax_scale,
                           int num_splits, const int32_t* splits_per_seq, double* out_partial,
                           double* lse_partial) {
    double* ql = (double*)malloc(sizeof(double) * (size_t)Dc);
    double* qr = (double*)malloc(sizeof(double) * (size_t)Dr);
    double cs = (double)ckv_scale;
    for (int b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        if (L < 0) L = 0;
        int64_t npages = (L + page_size - 1) / page_size;
        if (npages > max_pages) npages = max_pages;
        if (L > npages * page_size) L = npages * page_size;
        int64_t sb = seq_split_count(splits_per_seq, b, num_splits);
        int64_t pps = (npages + sb - 1) / sb;
        int64_t cap = pps * page_size > 0 ? pps * page_size : 1;
        double* sc = (double*)malloc(sizeof(double) * (size_t)cap);
        int64_t* where = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
        for (int h = 0; h < H; ++h) {
            for (int d = 0; d < Dc; ++d) ql[d] = orc_bf16_to_f64(q_lat[((int64_t)b * H + h) * Dc + d]);
            for (int r = 0; r < Dr; ++r) qr[r] = orc_bf16_to_f64(q_pe[((int64_t)b * H + h) * Dr + r]);
            for (int s = 0; s < num_splits; ++s) {
                int64_t row = ((int64_t)b * num_splits + s) * H + h;
                double* o = out_partial + row * Dc;
                int64_t p0 = (int64_t)s * pps, p1 = p0 + pps;
                if (p1 > npages) p1 = npages;
                int64_t n = 0;
                for (int64_t p = p0; p < p1; ++p) {
                    int64_t page = block_tables[(int64_t)b * max_pages + p];
                    if (page < 0 || page >= num_pages) continue;
                    for (int off = 0; off < page_size; ++off) {
                        if (p * page_size + off >= L) break;
                        int64_t slot = page * page_size + off;
                        double dot = 0.0;
                        for (int d = 0; d < Dc; ++d) dot += ql[d] * (orc_e4m3_to_f64(ckv_cache[slot * Dc + d]) * cs);
                        for (int r = 0; r < Dr; ++r) dot += qr[r] * orc_bf16_to_f64(kpe_cache[slot * Dr + r]);
                        sc[n] = softmax_scale * dot;
                        where[n] = slot;
                        ++n;
                    }
                }
                for (int d = 0; d < Dc; ++d) o[d] = 0.0;
                if (n == 0) { lse_partial[row] = -INFINITY; continue; }
                double m = sc[0];
                for (int64_t i = 1; i < n; ++i) if (sc[i] > m) m = sc[i];
                double l = 0.0;
                for (int64_t i = 0; i < n; ++i) l += exp(sc[i] - m);
                for (int64_t i = 0; i < n; ++i) {
                    double w = exp(sc[i] - m) / l;
                    for (int d = 0; d < Dc; ++d) o[d] += w * (orc_e4m3_to_f64(ckv_cache[where[i] * Dc + d]) * cs);
                }
                lse_partial[row] = m + log(l);
            }
        }
        free(where);
        free(sc);
    }
    free(qr);
    free(ql);
}

/*
 * Merge of S partials of one row: M = max_s lse_s; w_s = exp(lse_s - M);
 * out = sum_s w_s o_s / sum_s w_s; lse = M + ln sum_s w_s. A row whose every
 * split is empty (all lse = -inf) gives out = 0, lse = -inf.
 */
void orc_lse_merge(int B, int S, int Hq, int D, const double* out_partial,
                   const double* lse_partial, double* out, double* lse) {
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            double* orow = out + ((int64_t)b * Hq + h) * D;
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            double M = -INFINITY;
            for (int s = 0; s < S; ++s) {
                double x = lse_partial[((int64_t)b * S + s) * Hq + h];
                if (x > M) M = x;
            }
            if (M == -INFINITY) { lse[(int64_t)b * Hq + h] = -INFINITY; continue; }
            double W = 0.0;
            for (int s = 0; s < S; ++s) {
                int64_t r = ((int64_t)b * S + s) * Hq + h;
                double w = exp(lse_partial[r] - M);
                W += w;
                for (int d = 0; d < D; ++d) orow[d] += w * out_partial[r * D + d];
            }
            for (int d = 0; d < D; ++d) orow[d] /= W;
            lse[(int64_t)b * Hq + h] = M + log(W);
        }
    }
}
