/*
 * pkv.h -- C ABI of the paged-KV GQA decode step for NVIDIA GB300 (sm_103a).
 *
 * One decode step of transformer attention over a paged KV cache is three
 * calls on one CUDA stream (for multi-head latent attention, the MLA pair
 * pkv_mla_cache_write / pkv_paged_mla_decode takes the place of the first
 * two):
 *
 *   pkv_rope_kv_write     rotate q and k of the new token(s) (NeoX or
 *                         interleaved RoPE) and write k and v into the paged
 *                         cache as bf16 or static-scale FP8 E4M3 bytes.
 *   pkv_paged_gqa_decode  attention of each query head over the pages its
 *                         sequence's block table names, split-K over the
 *                         context, one partial output and LSE per split.
 *   pkv_lse_merge         log-sum-exp merge of the split partials into the
 *                         bf16 output.
 *
 * Sources of the operation (page title, section):
 *   - Loom Kernels, "Supported operator paths" table: row "Position and KV"
 *     (NeoX/interleaved RoPE + native/static-FP8 paged-KV write, packed QKV,
 *     NHD/HND cache views, static per-tensor/per-head FP8 E4M3 scales) and
 *     row "Attention" (paged MQA/GQA decode, local split-K/LSE merge).
 *   - mainarch, decode-attention section: split-KV online softmax with a
 *     combine of the partials, paged KV in the vLLM/SGLang sense (a block
 *     table maps logical blocks to physical pages), GQA reading each KV head
 *     once per group, OCP e4m3fn FP8.
 *
 * Conventions for every call:
 *   - Memory. All tensor pointers are DEVICE addresses of caller-owned memory
 *     (borrowed for the duration of the call's GPU work). The library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Streams. Every call only enqueues GPU work on `stream` (NULL = the
 *     legacy default stream) and returns; results are ready when that
 *     stream's work completes. Calls contain no host synchronisation.
 *   - Ordering. The step's kernels (cache write, decode, merge, copy) are
 *     launched as programmatic dependents, so one may start its prologue
 *     while its predecessor on the stream finishes; each waits for that
 *     predecessor (griddepcontrol.wait) before it reads anything another
 *     grid may have written, and before it can finish. Only the decodes
 *     (block tables, seq_lens, a split plan) and the planned merge (the
 *     plan's split counts) read index inputs before that wait, and only the
 *     cache writes and the decodes let their successor start early; no
 *     kernel writes index inputs. Calls on one stream therefore see each
 *     other's results exactly as plain stream order would give.
 *   - Status. The return value reports argument validation and launch
 *     errors only: PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED are returned
 *     before anything is launched; PKV_ERR_CUDA reports a launch failure
 *     (cudaGetLastError). Device-side problems with index VALUES (a slot,
 *     position, page id or sequence length out of range) are not visible to
 *     the host at call time: the kernels skip the offending element and OR a
 *     PKV_FLAG_* bit into *err_flag (a device int32 the caller zeroes; may be
 *     NULL). No kernel traps, asserts or faults on bad index values.
 *   - Tensors. A pkv_tensor is a strided view: shape and strides in ELEMENTS,
 *     outermost first. Innermost strides must be 1 where stated. Tensors are
 *     passed by pointer to their descriptor; the descriptor is read during
 *     the call only. Where a tensor is optional, a NULL descriptor pointer
 *     or a descriptor whose ptr is NULL both mean "absent".
 */
#ifndef PKV_H
#define PKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* shapes, strides, dtypes or enums inconsistent   */
    PKV_ERR_UNSUPPORTED = 2,  /* consistent but outside what the kernels handle  */
    PKV_ERR_CUDA = 3          /* a CUDA runtime/driver call or launch failed     */
} pkv_status;

typedef enum { PKV_NHD = 0, PKV_HND = 1 } pkv_layout;
typedef enum { PKV_ROPE_NEOX = 0, PKV_ROPE_INTERLEAVED = 1 } pkv_rope_style;
/* PKV_FP4_E2M1X2: one byte holding two E2M1 values, the even-indexed value
 * in the low nibble (the value caches of the NVFP4 entry points). */
typedef enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1, PKV_F32 = 2, PKV_I32 = 3, PKV_FP4_E2M1X2 = 4 } pkv_dtype;

/* Bits OR-ed into *err_flag by the kernels. */
#define PKV_FLAG_SLOT_RANGE     0x01  /* slot_mapping entry >= num_pages * page_size        */
#define PKV_FLAG_POSITION_RANGE 0x02  /* positions entry outside [0, cos_sin rows)          */
#define PKV_FLAG_PAGE_RANGE     0x04  /* a needed block-table entry outside [0, num_pages)   */
#define PKV_FLAG_SEQ_LEN_RANGE  0x08  /* seq_lens entry < 0 or > block-table width * 16      */
#define PKV_FLAG_DUPLICATE_SLOT 0x10  /* two tokens of one call map to the same slot         */
#define PKV_FLAG_WAIT_TIMEOUT   0x20  /* an in-kernel wait gave up after its time limit      */
#define PKV_FLAG_PLAN_RANGE     0x40  /* a split plan entry outside the batch or its records */

typedef struct {
    void*   ptr;        /* device address (NULL allowed only where stated) */
    int32_t dtype;      /* pkv_dtype                                        */
    int32_t ndim;       /* 1..4                                             */
    int64_t shape[4];   /* extents, outermost first                         */
    int64_t stride[4];  /* in elements                                      */
} pkv_tensor;

/*
 * pkv_rope_kv_write -- fused RoPE + paged-KV cache write.
 * (Loom Kernels, "Supported operator paths", row "Position and KV";
 *  "Evidence" table, rows "RoPE + paged-KV write" and "Static FP8 KV-cache
 *  write"; microLLM-rocm, optimisation checkpoints: split-half RoPE and
 *  positions-aware RoPE with a mapped KV store.)
 *
 * For every token t with slot_mapping[t] >= 0, with (c_i, s_i) =
 * cos_sin[positions[t], i] and cos_sin[positions[t], D/2 + i]:
 *   pairs (i, i + D/2) for NeoX or (2i, 2i+1) for interleaved, i < D/2:
 *     y1 = x1*c - x2*s,  y2 = x2*c + x1*s
 *   each product and the sum/difference rounded to float32, no fused
 *   multiply-add. Then:
 *   q[t]   <- bf16 round-to-nearest-even of the rotated q   (in place)
 *   k_cache[slot] <- rotated k, v_cache[slot] <- v, each as
 *     bf16 RNE (bf16 cache), or
 *     E4M3(y / scale): the correctly rounded float32 quotient, then
 *     saturating (to +-448) round-to-nearest-even OCP E4M3 (FP8 cache).
 *   slot = page * page_size + offset.
 *
 * q            [T, Hq, D]  bf16, innermost stride 1, rows 16-byte aligned;
 *              rotated IN PLACE. ptr may be NULL (cache fill without q).
 * k, v         [T, Hkv, D] bf16, read only, same alignment rule. Strided
 *              views of a packed QKV buffer are accepted.
 * positions    [T] int32, contiguous.
 * cos_sin      [max_pos, D] float32, innermost stride 1, 16-byte aligned rows:
 *              columns [0, D/2) cos, [D/2, D) sin of frequency index i.
 * k_cache,
 * v_cache      NHD: [num_pages, page_size, Hkv, D]; HND: [num_pages, Hkv,
 *              page_size, D]; dtype PKV_BF16 or PKV_FP8_E4M3 (both the same);
 *              innermost stride 1, other strides multiples of 16 bytes.
 * slot_mapping [T] int32; < 0 skips the token (q, k and v untouched).
 * k_scale,
 * v_scale      FP8 cache only: [1] (per tensor) or [Hkv] (per head) float32,
 *              positive; ignored (ptr may be NULL) for a bf16 cache.
 * layout       pkv_layout; rope_style pkv_rope_style.
 * Supported: D in {64, 128}; Hq a multiple of Hkv (or q NULL).
 * Errors: a slot >= num_pages*page_size sets PKV_FLAG_SLOT_RANGE, a position
 * outside [0, max_pos) sets PKV_FLAG_POSITION_RANGE; that token is skipped
 * entirely. Two tokens with the same slot: the surviving write is unspecified.
 * q must not alias k, v or the caches; the caches must not alias k or v.
 */
pkv_status pkv_rope_kv_write(const pkv_tensor* q, const pkv_tensor* k, const pkv_tensor* v, const pkv_tensor* positions,
                             const pkv_tensor* cos_sin, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                             const pkv_tensor* slot_mapping, const pkv_tensor* k_scale, const pkv_tensor* v_scale,
                             int32_t layout, int32_t rope_style, int32_t* err_flag,
                             pkv_stream_t stream);

/*
 * pkv_paged_gqa_decode -- paged MQA/GQA split-K decode attention.
 * (mainarch, decode-attention section: split-KV online softmax, paged KV
 *  with a block table and a shuffled page layout, GQA sharing each KV head
 *  load, FP8 KV dequantised in-kernel; Loom Kernels, "Attention" row.)
 *
 * For sequence b with L = seq_lens[b] (counting the new token) and
 * npages = ceil(L / 16), split s in [0, num_splits) covers logical pages
 * [s*pps, min((s+1)*pps, npages)), pps = ceil(npages / num_splits).
 * Query head h reads kv head h / (Hq/Hkv). Over the tokens of the split:
 *   score_t = softmax_scale * sum_d q[b,h,d] * K_t[d]
 *   out_partial[b,s,h,:] = sum_t exp(score_t - m) V_t / sum_t exp(score_t - m)
 *   lse_partial[b,s,h]   = m + ln sum_t exp(score_t - m)   (natural log)
 * with m = max_t score_t; an empty split gives 0 and -inf. K_t, V_t are the
 * cache values (FP8: byte * k_scale / v_scale of the kv head).
 *
 * q            [B, Hq, D] bf16 (already rotated), innermost stride 1.
 * k_cache,
 * v_cache      as for pkv_rope_kv_write; page_size must be 16; the base
 *              address 16-byte aligned.
 * block_tables [B, max_pages] int32, innermost stride 1; entries past a
 *              sequence's npages are never read.
 * seq_lens     [B] int32.
 * softmax_scale  multiplies q.k (natural-log units).
 * num_splits   >= 1, <= 4096 (see pkv_choose_num_splits).
 * out_partial  [B, num_splits, Hq, D] float32, innermost stride 1.
 * lse_partial  [B, num_splits, Hq] float32, innermost stride 1.
 * k_scale,
 * v_scale      as for pkv_rope_kv_write.
 * Supported: D in {64, 128}; 1 <= Hq/Hkv <= 16.
 * Errors: a block-table entry outside [0, num_pages) sets
 * PKV_FLAG_PAGE_RANGE and that page is left out; seq_lens[b] < 0 or
 * > 16*max_pages sets PKV_FLAG_SEQ_LEN_RANGE and L is clamped to [0,
 * 16*max_pages]. Outputs must not alias inputs.
 */
pkv_status pkv_paged_gqa_decode(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                const pkv_tensor* block_tables, const pkv_tensor* seq_lens, float softmax_scale,
                                int32_t num_splits, const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                const pkv_tensor* k_scale, const pkv_tensor* v_scale, int32_t layout,
                                int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_rope_kv_write_nvfp4 -- pkv_rope_kv_write into a 4-bit (NVFP4) cache.
 * (mainarch, decode-attention section: 4-bit E2M1 KV with block scales,
 *  dequantised in-kernel, with NVFP4 named as the open work. NVFP4 is the
 *  form used here: E2M1 values, one E4M3 scale per 16 consecutive values of
 *  a row, and a static float32 scale per tensor or per kv head.)
 *
 * RoPE and the rounding of every product and sum are those of
 * pkv_rope_kv_write. Each (token, kv head) row y of rotated k, or of v, is
 * then quantised block by block (16 values, blocks aligned to the row),
 * with g the static scale of the head:
 *   amax = max |y_i| over the block
 *   s    = E4M3( f32(amax / f32(6 g)) )      saturating RNE, the block's
 *                                            scale byte
 *   e_i  = E2M1( f32(y_i / f32(g s)) )       saturating (to +-6) RNE, the
 *                                            sign kept; every e_i = 0 when
 *                                            s = 0
 * where f32() is the correctly rounded float32 result. The stored value is
 * y_i ~ g * s * e_i.
 *
 * k_cache,
 * v_cache      NHD [num_pages, page_size, Hkv, D/2] or HND [num_pages, Hkv,
 *              page_size, D/2], dtype PKV_FP4_E2M1X2 (values 2j and 2j+1 of
 *              a row in byte j, low nibble first); innermost stride 1, other
 *              strides multiples of 16 bytes, base 16-byte aligned.
 * k_block_scale,
 * v_block_scale  the same layout with D/16 in place of D/2, dtype
 *              PKV_FP8_E4M3 (byte j = scale of values 16j..16j+15);
 *              innermost stride 1.
 * k_scale,
 * v_scale      [1] or [Hkv] float32, positive, required.
 * Every other argument, the supported sizes and the errors are those of
 * pkv_rope_kv_write. The caches and scale caches must not alias one another
 * or q, k, v.
 */
pkv_status pkv_rope_kv_write_nvfp4(const pkv_tensor* q, const pkv_tensor* k, const pkv_tensor* v,
                                   const pkv_tensor* positions, const pkv_tensor* cos_sin,
                                   const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                   const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                   const pkv_tensor* slot_mapping, const pkv_tensor* k_scale,
                                   const pkv_tensor* v_scale, int32_t layout, int32_t rope_style,
                                   int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_paged_gqa_decode_nvfp4 -- pkv_paged_gqa_decode over NVFP4 caches.
 * (mainarch, decode-attention section: paged + GQA + FP4 KV in one kernel,
 *  the block scales applied as the cache is read.)
 *
 * The same computation as pkv_paged_gqa_decode with cache values
 *   K_t[d] = k_scale[kvh] * s_k(t, d/16) * e_k(t, d)
 * (and likewise V), s the E4M3 block scale and e the E2M1 value.
 *
 * k_cache, v_cache, k_block_scale, v_block_scale  as for
 *              pkv_rope_kv_write_nvfp4, HND layout only (NHD returns
 *              PKV_ERR_UNSUPPORTED), page_size 16; the 16 x D/16 scale bytes
 *              of one (page, kv head) must be contiguous (innermost two
 *              strides 1 and D/16) and start on a 16-byte boundary (the
 *              outer two strides multiples of 16 bytes, base 16-byte aligned).
 * Every other argument, the supported sizes and the errors are those of
 * pkv_paged_gqa_decode; the partials feed pkv_lse_merge unchanged.
 */
pkv_status pkv_paged_gqa_decode_nvfp4(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                      const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                      const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                      float softmax_scale, int32_t num_splits, const pkv_tensor* out_partial,
                                      const pkv_tensor* lse_partial, const pkv_tensor* k_scale,
                                      const pkv_tensor* v_scale, int32_t layout, int32_t* err_flag,
                                      pkv_stream_t stream);

/*
 * pkv_mla_cache_write -- write of one or more tokens into a paged MLA
 * latent cache (multi-head latent attention, absorbed decode form).
 * (mainarch, MLA decode section: a paged latent cache holding FP8 E4M3 ckv
 *  beside BF16 kpe; the cache becomes a 512-value compressed latent plus a
 *  64-value positional part per token.)
 *
 * For every token t with slot_mapping[t] >= 0 (slot = page * P + offset):
 *   ckv_cache[page, offset, d] = E4M3( f32(ckv[t, d] / ckv_scale) )
 *       (correctly rounded quotient, saturating round-to-nearest-even, as
 *       the FP8 KV write);
 *   kpe_cache[page, offset, :] = bf16 RNE of RoPE(kpe[t, :]) and, when q_pe
 *   is given, q_pe[t, h, :] = bf16 RNE of RoPE(q_pe[t, h, :]) in place:
 *   the 64-value rotation of pkv_rope_kv_write (pairs (i, i+32) NeoX or
 *   (2i, 2i+1) interleaved, cos_sin row positions[t], products and sums each
 *   rounded to float32).
 *
 * q_pe         [T, H, 64] bf16, innermost stride 1, rows 16-byte aligned;
 *              rotated IN PLACE; ptr may be NULL. 1 <= H <= 200.
 * ckv          [T, 512] bf16 (the compressed latent), kpe [T, 64] bf16; read
 *              only; innermost stride 1, rows 16-byte aligned.
 * positions, slot_mapping  [T] int32, contiguous; slot < 0 skips the token.
 * cos_sin      [max_pos, 64] float32, columns [0, 32) cos, [32, 64) sin.
 * ckv_cache    [num_pages, P, 512] PKV_FP8_E4M3; kpe_cache [num_pages, P, 64]
 *              PKV_BF16; innermost stride 1, other strides multiples of 16
 *              bytes, bases 16-byte aligned. Any P >= 1 (the decode takes 64).
 * ckv_scale    [1] float32, positive (static per-tensor scale).
 * rope_style   pkv_rope_style.
 * Errors: as pkv_rope_kv_write (PKV_FLAG_SLOT_RANGE, PKV_FLAG_POSITION_RANGE;
 * that token is skipped, q_pe untouched).
 */
pkv_status pkv_mla_cache_write(const pkv_tensor* q_pe, const pkv_tensor* ckv, const pkv_tensor* kpe,
                               const pkv_tensor* positions, const pkv_tensor* cos_sin,
                               const pkv_tensor* ckv_cache, const pkv_tensor* kpe_cache,
                               const pkv_tensor* slot_mapping, const pkv_tensor* ckv_scale, int32_t rope_style,
                               int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_paged_mla_decode -- paged MLA split-K decode, absorbed form.
 * (mainarch, MLA decode section: per-head dot scores, local softmax with
 *  exported LSE, softmax-weighted output tiles, split-K across the sequence
 *  with a stage-2 merge of the partial records.)
 *
 * Every query head h of sequence b attends to the same latent rows. For
 * L = seq_lens[b], npages = ceil(L/64), split s covers logical pages
 * [s*pps, min((s+1)*pps, npages)), pps = ceil(npages / num_splits):
 *   score_t = softmax_scale * ( sum_d q_lat[b,h,d] * ckv_t[d]
 *                             + sum_r q_pe[b,h,r]  * kpe_t[r] ),
 *   ckv_t[d] = E4M3 value * ckv_scale,
 *   out_partial[b,s,h,:] = sum_t exp(score_t - m) ckv_t / sum_t exp(score_t - m)
 *   lse_partial[b,s,h]   = m + ln sum_t exp(score_t - m)
 * (empty split: 0 and -inf). pkv_lse_merge with D = 512 merges the splits.
 * Arithmetic: the tensor cores read the E4M3 cache bytes as they are, with
 * q_lat as two E4M3 terms under a per-head power-of-two scale (exact for
 * every value within 2^9 of the head's largest magnitude) and the softmax
 * weights as three E5M2 terms that sum exactly to their f16 rounding; sums
 * in float32.
 *
 * q_lat        [B, H, 512] bf16: the query already projected into the latent
 *              space; q_pe [B, H, 64] bf16, already rotated. Innermost stride
 *              1, other strides even, base 4-byte aligned. 1 <= H <= 16.
 * ckv_cache,
 * kpe_cache    as for pkv_mla_cache_write with P = 64.
 * block_tables [B, max_pages] int32 (64-token pages), seq_lens [B] int32.
 * out_partial  [B, num_splits, H, 512] float32 (innermost stride 1, other
 *              strides even, base 8-byte aligned); lse_partial
 *              [B, num_splits, H] float32.
 * ckv_scale    [1] float32.
 * num_splits   >= 1, <= 4096 (see pkv_choose_num_splits_mla).
 * Errors: as pkv_paged_gqa_decode.
 */
pkv_status pkv_paged_mla_decode(const pkv_tensor* q_lat, const pkv_tensor* q_pe, const pkv_tensor* ckv_cache,
                                const pkv_tensor* kpe_cache, const pkv_tensor* block_tables,
                                const pkv_tensor* seq_lens, float softmax_scale, int32_t num_splits,
                                const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                const pkv_tensor* ckv_scale, int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_choose_num_splits_mla -- split count for pkv_paged_mla_decode (host
 * only). B sequences, H heads, total_pages / max_pages in 64-token pages,
 * sm_count the device's SM count. Models the persistent decode (two CTAs
 * per SM taking the (sequence, split) items): a fixed cost per item and a
 * per-chunk time (128 tokens, two pages; higher when two CTAs share an SM)
 * for the longest sequence and a mean other one, the larger of a CTA's share
 * of the items, the largest item and the HBM time, plus the partial
 * records. Returns a value in [1, min(1024, max_pages)]; 1 for empty or
 * invalid input.
 */
int32_t pkv_choose_num_splits_mla(int32_t B, int32_t H, int64_t total_pages, int32_t max_pages, int32_t sm_count);

/*
 * pkv_lse_merge -- merge of the split partials.
 * (mainarch, decode-attention section: the combine of split-KV partials;
 *  Loom Kernels, "Attention" row: local split-K/LSE merge.)
 *
 *   M = max_s lse_partial[b,s,h];  w_s = exp(lse_partial[b,s,h] - M)
 *   out[b,h,:] = bf16_rne( sum_s w_s out_partial[b,s,h,:] / sum_s w_s )
 *   lse_out[b,h] = M + ln sum_s w_s
 * A row whose every split is empty gives out = 0 and lse_out = -inf.
 *
 * out_partial  [B, S, Hq, D] float32, innermost stride 1.
 * lse_partial  [B, S, Hq] float32, innermost stride 1.
 * out          [B, Hq, D] bf16, innermost stride 1.
 * lse_out      [B, Hq] float32; ptr may be NULL.
 * Supported: D in {64, 128, 512} (512: the latent output of
 * pkv_paged_mla_decode).
 */
pkv_status pkv_lse_merge(const pkv_tensor* out_partial, const pkv_tensor* lse_partial, const pkv_tensor* out,
                         const pkv_tensor* lse_out, pkv_stream_t stream);

/*
 * Split plans: a split count of its own for every sequence.
 * (Loom Kernels, "Evidence" table, row "Local split-K paged decode": the
 *  split-K is local to each sequence; mainarch, decode-attention section:
 *  split-KV over long contexts, then the combine.)
 *
 * With one split count for the whole batch, a batch of mixed lengths gives
 * CTAs of very different sizes and the step waits for the longest. A plan
 * deals sequence b's pages into S_b splits of its own, so that every CTA
 * streams about the same number of pages: for sequence b (npages =
 * ceil(L/16)), split s in [0, S_b) covers pages [s*pps, min((s+1)*pps,
 * npages)), pps = ceil(npages / S_b) -- pkv_paged_gqa_decode's rule with
 * S_b in place of num_splits. The partial records keep the layout
 * [B, S, Hq, D] (S >= max S_b); sequence b writes records [0, S_b) and its
 * records [S_b, S) are neither written nor read.
 */

/*
 * pkv_plan_splits -- the host-side plan (no CUDA call).
 *
 * seq_lens       host [B] int32 (each clamped to [0, 16*max_pages], as the
 *                decode does).
 * Hkv, Hq, D, cache_dtype, sm_count  as for pkv_choose_num_splits
 *                (cache_dtype PKV_BF16, PKV_FP8_E4M3 or PKV_FP4_E2M1X2).
 * max_pages      the block-table width.
 * max_splits     the largest S_b allowed, in [1, 4095] (the records the
 *                caller will allocate at most).
 * target_pages   pages per split to aim for; 0 = chosen by a cost model of
 *                the decode on GB300 (per-CTA start-up, per-page streaming,
 *                HBM time, partial records), the plan's counterpart of
 *                pkv_choose_num_splits.
 * splits_per_seq host [B] int32, out: S_b = min(max_splits,
 *                ceil(npages / T)), at least 1, reduced to the splits that
 *                hold pages when that keeps the same page ranges.
 * num_records    out: max_b S_b, the S to allocate the partials with.
 * work           host [work_capacity, 2] int32, out (may be NULL with
 *                work_capacity 0 to size the plan): one (sequence, split)
 *                item per CTA, item i = ((b << 12) | s, first page of the
 *                split), ordered by decreasing page count (ties by b, s) so
 *                the longest items are dispatched first.
 * num_work       out: sum_b S_b, the number of items.
 * Returns PKV_ERR_INVALID_ARG on inconsistent sizes or null outputs, or when
 * work is given and work_capacity < num_work (the counts are still
 * written); PKV_ERR_UNSUPPORTED for B > 2^19 or max_pages > 2^26.
 */
pkv_status pkv_plan_splits(const int32_t* seq_lens, int32_t B, int32_t Hkv, int32_t Hq, int32_t D,
                           int32_t max_pages, int32_t cache_dtype, int32_t sm_count, int32_t max_splits,
                           int32_t target_pages, int32_t* splits_per_seq, int32_t* num_records, int32_t* work,
                           int64_t work_capacity, int64_t* num_work);

/*
 * pkv_paged_gqa_decode_planned -- pkv_paged_gqa_decode (or, with block
 * scales, pkv_paged_gqa_decode_nvfp4) under a split plan: one CTA per work
 * item and kv head.
 *
 * k_block_scale,
 * v_block_scale  NULL (or ptr NULL) for bf16 / FP8 caches; the NVFP4 block-
 *                scale caches for NVFP4 caches (HND only).
 * splits_per_seq device [B] int32: the plan's S_b.
 * work           device [W, 2] int32 (strides 2, 1; 8-byte aligned): the
 *                plan's items. Every (b, s < S_b) should appear once; the
 *                second word is only a hint for an early block-table read
 *                (a plan made from other lengths stays correct, its page
 *                ranges follow this call's seq_lens).
 * out_partial    [B, S, Hq, D] float32 with S >= every S_b, S <= 4095.
 * lse_partial    [B, S, Hq] float32.
 * Every other argument is that of the uniform decode. The computation of
 * each written record is that of pkv_paged_gqa_decode with S_b splits.
 * Errors: besides the uniform decode's, an item whose sequence is outside
 * [0, B) or whose split is >= S is skipped and S_b outside [1, S], or an
 * item with s >= S_b, sets PKV_FLAG_PLAN_RANGE (S_b is clamped).
 */
pkv_status pkv_paged_gqa_decode_planned(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                        const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                        const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                        float softmax_scale, const pkv_tensor* splits_per_seq,
                                        const pkv_tensor* work, const pkv_tensor* out_partial,
                                        const pkv_tensor* lse_partial, const pkv_tensor* k_scale,
                                        const pkv_tensor* v_scale, int32_t layout, int32_t* err_flag,
                                        pkv_stream_t stream);

/*
 * pkv_plan_splits_mla -- the split plan of the MLA decode (host only; no CUDA
 * call). The persistent MLA decode (two CTAs per SM) takes the plan's items
 * in order; when every sequence can have a CTA of its own, the automatic
 * plan (target_pages = 0) makes at most one item per CTA, all of nearly
 * equal length: the smallest even page target (whole 128-token chunks)
 * whose items fit the CTAs; past that, the longest split of
 * pkv_choose_num_splits_mla. seq_lens counts tokens, pages are the cache's
 * 64-token pages (max_pages = the block-table width); every other argument
 * and output is that of pkv_plan_splits.
 */
pkv_status pkv_plan_splits_mla(const int32_t* seq_lens, int32_t B, int32_t H, int32_t max_pages, int32_t sm_count,
                               int32_t max_splits, int32_t target_pages, int32_t* splits_per_seq,
                               int32_t* num_records, int32_t* work, int64_t work_capacity, int64_t* num_work);

/*
 * pkv_paged_mla_decode_planned -- pkv_paged_mla_decode under a split plan
 * (splits_per_seq device [B] int32, work device [W, 2] int32 with strides 2,
 * 1, as for pkv_paged_gqa_decode_planned); out_partial [B, S, H, 512] and
 * lse_partial [B, S, H] with S >= every S_b, S <= 4095. Each written record
 * is that of pkv_paged_mla_decode with S_b splits; records [S_b, S) of
 * sequence b are not written. Merge with pkv_lse_merge_planned (D = 512).
 * Errors: besides pkv_paged_mla_decode's, an item whose sequence is outside
 * [0, B) or whose split is >= S is skipped and S_b outside [1, S], or an
 * item with s >= S_b, sets PKV_FLAG_PLAN_RANGE (S_b is clamped).
 */
pkv_status pkv_paged_mla_decode_planned(const pkv_tensor* q_lat, const pkv_tensor* q_pe, const pkv_tensor* ckv_cache,
                                        const pkv_tensor* kpe_cache, const pkv_tensor* block_tables,
                                        const pkv_tensor* seq_lens, float softmax_scale,
                                        const pkv_tensor* splits_per_seq, const pkv_tensor* work,
                                        const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                        const pkv_tensor* ckv_scale, int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_lse_merge_planned -- pkv_lse_merge of each sequence's own records
 * [0, S_b) (S_b = splits_per_seq[b], device [B] int32, clamped to [1, S]).
 */
pkv_status pkv_lse_merge_planned(const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                 const pkv_tensor* splits_per_seq, const pkv_tensor* out, const pkv_tensor* lse_out,
                                 pkv_stream_t stream);

/*
 * pkv_choose_num_splits -- split count for pkv_paged_gqa_decode (host only,
 * no GPU work). (mainarch, MLA decode section: split-K of 64 vs 8 changes the
 * per-token time about threefold; Loom Kernels, "Evidence" table, row
 * "Local split-K paged decode".)
 *
 * B, Hkv: batch and kv heads; total_pages = sum over the batch of
 * ceil(seq_len/16); max_pages = the largest ceil(seq_len/16); cache_dtype the
 * value cache's pkv_dtype (PKV_BF16, PKV_FP8_E4M3 or PKV_FP4_E2M1X2); sm_count the device's SM count. Models each split as one CTA
 * (a fixed start-up plus a per-page streaming time, measured on GB300)
 * and returns the S in [1, min(1024, max_pages)] with the lowest estimated
 * step time: the larger of the HBM-bound streaming time (with the CTAs'
 * start-up and, past one wave of CTAs, part of the longest split's excess)
 * and the longest split's own time, plus the partial records' traffic.
 * Returns 1 for empty or invalid input.
 */
int32_t pkv_choose_num_splits(int32_t B, int32_t Hkv, int32_t Hq, int32_t D, int64_t total_pages,
                              int32_t max_pages, int32_t cache_dtype, int32_t sm_count);

/*
 * pkv_validate_indices -- device check of index values before a step.
 * (The pages' test practice of checking every span before the GPU uses it:
 *  mainarch, kernel ABI layer; Loom Kernels, "What Loom owns": invalid-input
 *  behaviour is part of the contract.)
 *
 * Sets PKV_FLAG_SEQ_LEN_RANGE for seq_lens entries < 0 or > 16*max_pages,
 * PKV_FLAG_PAGE_RANGE for block-table entries a sequence needs that are
 * outside [0, num_pages), PKV_FLAG_SLOT_RANGE for slot_mapping entries >=
 * num_pages*16 and, when slot_bitmap is given, PKV_FLAG_DUPLICATE_SLOT if
 * two non-negative slot_mapping entries are equal.
 * block_tables [B, max_pages] int32; seq_lens [B] int32; slot_mapping [T]
 * int32 (ptr may be NULL to skip slot checks); slot_bitmap: caller-provided
 * device scratch of ceil(num_pages*16/32) int32 words, which this call
 * zeroes and then uses (ptr may be NULL to skip the duplicate check).
 * err_flag must be non-NULL.
 */
pkv_status pkv_validate_indices(const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                const pkv_tensor* slot_mapping, int64_t num_pages,
                                const pkv_tensor* slot_bitmap, int32_t* err_flag, pkv_stream_t stream);

/*
 * pkv_validate_indices_static -- the same check as pkv_validate_indices,
 * including the duplicate-slot check, for callers that cannot allocate
 * device memory. (No counterpart on the pages: this entry point exists for
 * callers of this library, not for the method.)
 *
 * Who needs it: an engine whose allocator has already taken all free device
 * memory for its KV-cache pool cannot hand out a fresh scratch buffer for
 * the slot bitmap, and a latency-critical path may not call cudaMalloc or
 * cudaFree at all, because both can synchronise the whole device. This entry
 * point therefore takes no scratch argument and allocates nothing: the
 * bitmap lives in a fixed device array inside the library, of
 * PKV_STATIC_VALIDATE_MAX_SLOTS bits (1 MiB), which every GPU that loads the
 * library keeps until the process exits.
 *
 * Arguments are those of pkv_validate_indices without slot_bitmap.
 * num_pages * 16 must not exceed PKV_STATIC_VALIDATE_MAX_SLOTS, else the call
 * returns PKV_ERR_UNSUPPORTED and launches nothing. The first call on a
 * device looks up the array's device address (once per device, with that
 * device current); make that first call before any stream capture. If that
 * lookup fails, the call returns PKV_ERR_CUDA and the next call on the device
 * tries the lookup again; once it has succeeded it is not repeated. Every
 * call clears the part of the bitmap its pool uses (num_pages * 16 bits) on
 * `stream` before using it; bits an earlier call left above that part are
 * never read, because slots past the pool are flagged as out of range
 * before the bitmap is touched. All calls share
 * the one array: calls whose GPU work overlaps (on different streams, or
 * different host threads on one device) race on it and may report false or
 * missed duplicates. Calls ordered on one stream are safe.
 */
#define PKV_STATIC_VALIDATE_MAX_SLOTS (1 << 23)
pkv_status pkv_validate_indices_static(const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                       const pkv_tensor* slot_mapping, int64_t num_pages, int32_t* err_flag,
                                       pkv_stream_t stream);

/*
 * pkv_copy -- copy of `bytes` bytes from src to dst by the SMs, on `stream`
 * (moves a decode step's inputs in and its results out; not one of the
 * step's calls).
 *
 * dst, src     each device memory of the current device, managed memory,
 *              or host memory that CUDA has page-locked and mapped at the
 *              same address (the pinned allocations of cudaHostAlloc /
 *              cudaMallocHost under unified addressing, which the SMs of a
 *              GB300 read and write over NVLink-C2C); each must hold
 *              `bytes` bytes; the ranges must not overlap. Any alignment
 *              (16-byte aligned pairs move in 16-byte words).
 * Launched as a programmatic dependent: it waits for the preceding grid on
 * the stream before reading src, and the next grid starts only once the
 * copy has finished (so the copied bytes may be any later call's inputs,
 * index inputs included). Errors: bytes < 0, a NULL pointer or
 * overlapping ranges give PKV_ERR_INVALID_ARG; a pointer the SMs cannot
 * address (by cudaPointerGetAttributes) gives PKV_ERR_UNSUPPORTED, and
 * nothing is launched. bytes == 0 launches nothing.
 */
pkv_status pkv_copy(void* dst, const void* src, int64_t bytes, pkv_stream_t stream);

/*
 * pkv_stream_read -- streaming-read ceiling (a measurement helper; not one of
 * the decode step's calls). (mainarch, decode-attention section: a pure
 * device-memory streaming read is measured first and is the ceiling each
 * decode kernel is held to.)
 *
 * Reads `bytes` bytes at `buf` once, in one launch of `ctas` CTAs, with
 * 16-byte non-caching loads, and writes one folded word per CTA to sink[0,
 * ctas). buf: device memory, 16-byte aligned; bytes: a multiple of 16;
 * sink: device memory of at least `ctas` uint32 words; 1 <= ctas <= 65535.
 */
pkv_status pkv_stream_read(const void* buf, int64_t bytes, uint32_t* sink, int32_t ctas,
                           pkv_stream_t stream);

/*
 * pkv_selftest_bounded_wait -- self-test of the bounded in-kernel waits
 * behind PKV_FLAG_WAIT_TIMEOUT (a diagnostic; not one of the decode step's
 * calls). One CTA waits on mbarriers that nothing completes: one warp gives
 * up after about limit_ns and ORs PKV_FLAG_WAIT_TIMEOUT into *err_flag; a
 * second warp, with a limit 100 times longer, stops on the first one's
 * abort signal. elapsed_ns[0] and [1] receive the two waiting times. The
 * GPU context stays usable afterwards.
 * limit_ns: 100,000 .. 10,000,000 (0.1 .. 10 ms); err_flag: device int32
 * (the caller zeroes it); elapsed_ns: device memory of two uint64 words.
 */
pkv_status pkv_selftest_bounded_wait(int64_t limit_ns, int32_t* err_flag, uint64_t* elapsed_ns,
                                     pkv_stream_t stream);

/* Static description of a status code. */
const char* pkv_status_string(int32_t status);

/* ABI version of this header (bumped on any signature change). */
int32_t pkv_abi_version(void);
#define PKV_ABI_VERSION 7

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
