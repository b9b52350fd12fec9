/*
 * oracle.h -- plain, slow, float64 CPU oracle for the paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or
 * calls this code: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no source, header, table or constant with the
 * CUDA library.
 *
 * What it computes (the three calls of the hot path):
 *   orc_rope_kv_write  -- RoPE of q and k (NeoX or interleaved pairs), then
 *                         bf16 or static-scale FP8 E4M3 cache bytes written
 *                         at slot_mapping into NHD/HND page views.
 *                         (Loom Kernels, "Supported operator paths" table,
 *                         row "Position and KV"; "Evidence" table, row
 *                         "Static FP8 KV-cache write".)
 *   orc_decode_head /
 *   orc_paged_decode   -- paged MQA/GQA decode attention, split-K over the
 *                         context, one normalised partial output and one LSE
 *                         per split. (mainarch, decode-attention section:
 *                         split-KV online softmax, paged KV with a block
 *                         table, GQA; Loom Kernels, "Attention" row.)
 *   orc_lse_merge      -- log-sum-exp merge of the split partials
 *                         (mainarch, decode-attention section, "tree
 *                         combine"; Loom Kernels, "local split-K/LSE merge").
 *
 * Readings where the pages are silent are stated beside each function.
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scalar encoders and decoders (own bit-level definitions). */
uint16_t orc_bf16_rne(float x);
double   orc_bf16_to_f64(uint16_t b);
uint8_t  orc_e4m3_sat_rne(float x);
double   orc_e4m3_to_f64(uint8_t b);
float    orc_f32(double x);

/* E2M1 (4-bit, e2m1fn) codes and the NVFP4 block quantiser. */
uint8_t  orc_e2m1_sat_rne(float x);
double   orc_e2m1_to_f64(uint8_t code);
void     orc_nvfp4_block(const float* y, float g, uint8_t* packed, uint8_t* scale_byte);

/* Vector forms of the encoders, for exhaustive tests. */
void orc_e2m1_sat_rne_n(const float* x, uint8_t* out, int64_t n);
void orc_bf16_rne_n(const float* x, uint16_t* out, int64_t n);
void orc_e4m3_sat_rne_n(const float* x, uint8_t* out, int64_t n);

/* Analytic rotation in float64 (no table, no rounding): for invariants. */
void orc_rope_rotate_f64(const double* x, double* y, int D, double pos, double base, int interleaved);

/* Byte-exact rotation of one bf16 row with a float32 table row, giving the
 * float32 results (before any cache encoding). */
void orc_rope_row_f32(const uint16_t* x, const float* cs_row, float* y, int D, int interleaved);

/*
 * Cache write. T tokens. q (may be NULL) is [T,Hq,D] bf16 bits, rotated in
 * place and re-encoded bf16. k, v [T,Hkv,D] bf16 bits (read only). The
 * caches are contiguous arrays of num_pages pages in the given layout
 * (0 = NHD [pages,P,Hkv,D], 1 = HND [pages,Hkv,P,D]) of bf16 bits
 * (fp8 = 0) or E4M3 bytes (fp8 = 1). Scales: n_scale = 1 or Hkv floats.
 * Tokens whose slot is negative are skipped; tokens whose slot is beyond the
 * pool, or whose position is outside [0, max_pos), are skipped and counted.
 * Returns the number of skipped-and-counted tokens.
 */
int64_t orc_rope_kv_write(int64_t T, int Hq, int Hkv, int D, int page_size,
                          uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* positions, const float* cos_sin, int64_t max_pos,
                          void* k_cache, void* v_cache, int64_t num_pages, int layout,
                          int interleaved, int fp8, const float* k_scale, const float* v_scale,
                          int n_scale, const int32_t* slot_mapping);

/*
 * Decode of one query head h of sequence b into num_splits partials:
 * out_partial[s*D + d], lse_partial[s]. q_row is the (rotated) bf16 q of
 * that head, D values.
 */
void orc_decode_head(int b, int h, int Hq, int Hkv, int D, int page_size,
                     const uint16_t* q_row, const void* k_cache, const void* v_cache,
                     int64_t num_pages, int layout, int fp8, const float* k_scale,
                     const float* v_scale, int n_scale, const int32_t* block_tables,
                     int max_pages, const int32_t* seq_lens, double softmax_scale,
                     int num_splits, double* out_partial, double* lse_partial);

/* All heads: q [B,Hq,D]; out_partial [B,S,Hq,D]; lse_partial [B,S,Hq]. */
void orc_paged_decode(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                      const void* k_cache, const void* v_cache, int64_t num_pages, int layout,
                      int fp8, const float* k_scale, const float* v_scale, int n_scale,
                      const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                      double softmax_scale, int num_splits, double* out_partial,
                      double* lse_partial);

/* NVFP4 caches (packed E2M1 values + one E4M3 scale byte per 16 elements,
 * static scales g per tensor or per head); see oracle.c. */
int64_t orc_rope_kv_write_nvfp4(int64_t T, int Hq, int Hkv, int D, int page_size,
                                uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const int32_t* positions, const float* cos_sin, int64_t max_pos,
                                uint8_t* k_cache, uint8_t* v_cache, uint8_t* k_block_scale,
                                uint8_t* v_block_scale, int64_t num_pages, int layout, int interleaved,
                                const float* k_scale, const float* v_scale, int n_scale,
                                const int32_t* slot_mapping);
void orc_decode_head_nvfp4(int b, int h, int Hq, int Hkv, int D, int page_size,
                           const uint16_t* q_row, const uint8_t* k_cache, const uint8_t* v_cache,
                           const uint8_t* k_block_scale, const uint8_t* v_block_scale, int64_t num_pages,
                           int layout, const float* k_scale, const float* v_scale, int n_scale,
                           const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                           double softmax_scale, int num_splits, double* out_partial, double* lse_partial);
void orc_paged_decode_nvfp4(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                            const uint8_t* k_cache, const uint8_t* v_cache, const uint8_t* k_block_scale,
                            const uint8_t* v_block_scale, int64_t num_pages, int layout, const float* k_scale,
                            const float* v_scale, int n_scale, const int32_t* block_tables, int max_pages,
                            const int32_t* seq_lens, double softmax_scale, int num_splits,
                            double* out_partial, double* lse_partial);

/* The decodes above with a split count per sequence: sequence b's pages are
 * dealt into splits_per_seq[b] splits (clamped to [1, num_splits]; NULL =
 * num_splits for every sequence); the partial records keep num_splits slots
 * per sequence, and the slots past a sequence's own splits are empty. */
void orc_paged_decode_splits(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                             const void* k_cache, const void* v_cache, int64_t num_pages, int layout,
                             int fp8, const float* k_scale, const float* v_scale, int n_scale,
                             const int32_t* block_tables, int max_pages, const int32_t* seq_lens,
                             double softmax_scale, int num_splits, const int32_t* splits_per_seq,
                             double* out_partial, double* lse_partial);
void orc_paged_decode_nvfp4_splits(int B, int Hq, int Hkv, int D, int page_size, const uint16_t* q,
                                   const uint8_t* k_cache, const uint8_t* v_cache, const uint8_t* k_block_scale,
                                   const uint8_t* v_block_scale, int64_t num_pages, int layout, const float* k_scale,
                                   const float* v_scale, int n_scale, const int32_t* block_tables, int max_pages,
                                   const int32_t* seq_lens, double softmax_scale, int num_splits,
                                   const int32_t* splits_per_seq, double* out_partial, double* lse_partial);

/* MLA (absorbed decode form): latent cache ckv [pages][P][Dc] E4M3 bytes and
 * kpe [pages][P][Dr] bf16 bits; see oracle.c. */
int64_t orc_mla_cache_write(int64_t T, int H, int Dc, int Dr, int page_size, uint16_t* q_pe,
                            const uint16_t* ckv, const uint16_t* kpe, const int32_t* positions,
                            const float* cos_sin, int64_t max_pos, uint8_t* ckv_cache, uint16_t* kpe_cache,
                            int64_t num_pages, int interleaved, float ckv_scale, const int32_t* slot_mapping);
void orc_mla_decode(int B, int H, int Dc, int Dr, int page_size, const uint16_t* q_lat, const uint16_t* q_pe,
                    const uint8_t* ckv_cache, const uint16_t* kpe_cache, int64_t num_pages, float ckv_scale,
                    const int32_t* block_tables, int max_pages, const int32_t* seq_lens, double softmax_scale,
                    int num_splits, double* out_partial, double* lse_partial);
/* orc_mla_decode with a split count per sequence (clamped to [1, num_splits];
 * NULL = num_splits for every sequence); records past it are empty. */
void orc_mla_decode_splits(int B, int H, int Dc, int Dr, int page_size, const uint16_t* q_lat, const uint16_t* q_pe,
                           const uint8_t* ckv_cache, const uint16_t* kpe_cache, int64_t num_pages, float ckv_scale,
                           const int32_t* block_tables, int max_pages, const int32_t* seq_lens, double softmax_scale,
                           int num_splits, const int32_t* splits_per_seq, double* out_partial,
                           double* lse_partial);

/* Merge: out_partial [B,S,Hq,D], lse_partial [B,S,Hq] -> out [B,Hq,D],
 * lse [B,Hq]. */
void orc_lse_merge(int B, int S, int Hq, int D, const double* out_partial,
                   const double* lse_partial, double* out, double* lse);

#ifdef __cplusplus
}
#endif
#endif
