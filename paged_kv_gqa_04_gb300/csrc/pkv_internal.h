// pkv_internal.h -- argument blocks passed from the C-ABI layer (pkv_abi.cu)
// to the kernel launchers. Host and device code both include this header.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPageSize = 16;  // tokens per page for the decode kernel

// Cache formats: bf16 values, static-scale E4M3 bytes, or NVFP4 (packed
// E2M1 pairs + one E4M3 block-scale byte per 16 values + a static scale).
enum CacheKind : int { kBf16 = 0, kFp8 = 1, kFp4 = 2 };

struct RopeArgs {
    uint16_t* q;               // bf16 bits, may be null
    int64_t q_s0, q_s1;        // element strides (token, head)
    const uint16_t* k;
    int64_t k_s0, k_s1;
    const uint16_t* v;
    int64_t v_s0, v_s1;
    const int32_t* positions;
    const int32_t* slots;
    const float* cos_sin;
    int64_t cs_s0;             // row stride (elements)
    int64_t max_pos;
    void* k_cache;
    void* v_cache;
    int64_t kc_s[4];           // element strides of the 4 cache dims, tensor order
    int64_t vc_s[4];
    int64_t num_pages;
    int32_t page_size;
    int32_t layout;            // pkv_layout
    const float* k_scale;      // fp8 / nvfp4 only
    const float* v_scale;
    int32_t n_scale;           // 1 or Hkv
    uint8_t* k_bs;             // nvfp4 block scales (E4M3 bytes), else null
    uint8_t* v_bs;
    int64_t kbs_s[4];          // byte strides of the 4 block-scale dims, tensor order
    int64_t vbs_s[4];
    int64_t T;
    int32_t Hq;                // 0 when q is null
    int32_t Hkv;
    int32_t D;
    int32_t interleaved;
    int32_t kind;              // CacheKind
    int32_t toks;              // tokens per group of a CTA (set by the launcher)
    int32_t* err;
};

struct DecodeArgs {
    const uint16_t* q;         // [B, Hq, D] bf16 bits
    int64_t q_s0, q_s1;
    const int32_t* block_tables;
    int64_t bt_s0;
    int32_t max_pages;
    const int32_t* seq_lens;
    int64_t num_pages;
    float scale_log2;          // softmax_scale * log2(e)
    const float* k_scale;      // fp8 / nvfp4 only
    const float* v_scale;
    int32_t n_scale;
    const uint8_t* k_bs;       // nvfp4 block scales: the P x D/16 bytes of
    const uint8_t* v_bs;       // (page, kv head) start at page*s0 + kvh*s1
    int64_t kbs_s0, kbs_s1;    // (bytes)
    int64_t vbs_s0, vbs_s1;
    int32_t num_splits;
    float* out_partial;
    int64_t op_s0, op_s1, op_s2;
    float* lse_partial;
    int64_t lp_s0, lp_s1;
    int32_t B, Hq, Hkv, D, G;
    int32_t kind;              // CacheKind
    int32_t layout;            // pkv_layout (selects the TMA coordinate order)
    // Planned launches (a split count per sequence): work[2 i] = (b << 12) | s,
    // work[2 i + 1] = the split's first page per the plan (a hint for the
    // early block-table read); splits_per_seq[b] = the sequence's split count.
    // Both null for a uniform launch (every sequence in num_splits splits).
    const int32_t* work;
    int64_t n_work;
    const int32_t* splits_per_seq;
    int32_t* err;
};

// Multi-head latent attention (absorbed decode form): every query head
// attends to the same latent cache rows.
constexpr int kMlaDc = 512;        // latent (ckv) values per token, E4M3 bytes
constexpr int kMlaDr = 64;         // positional (kpe) values per token, bf16
constexpr int kMlaPage = 64;       // tokens per page of the latent cache

struct MlaDecodeArgs {
    const uint16_t* q_lat;     // [B, H, 512] bf16 bits
    int64_t ql_s0, ql_s1;
    const uint16_t* q_pe;      // [B, H, 64] bf16 bits (rotated)
    int64_t qp_s0, qp_s1;
    const int32_t* block_tables;
    int64_t bt_s0;
    int32_t max_pages;
    const int32_t* seq_lens;
    int64_t num_pages;
    float scale_log2;          // softmax_scale * log2(e)
    const float* ckv_scale;    // [1]
    int32_t num_splits;
    float* out_partial;        // [B, S, H, 512]
    int64_t op_s0, op_s1, op_s2;
    float* lse_partial;        // [B, S, H]
    int64_t lp_s0, lp_s1;
    int32_t B, H;
    // A split plan (both null: every sequence in num_splits splits): item i
    // = work[2 i] = (b << 12) | s in the plan's order, splits_per_seq[b] the
    // sequence's split count.
    const int32_t* work;
    int64_t n_work;
    const int32_t* splits_per_seq;
    int32_t* err;
};

struct MlaWriteArgs {
    uint16_t* q_pe;            // [T, H, 64] bf16 bits, rotated in place; may be null
    int64_t qp_s0, qp_s1;
    const uint16_t* ckv;       // [T, 512]
    int64_t ckv_s0;
    const uint16_t* kpe;       // [T, 64]
    int64_t kpe_s0;
    const int32_t* positions;
    const int32_t* slots;
    const float* cos_sin;      // [max_pos, 64]
    int64_t cs_s0;
    int64_t max_pos;
    uint8_t* ckv_cache;        // [pages, P, 512] E4M3 bytes
    int64_t cc_s0, cc_s1;
    uint16_t* kpe_cache;       // [pages, P, 64] bf16 bits
    int64_t kc_s0, kc_s1;
    int64_t num_pages;
    int32_t page_size;
    int32_t page_shift;        // log2(page_size) when it is a power of two, else -1
    const float* ckv_scale;    // [1]
    int64_t T;
    int32_t H;                 // 0 when q_pe is null
    int32_t interleaved;
    int32_t* err;
};

struct MergeArgs {
    const float* out_partial;
    int64_t op_s0, op_s1, op_s2;
    const float* lse_partial;
    int64_t lp_s0, lp_s1;
    uint16_t* out;             // bf16 bits
    int64_t o_s0, o_s1;
    float* lse_out;            // may be null
    int64_t lo_s0, lo_s1;
    int32_t B, S, Hq, D;
    const int32_t* splits_per_seq;  // records merged per sequence (clamped to [1, S]); null = S
};

struct ValidateArgs {
    const int32_t* block_tables;
    int64_t bt_s0, bt_s1;
    int32_t max_pages;
    const int32_t* seq_lens;
    int64_t sl_s0;
    int32_t B;
    const int32_t* slots;      // may be null
    int64_t sm_s0;
    int64_t T;
    int64_t num_pages;
    uint32_t* bitmap;          // may be null
    int64_t bitmap_words;
    int32_t* err;
};

// Launch as a programmatic dependent of the preceding work in the stream:
// the kernel may start while the preceding kernel finishes, and orders its
// reads and writes of data that kernel touches after griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

cudaError_t launch_rope_kv_write(const RopeArgs& a, cudaStream_t s);
cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                cudaStream_t s);
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s);
cudaError_t launch_mla_decode(const MlaDecodeArgs& a, const CUtensorMap& tckv, const CUtensorMap& tkpe,
                              cudaStream_t s);
cudaError_t launch_mla_cache_write(const MlaWriteArgs& a, cudaStream_t s);
int mla_decode_ctas_per_sm(int H);
// Number of SMs of the current device (cached per device).
cudaError_t device_sm_count(int* n);
cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s);
cudaError_t static_slot_bitmap(uint32_t** ptr, int64_t* words);
cudaError_t launch_stream_read(const void* buf, int64_t bytes, uint32_t* sink, int ctas, cudaStream_t s);
cudaError_t launch_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s);
cudaError_t launch_selftest_wait(uint64_t limit_ns, int32_t* err, uint64_t* elapsed_ns, cudaStream_t s);

// Occupancy-related constants of the decode kernel, shared with the split
// heuristic on the host.
int decode_ctas_per_sm(int D, int kind, int G);

}  // namespace pkv
