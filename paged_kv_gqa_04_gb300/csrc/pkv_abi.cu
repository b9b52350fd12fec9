// pkv_abi.cu -- the C ABI: argument validation, TMA descriptors, launches.
//
// Loom Kernels, "Architecture": every operator checks the exact contract
// (dtypes, shapes, layouts, aliasing) at the boundary and either accepts it
// or returns an error; there is no fallback path. Nothing here allocates
// device memory or synchronises the host.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <vector>
#include <algorithm>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

using pkv::kPageSize;

namespace {

int elem_bytes(int32_t dtype) {
    switch (dtype) {
        case PKV_BF16: return 2;
        case PKV_FP8_E4M3: return 1;
        case PKV_F32: return 4;
        case PKV_I32: return 4;
        case PKV_FP4_E2M1X2: return 1;
        default: return 0;
    }
}

bool shape_ok(const pkv_tensor& t, int ndim, int32_t dtype) {
    if (t.ndim != ndim || t.dtype != dtype) return false;
    for (int i = 0; i < ndim; ++i)
        if (t.shape[i] < 0) return false;
    return true;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Strides of the given dims, in bytes, multiples of `n`.
bool strides_multiple(const pkv_tensor& t, int upto, int64_t n) {
    const int e = elem_bytes(t.dtype);
    for (int i = 0; i < upto; ++i)
        if ((t.stride[i] * e) % n != 0) return false;
    return true;
}

const pkv_tensor kAbsent{};
// An absent optional tensor may be given as a NULL descriptor pointer.
const pkv_tensor& arg(const pkv_tensor* p) { return p ? *p : kAbsent; }

pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tile map over a cache tensor [pages, a, b, W] (NHD: a = P, b = Hkv; HND:
// a = Hkv, b = P; W = D values, or D/2 bytes of E2M1 pairs). One box = 16
// token rows of one kv head x (128, 64 or 32 bytes of the row), swizzled to
// the same span.
bool make_cache_map(CUtensorMap* m, const pkv_tensor& c, int32_t layout) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int e = elem_bytes(c.dtype);
    const int W = static_cast<int>(c.shape[3]);
    const int row = W * e;
    const int boxb = row >= 128 ? 128 : row;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(c.shape[2]),
                          static_cast<cuuint64_t>(c.shape[1]), static_cast<cuuint64_t>(c.shape[0])};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(c.stride[2] * e), static_cast<cuuint64_t>(c.stride[1] * e),
                             static_cast<cuuint64_t>(c.stride[0] * e)};
    cuuint32_t box[4];
    box[0] = static_cast<cuuint32_t>(boxb / e);
    box[1] = layout == PKV_HND ? kPageSize : 1;
    box[2] = layout == PKV_HND ? 1 : kPageSize;
    box[3] = 1;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle swz = boxb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : (boxb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    CUresult r = enc(m, c.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                     c.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tile map over an MLA cache [pages, P, W] (W = 512 E4M3 bytes of ckv or 64
// bf16 values of kpe): one box = the 64 token rows of a page x 128 bytes,
// 128-byte swizzle.
bool make_mla_map(CUtensorMap* m, const pkv_tensor& c) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int e = elem_bytes(c.dtype);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(c.shape[2]), static_cast<cuuint64_t>(c.shape[1]),
                          static_cast<cuuint64_t>(c.shape[0])};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(c.stride[1] * e), static_cast<cuuint64_t>(c.stride[0] * e)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / e), static_cast<cuuint32_t>(pkv::kMlaPage), 1};  // one page
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, c.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                     c.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An MLA latent cache pair: ckv [pages, P, 512] E4M3, kpe [pages, P, 64]
// bf16; innermost stride 1, other strides multiples of 16 bytes, bases
// 16-byte aligned.
pkv_status check_mla_caches(const pkv_tensor& cc, const pkv_tensor& kc, int64_t* num_pages, int* P) {
    if (!shape_ok(cc, 3, PKV_FP8_E4M3) || !shape_ok(kc, 3, PKV_BF16)) return PKV_ERR_INVALID_ARG;
    if (cc.shape[2] != pkv::kMlaDc || kc.shape[2] != pkv::kMlaDr) return PKV_ERR_UNSUPPORTED;
    if (cc.shape[0] != kc.shape[0] || cc.shape[1] != kc.shape[1]) return PKV_ERR_INVALID_ARG;
    if (!cc.ptr || !kc.ptr) return PKV_ERR_INVALID_ARG;
    *num_pages = cc.shape[0];
    *P = static_cast<int>(cc.shape[1]);
    if (*num_pages < 1 || *P < 1) return PKV_ERR_INVALID_ARG;
    if (cc.stride[2] != 1 || kc.stride[2] != 1) return PKV_ERR_UNSUPPORTED;
    if (!strides_multiple(cc, 2, 16) || !strides_multiple(kc, 2, 16)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(cc.ptr, 16) || !aligned(kc.ptr, 16)) return PKV_ERR_UNSUPPORTED;
    if (*num_pages > 0x7FFFFFFF / 64) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// Common checks of a cache pair. Returns PKV_OK and fills the dims. NVFP4
// value caches (PKV_FP4_E2M1X2) hold D/2 bytes per row; the others D values.
pkv_status check_caches(const pkv_tensor& kc, const pkv_tensor& vc, int32_t layout, int64_t* num_pages,
                        int* P, int* Hkv, int* D, bool nvfp4 = false) {
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (kc.ndim != 4 || vc.ndim != 4 || kc.dtype != vc.dtype) return PKV_ERR_INVALID_ARG;
    if (nvfp4 ? kc.dtype != PKV_FP4_E2M1X2 : (kc.dtype != PKV_BF16 && kc.dtype != PKV_FP8_E4M3))
        return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (kc.shape[i] != vc.shape[i] || kc.shape[i] < 0) return PKV_ERR_INVALID_ARG;
    if (!kc.ptr || !vc.ptr) return PKV_ERR_INVALID_ARG;
    *num_pages = kc.shape[0];
    *P = static_cast<int>(layout == PKV_HND ? kc.shape[2] : kc.shape[1]);
    *Hkv = static_cast<int>(layout == PKV_HND ? kc.shape[1] : kc.shape[2]);
    *D = static_cast<int>(nvfp4 ? 2 * kc.shape[3] : kc.shape[3]);
    if (*num_pages < 1 || *P < 1 || *Hkv < 1) return PKV_ERR_INVALID_ARG;
    if (kc.stride[3] != 1 || vc.stride[3] != 1) return PKV_ERR_UNSUPPORTED;
    if (*D != 64 && *D != 128) return PKV_ERR_UNSUPPORTED;
    if (!strides_multiple(kc, 3, 16) || !strides_multiple(vc, 3, 16)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(kc.ptr, 16) || !aligned(vc.ptr, 16)) return PKV_ERR_UNSUPPORTED;
    if (*num_pages > 0x7FFFFFFF / 16) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

// NVFP4 block-scale caches: E4M3 bytes, the value caches' layout with D/16
// in the last dim, innermost stride 1. With `contiguous` (the decode's bulk
// copies), the P x D/16 bytes of a (page, kv head) are contiguous and start
// on 16-byte boundaries (HND only).
pkv_status check_block_scales(const pkv_tensor& kc, const pkv_tensor& ks, const pkv_tensor& vs, int D,
                              bool contiguous) {
    for (const pkv_tensor* t : {&ks, &vs}) {
        if (!t->ptr || t->ndim != 4 || t->dtype != PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
        for (int i = 0; i < 3; ++i)
            if (t->shape[i] != kc.shape[i]) return PKV_ERR_INVALID_ARG;
        if (t->shape[3] != D / 16) return PKV_ERR_INVALID_ARG;
        if (t->stride[3] != 1) return PKV_ERR_UNSUPPORTED;
        if (contiguous) {
            if (t->stride[2] != D / 16 || !aligned(t->ptr, 16) || !strides_multiple(*t, 2, 16))
                return PKV_ERR_UNSUPPORTED;
        }
    }
    return PKV_OK;
}

pkv_status check_scales(const pkv_tensor& ks, const pkv_tensor& vs, int Hkv, int* n_scale) {
    if (!ks.ptr || !vs.ptr) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(ks, 1, PKV_F32) || !shape_ok(vs, 1, PKV_F32)) return PKV_ERR_INVALID_ARG;
    if (ks.shape[0] != vs.shape[0]) return PKV_ERR_INVALID_ARG;
    if (ks.shape[0] != 1 && ks.shape[0] != Hkv) return PKV_ERR_INVALID_ARG;
    if (ks.stride[0] != 1 || vs.stride[0] != 1) return PKV_ERR_INVALID_ARG;
    *n_scale = static_cast<int>(ks.shape[0]);
    return PKV_OK;
}

// bf16 rows read with 16-byte vectors: innermost stride 1, other strides and
// the base 16-byte aligned.
bool row16(const pkv_tensor& t, int outer) {
    return t.stride[outer] == 1 && aligned(t.ptr, 16) && strides_multiple(t, outer, 16);
}

}  // namespace

namespace pkv {

cudaError_t device_sm_count(int* n) {
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
        const int v = cached[dev].load(std::memory_order_relaxed);
        if (v > 0) {
            *n = v;
            return cudaSuccess;
        }
    }
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cached[dev].store(v, std::memory_order_relaxed);
    *n = v;
    return cudaSuccess;
}

}  // namespace pkv

extern "C" {

int32_t pkv_abi_version(void) { return PKV_ABI_VERSION; }

const char* pkv_status_string(int32_t status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument (shape, stride, dtype or enum)";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration (head dim, group size, page size or alignment)";
        case PKV_ERR_CUDA: return "CUDA launch or driver call failed";
        default: return "unknown status";
    }
}

// The cache write for every cache format; kbs/vbs are the NVFP4 block-scale
// caches (null otherwise).
static pkv_status rope_kv_write_impl(const pkv_tensor* q_p, const pkv_tensor* k_p, const pkv_tensor* v_p,
                                     const pkv_tensor* positions_p, const pkv_tensor* cos_sin_p,
                                     const pkv_tensor* k_cache_p, const pkv_tensor* v_cache_p,
                                     const pkv_tensor* kbs_p, const pkv_tensor* vbs_p,
                                     const pkv_tensor* slot_mapping_p, const pkv_tensor* k_scale_p,
                                     const pkv_tensor* v_scale_p, int32_t layout, int32_t rope_style,
                                     int32_t* err_flag, pkv_stream_t stream, bool nvfp4) {
    const pkv_tensor& q = arg(q_p);
    const pkv_tensor& k = arg(k_p);
    const pkv_tensor& v = arg(v_p);
    const pkv_tensor& positions = arg(positions_p);
    const pkv_tensor& cos_sin = arg(cos_sin_p);
    const pkv_tensor& k_cache = arg(k_cache_p);
    const pkv_tensor& v_cache = arg(v_cache_p);
    const pkv_tensor& slot_mapping = arg(slot_mapping_p);
    const pkv_tensor& k_scale = arg(k_scale_p);
    const pkv_tensor& v_scale = arg(v_scale_p);
    if (rope_style != PKV_ROPE_NEOX && rope_style != PKV_ROPE_INTERLEAVED) return PKV_ERR_INVALID_ARG;
    int64_t num_pages;
    int P, Hkv, D;
    pkv_status st = check_caches(k_cache, v_cache, layout, &num_pages, &P, &Hkv, &D, nvfp4);
    if (st != PKV_OK) return st;
    if (nvfp4) {
        st = check_block_scales(k_cache, arg(kbs_p), arg(vbs_p), D, false);
        if (st != PKV_OK) return st;
    }
    if (!shape_ok(k, 3, PKV_BF16) || !shape_ok(v, 3, PKV_BF16)) return PKV_ERR_INVALID_ARG;
    const int64_t T = k.shape[0];
    if (k.shape[1] != Hkv || k.shape[2] != D || v.shape[0] != T || v.shape[1] != Hkv || v.shape[2] != D)
        return PKV_ERR_INVALID_ARG;
    int Hq = 0;
    if (q.ptr) {
        if (!shape_ok(q, 3, PKV_BF16) || q.shape[0] != T || q.shape[2] != D) return PKV_ERR_INVALID_ARG;
        Hq = static_cast<int>(q.shape[1]);
        if (Hq < 1 || Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    }
    if (!shape_ok(positions, 1, PKV_I32) || !shape_ok(slot_mapping, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
    if (positions.shape[0] != T || slot_mapping.shape[0] != T) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(cos_sin, 2, PKV_F32) || cos_sin.shape[1] != D || cos_sin.shape[0] < 1) return PKV_ERR_INVALID_ARG;
    const int kind = nvfp4 ? pkv::kFp4 : (k_cache.dtype == PKV_FP8_E4M3 ? pkv::kFp8 : pkv::kBf16);
    int n_scale = 0;
    if (kind != pkv::kBf16) {
        st = check_scales(k_scale, v_scale, Hkv, &n_scale);
        if (st != PKV_OK) return st;
    }
    if (T == 0) return PKV_OK;
    if (!k.ptr || !v.ptr || !positions.ptr || !slot_mapping.ptr || !cos_sin.ptr) return PKV_ERR_INVALID_ARG;
    if (positions.stride[0] != 1 || slot_mapping.stride[0] != 1) return PKV_ERR_UNSUPPORTED;
    if (!row16(k, 2) || !row16(v, 2) || (q.ptr && !row16(q, 2))) return PKV_ERR_UNSUPPORTED;
    if (!row16(cos_sin, 1)) return PKV_ERR_UNSUPPORTED;
    if ((Hq + 2 * Hkv) * (D / 16) > 1024) return PKV_ERR_UNSUPPORTED;  // one token's rows per CTA

    pkv::RopeArgs a{};
    a.q = static_cast<uint16_t*>(q.ptr);
    a.q_s0 = q.ptr ? q.stride[0] : 0;
    a.q_s1 = q.ptr ? q.stride[1] : 0;
    a.k = static_cast<const uint16_t*>(k.ptr);
    a.k_s0 = k.stride[0];
    a.k_s1 = k.stride[1];
    a.v = static_cast<const uint16_t*>(v.ptr);
    a.v_s0 = v.stride[0];
    a.v_s1 = v.stride[1];
    a.positions = static_cast<const int32_t*>(positions.ptr);
    a.slots = static_cast<const int32_t*>(slot_mapping.ptr);
    a.cos_sin = static_cast<const float*>(cos_sin.ptr);
    a.cs_s0 = cos_sin.stride[0];
    a.max_pos = cos_sin.shape[0];
    a.k_cache = k_cache.ptr;
    a.v_cache = v_cache.ptr;
    for (int i = 0; i < 4; ++i) {
        a.kc_s[i] = k_cache.stride[i];
        a.vc_s[i] = v_cache.stride[i];
    }
    a.num_pages = num_pages;
    a.page_size = P;
    a.layout = layout;
    a.k_scale = kind != pkv::kBf16 ? static_cast<const float*>(k_scale.ptr) : nullptr;
    a.v_scale = kind != pkv::kBf16 ? static_cast<const float*>(v_scale.ptr) : nullptr;
    a.n_scale = n_scale;
    if (nvfp4) {
        a.k_bs = static_cast<uint8_t*>(arg(kbs_p).ptr);
        a.v_bs = static_cast<uint8_t*>(arg(vbs_p).ptr);
        for (int i = 0; i < 4; ++i) {
            a.kbs_s[i] = arg(kbs_p).stride[i];
            a.vbs_s[i] = arg(vbs_p).stride[i];
        }
    }
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.interleaved = rope_style == PKV_ROPE_INTERLEAVED;
    a.kind = kind;
    a.err = err_flag;
    return cuda_status(pkv::launch_rope_kv_write(a, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_rope_kv_write(const pkv_tensor* q, const pkv_tensor* k, const pkv_tensor* v,
                             const pkv_tensor* positions, const pkv_tensor* cos_sin, const pkv_tensor* k_cache,
                             const pkv_tensor* v_cache, const pkv_tensor* slot_mapping, const pkv_tensor* k_scale,
                             const pkv_tensor* v_scale, int32_t layout, int32_t rope_style, int32_t* err_flag,
                             pkv_stream_t stream) {
    return rope_kv_write_impl(q, k, v, positions, cos_sin, k_cache, v_cache, nullptr, nullptr, slot_mapping,
                              k_scale, v_scale, layout, rope_style, err_flag, stream, false);
}

pkv_status pkv_rope_kv_write_nvfp4(const pkv_tensor* q, const pkv_tensor* k, const pkv_tensor* v,
                                   const pkv_tensor* positions, const pkv_tensor* cos_sin,
                                   const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                   const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                   const pkv_tensor* slot_mapping, const pkv_tensor* k_scale,
                                   const pkv_tensor* v_scale, int32_t layout, int32_t rope_style,
                                   int32_t* err_flag, pkv_stream_t stream) {
    return rope_kv_write_impl(q, k, v, positions, cos_sin, k_cache, v_cache, k_block_scale, v_block_scale,
                              slot_mapping, k_scale, v_scale, layout, rope_style, err_flag, stream, true);
}

// The decode for every cache format; kbs/vbs are the NVFP4 block-scale
// caches (null otherwise).
static pkv_status paged_gqa_decode_impl(const pkv_tensor* q_p, const pkv_tensor* k_cache_p,
                                        const pkv_tensor* v_cache_p, const pkv_tensor* kbs_p,
                                        const pkv_tensor* vbs_p, const pkv_tensor* block_tables_p,
                                        const pkv_tensor* seq_lens_p, float softmax_scale, int32_t num_splits,
                                        const pkv_tensor* out_partial_p, const pkv_tensor* lse_partial_p,
                                        const pkv_tensor* k_scale_p, const pkv_tensor* v_scale_p, int32_t layout,
                                        int32_t* err_flag, pkv_stream_t stream, bool nvfp4,
                                        const pkv_tensor* splits_per_seq_p = nullptr,
                                        const pkv_tensor* work_p = nullptr) {
    const pkv_tensor& q = arg(q_p);
    const pkv_tensor& k_cache = arg(k_cache_p);
    const pkv_tensor& v_cache = arg(v_cache_p);
    const pkv_tensor& block_tables = arg(block_tables_p);
    const pkv_tensor& seq_lens = arg(seq_lens_p);
    const pkv_tensor& out_partial = arg(out_partial_p);
    const pkv_tensor& lse_partial = arg(lse_partial_p);
    const pkv_tensor& k_scale = arg(k_scale_p);
    const pkv_tensor& v_scale = arg(v_scale_p);
    int64_t num_pages;
    int P, Hkv, D;
    pkv_status st = check_caches(k_cache, v_cache, layout, &num_pages, &P, &Hkv, &D, nvfp4);
    if (st != PKV_OK) return st;
    if (nvfp4) {
        st = check_block_scales(k_cache, arg(kbs_p), arg(vbs_p), D, true);
        if (st != PKV_OK) return st;
    }
    if (!shape_ok(q, 3, PKV_BF16) || q.shape[2] != D) return PKV_ERR_INVALID_ARG;
    const int64_t B = q.shape[0];
    const int64_t Hq = q.shape[1];
    if (Hq < 1 || Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (num_splits < 1) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(block_tables, 2, PKV_I32) || block_tables.shape[0] != B) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(seq_lens, 1, PKV_I32) || seq_lens.shape[0] != B) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(out_partial, 4, PKV_F32) || out_partial.shape[0] != B || out_partial.shape[1] != num_splits ||
        out_partial.shape[2] != Hq || out_partial.shape[3] != D)
        return PKV_ERR_INVALID_ARG;
    if (!shape_ok(lse_partial, 3, PKV_F32) || lse_partial.shape[0] != B || lse_partial.shape[1] != num_splits ||
        lse_partial.shape[2] != Hq)
        return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale)) return PKV_ERR_INVALID_ARG;
    const int kind = nvfp4 ? pkv::kFp4 : (k_cache.dtype == PKV_FP8_E4M3 ? pkv::kFp8 : pkv::kBf16);
    int n_scale = 0;
    if (kind != pkv::kBf16) {
        st = check_scales(k_scale, v_scale, Hkv, &n_scale);
        if (st != PKV_OK) return st;
    }
    const int64_t G = Hq / Hkv;
    if (P != kPageSize) return PKV_ERR_UNSUPPORTED;
    if (nvfp4 && layout != PKV_HND) return PKV_ERR_UNSUPPORTED;
    if (G > 16) return PKV_ERR_UNSUPPORTED;
    if (num_splits > 4096 || B > 65535 || Hkv > 65535) return PKV_ERR_UNSUPPORTED;
    if (B == 0) return PKV_OK;
    if (!q.ptr || !block_tables.ptr || !seq_lens.ptr || !out_partial.ptr || !lse_partial.ptr)
        return PKV_ERR_INVALID_ARG;
    const int64_t max_pages = block_tables.shape[1];
    if (max_pages < 1) return PKV_ERR_INVALID_ARG;
    if (max_pages > (int64_t{1} << 26)) return PKV_ERR_UNSUPPORTED;
    if (q.stride[2] != 1 || !aligned(q.ptr, 4) || (q.stride[0] % 2) || (q.stride[1] % 2)) return PKV_ERR_UNSUPPORTED;
    if (block_tables.stride[1] != 1 || seq_lens.stride[0] != 1) return PKV_ERR_UNSUPPORTED;
    if (out_partial.stride[3] != 1 || lse_partial.stride[2] != 1) return PKV_ERR_UNSUPPORTED;

    const bool planned = work_p != nullptr;
    int64_t n_work = 0;
    if (planned) {
        const pkv_tensor& sp = arg(splits_per_seq_p);
        const pkv_tensor& wk = arg(work_p);
        if (!shape_ok(sp, 1, PKV_I32) || sp.shape[0] != B || !sp.ptr) return PKV_ERR_INVALID_ARG;
        if (!shape_ok(wk, 2, PKV_I32) || wk.shape[1] != 2) return PKV_ERR_INVALID_ARG;
        n_work = wk.shape[0];
        if (n_work > 0 && !wk.ptr) return PKV_ERR_INVALID_ARG;
        if (sp.stride[0] != 1 || wk.stride[1] != 1 || wk.stride[0] != 2 || !aligned(wk.ptr, 8))
            return PKV_ERR_UNSUPPORTED;
        if (n_work * Hkv > 0x7FFFFFFF || num_splits > 4095 || B > (1 << 19)) return PKV_ERR_UNSUPPORTED;
    }

    CUtensorMap tk, tv;
    if (!make_cache_map(&tk, k_cache, layout) || !make_cache_map(&tv, v_cache, layout)) return PKV_ERR_CUDA;

    pkv::DecodeArgs a{};
    if (planned) {
        a.splits_per_seq = static_cast<const int32_t*>(arg(splits_per_seq_p).ptr);
        a.work = static_cast<const int32_t*>(arg(work_p).ptr);
        a.n_work = n_work;
    }
    a.q = static_cast<const uint16_t*>(q.ptr);
    a.q_s0 = q.stride[0];
    a.q_s1 = q.stride[1];
    a.block_tables = static_cast<const int32_t*>(block_tables.ptr);
    a.bt_s0 = block_tables.stride[0];
    a.max_pages = static_cast<int32_t>(max_pages);
    a.seq_lens = static_cast<const int32_t*>(seq_lens.ptr);
    a.num_pages = num_pages;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.k_scale = kind != pkv::kBf16 ? static_cast<const float*>(k_scale.ptr) : nullptr;
    a.v_scale = kind != pkv::kBf16 ? static_cast<const float*>(v_scale.ptr) : nullptr;
    a.n_scale = n_scale;
    if (nvfp4) {
        a.k_bs = static_cast<const uint8_t*>(arg(kbs_p).ptr);
        a.v_bs = static_cast<const uint8_t*>(arg(vbs_p).ptr);
        a.kbs_s0 = arg(kbs_p).stride[0];
        a.kbs_s1 = arg(kbs_p).stride[1];
        a.vbs_s0 = arg(vbs_p).stride[0];
        a.vbs_s1 = arg(vbs_p).stride[1];
    }
    a.num_splits = num_splits;
    a.out_partial = static_cast<float*>(out_partial.ptr);
    a.op_s0 = out_partial.stride[0];
    a.op_s1 = out_partial.stride[1];
    a.op_s2 = out_partial.stride[2];
    a.lse_partial = static_cast<float*>(lse_partial.ptr);
    a.lp_s0 = lse_partial.stride[0];
    a.lp_s1 = lse_partial.stride[1];
    a.B = static_cast<int32_t>(B);
    a.Hq = static_cast<int32_t>(Hq);
    a.Hkv = Hkv;
    a.D = D;
    a.G = static_cast<int32_t>(G);
    a.kind = kind;
    a.layout = layout;
    a.err = err_flag;
    return cuda_status(pkv::launch_paged_decode(a, tk, tv, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_gqa_decode(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                const pkv_tensor* block_tables, const pkv_tensor* seq_lens, float softmax_scale,
                                int32_t num_splits, const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                const pkv_tensor* k_scale, const pkv_tensor* v_scale, int32_t layout,
                                int32_t* err_flag, pkv_stream_t stream) {
    return paged_gqa_decode_impl(q, k_cache, v_cache, nullptr, nullptr, block_tables, seq_lens, softmax_scale,
                                 num_splits, out_partial, lse_partial, k_scale, v_scale, layout, err_flag, stream,
                                 false);
}

pkv_status pkv_paged_gqa_decode_nvfp4(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                      const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                      const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                      float softmax_scale, int32_t num_splits, const pkv_tensor* out_partial,
                                      const pkv_tensor* lse_partial, const pkv_tensor* k_scale,
                                      const pkv_tensor* v_scale, int32_t layout, int32_t* err_flag,
                                      pkv_stream_t stream) {
    return paged_gqa_decode_impl(q, k_cache, v_cache, k_block_scale, v_block_scale, block_tables, seq_lens,
                                 softmax_scale, num_splits, out_partial, lse_partial, k_scale, v_scale, layout,
                                 err_flag, stream, true);
}

pkv_status pkv_paged_gqa_decode_planned(const pkv_tensor* q, const pkv_tensor* k_cache, const pkv_tensor* v_cache,
                                        const pkv_tensor* k_block_scale, const pkv_tensor* v_block_scale,
                                        const pkv_tensor* block_tables, const pkv_tensor* seq_lens,
                                        float softmax_scale, const pkv_tensor* splits_per_seq,
                                        const pkv_tensor* work, const pkv_tensor* out_partial,
                                        const pkv_tensor* lse_partial, const pkv_tensor* k_scale,
                                        const pkv_tensor* v_scale, int32_t layout, int32_t* err_flag,
                                        pkv_stream_t stream) {
    if (!splits_per_seq || !work || !out_partial) return PKV_ERR_INVALID_ARG;
    const bool nvfp4 = k_block_scale != nullptr && k_block_scale->ptr != nullptr;
    const pkv_tensor& op = arg(out_partial);
    if (op.ndim != 4) return PKV_ERR_INVALID_ARG;
    if (op.shape[1] < 1 || op.shape[1] > 4095) return op.shape[1] < 1 ? PKV_ERR_INVALID_ARG : PKV_ERR_UNSUPPORTED;
    return paged_gqa_decode_impl(q, k_cache, v_cache, nvfp4 ? k_block_scale : nullptr,
                                 nvfp4 ? v_block_scale : nullptr, block_tables, seq_lens, softmax_scale,
                                 static_cast<int32_t>(op.shape[1]), out_partial, lse_partial, k_scale, v_scale,
                                 layout, err_flag, stream, nvfp4, splits_per_seq, work);
}

static pkv_status lse_merge_impl(const pkv_tensor* out_partial_p, const pkv_tensor* lse_partial_p,
                                 const pkv_tensor* out_p, const pkv_tensor* lse_out_p, pkv_stream_t stream,
                                 const pkv_tensor* splits_per_seq_p) {
    const pkv_tensor& out_partial = arg(out_partial_p);
    const pkv_tensor& lse_partial = arg(lse_partial_p);
    const pkv_tensor& out = arg(out_p);
    const pkv_tensor& lse_out = arg(lse_out_p);
    if (!shape_ok(out_partial, 4, PKV_F32)) return PKV_ERR_INVALID_ARG;
    const int64_t B = out_partial.shape[0], S = out_partial.shape[1], Hq = out_partial.shape[2],
                  D = out_partial.shape[3];
    if (!shape_ok(lse_partial, 3, PKV_F32) || lse_partial.shape[0] != B || lse_partial.shape[1] != S ||
        lse_partial.shape[2] != Hq)
        return PKV_ERR_INVALID_ARG;
    if (!shape_ok(out, 3, PKV_BF16) || out.shape[0] != B || out.shape[1] != Hq || out.shape[2] != D)
        return PKV_ERR_INVALID_ARG;
    if (lse_out.ptr && (!shape_ok(lse_out, 2, PKV_F32) || lse_out.shape[0] != B || lse_out.shape[1] != Hq))
        return PKV_ERR_INVALID_ARG;
    if (S < 1) return PKV_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 512) return PKV_ERR_UNSUPPORTED;
    if (B * Hq == 0) return PKV_OK;
    if (!out_partial.ptr || !lse_partial.ptr || !out.ptr) return PKV_ERR_INVALID_ARG;
    if (out_partial.stride[3] != 1 || lse_partial.stride[2] != 1 || out.stride[2] != 1) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out_partial.ptr, 16) || !strides_multiple(out_partial, 3, 16)) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out.ptr, 8) || !strides_multiple(out, 2, 8)) return PKV_ERR_UNSUPPORTED;
    if (S > 0x7FFFFFFF) return PKV_ERR_UNSUPPORTED;
    const int32_t* spp = nullptr;
    if (splits_per_seq_p) {
        const pkv_tensor& sp = arg(splits_per_seq_p);
        if (!shape_ok(sp, 1, PKV_I32) || sp.shape[0] != B || !sp.ptr) return PKV_ERR_INVALID_ARG;
        if (sp.stride[0] != 1) return PKV_ERR_UNSUPPORTED;
        spp = static_cast<const int32_t*>(sp.ptr);
    }

    pkv::MergeArgs a{};
    a.splits_per_seq = spp;
    a.out_partial = static_cast<const float*>(out_partial.ptr);
    a.op_s0 = out_partial.stride[0];
    a.op_s1 = out_partial.stride[1];
    a.op_s2 = out_partial.stride[2];
    a.lse_partial = static_cast<const float*>(lse_partial.ptr);
    a.lp_s0 = lse_partial.stride[0];
    a.lp_s1 = lse_partial.stride[1];
    a.out = static_cast<uint16_t*>(out.ptr);
    a.o_s0 = out.stride[0];
    a.o_s1 = out.stride[1];
    a.lse_out = static_cast<float*>(lse_out.ptr);
    a.lo_s0 = lse_out.ptr ? lse_out.stride[0] : 0;
    a.lo_s1 = lse_out.ptr ? lse_out.stride[1] : 0;
    a.B = static_cast<int32_t>(B);
    a.S = static_cast<int32_t>(S);
    a.Hq = static_cast<int32_t>(Hq);
    a.D = static_cast<int32_t>(D);
    return cuda_status(pkv::launch_lse_merge(a, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_lse_merge(const pkv_tensor* out_partial, const pkv_tensor* lse_partial, const pkv_tensor* out,
                         const pkv_tensor* lse_out, pkv_stream_t stream) {
    return lse_merge_impl(out_partial, lse_partial, out, lse_out, stream, nullptr);
}

pkv_status pkv_lse_merge_planned(const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                 const pkv_tensor* splits_per_seq, const pkv_tensor* out, const pkv_tensor* lse_out,
                                 pkv_stream_t stream) {
    if (!splits_per_seq) return PKV_ERR_INVALID_ARG;
    return lse_merge_impl(out_partial, lse_partial, out, lse_out, stream, splits_per_seq);
}

pkv_status pkv_mla_cache_write(const pkv_tensor* q_pe_p, const pkv_tensor* ckv_p, const pkv_tensor* kpe_p,
                               const pkv_tensor* positions_p, const pkv_tensor* cos_sin_p,
                               const pkv_tensor* ckv_cache_p, const pkv_tensor* kpe_cache_p,
                               const pkv_tensor* slot_mapping_p, const pkv_tensor* ckv_scale_p, int32_t rope_style,
                               int32_t* err_flag, pkv_stream_t stream) {
    const pkv_tensor& q_pe = arg(q_pe_p);
    const pkv_tensor& ckv = arg(ckv_p);
    const pkv_tensor& kpe = arg(kpe_p);
    const pkv_tensor& positions = arg(positions_p);
    const pkv_tensor& cos_sin = arg(cos_sin_p);
    const pkv_tensor& ckv_cache = arg(ckv_cache_p);
    const pkv_tensor& kpe_cache = arg(kpe_cache_p);
    const pkv_tensor& slot_mapping = arg(slot_mapping_p);
    const pkv_tensor& ckv_scale = arg(ckv_scale_p);
    if (rope_style != PKV_ROPE_NEOX && rope_style != PKV_ROPE_INTERLEAVED) return PKV_ERR_INVALID_ARG;
    int64_t num_pages;
    int P;
    pkv_status st = check_mla_caches(ckv_cache, kpe_cache, &num_pages, &P);
    if (st != PKV_OK) return st;
    if (!shape_ok(ckv, 2, PKV_BF16) || !shape_ok(kpe, 2, PKV_BF16)) return PKV_ERR_INVALID_ARG;
    const int64_t T = ckv.shape[0];
    if (ckv.shape[1] != pkv::kMlaDc || kpe.shape[0] != T || kpe.shape[1] != pkv::kMlaDr) return PKV_ERR_INVALID_ARG;
    int H = 0;
    if (q_pe.ptr) {
        if (!shape_ok(q_pe, 3, PKV_BF16) || q_pe.shape[0] != T || q_pe.shape[2] != pkv::kMlaDr)
            return PKV_ERR_INVALID_ARG;
        if (q_pe.shape[1] < 1) return PKV_ERR_INVALID_ARG;
        if (q_pe.shape[1] > 200) return PKV_ERR_UNSUPPORTED;  // one token's rows per CTA
        H = static_cast<int>(q_pe.shape[1]);
    }
    if (!shape_ok(positions, 1, PKV_I32) || !shape_ok(slot_mapping, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
    if (positions.shape[0] != T || slot_mapping.shape[0] != T) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(cos_sin, 2, PKV_F32) || cos_sin.shape[1] != pkv::kMlaDr || cos_sin.shape[0] < 1)
        return PKV_ERR_INVALID_ARG;
    if (!ckv_scale.ptr || !shape_ok(ckv_scale, 1, PKV_F32) || ckv_scale.shape[0] != 1) return PKV_ERR_INVALID_ARG;
    if (T == 0) return PKV_OK;
    if (!ckv.ptr || !kpe.ptr || !positions.ptr || !slot_mapping.ptr || !cos_sin.ptr) return PKV_ERR_INVALID_ARG;
    if (positions.stride[0] != 1 || slot_mapping.stride[0] != 1) return PKV_ERR_UNSUPPORTED;
    if (!row16(ckv, 1) || !row16(kpe, 1) || (q_pe.ptr && !row16(q_pe, 2)) || !row16(cos_sin, 1))
        return PKV_ERR_UNSUPPORTED;

    pkv::MlaWriteArgs a{};
    a.q_pe = static_cast<uint16_t*>(q_pe.ptr);
    a.qp_s0 = q_pe.ptr ? q_pe.stride[0] : 0;
    a.qp_s1 = q_pe.ptr ? q_pe.stride[1] : 0;
    a.ckv = static_cast<const uint16_t*>(ckv.ptr);
    a.ckv_s0 = ckv.stride[0];
    a.kpe = static_cast<const uint16_t*>(kpe.ptr);
    a.kpe_s0 = kpe.stride[0];
    a.positions = static_cast<const int32_t*>(positions.ptr);
    a.slots = static_cast<const int32_t*>(slot_mapping.ptr);
    a.cos_sin = static_cast<const float*>(cos_sin.ptr);
    a.cs_s0 = cos_sin.stride[0];
    a.max_pos = cos_sin.shape[0];
    a.ckv_cache = static_cast<uint8_t*>(ckv_cache.ptr);
    a.cc_s0 = ckv_cache.stride[0];
    a.cc_s1 = ckv_cache.stride[1];
    a.kpe_cache = static_cast<uint16_t*>(kpe_cache.ptr);
    a.kc_s0 = kpe_cache.stride[0];
    a.kc_s1 = kpe_cache.stride[1];
    a.num_pages = num_pages;
    a.page_size = P;
    a.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == P) a.page_shift = sh;
    a.ckv_scale = static_cast<const float*>(ckv_scale.ptr);
    a.T = T;
    a.H = H;
    a.interleaved = rope_style == PKV_ROPE_INTERLEAVED;
    a.err = err_flag;
    return cuda_status(pkv::launch_mla_cache_write(a, reinterpret_cast<cudaStream_t>(stream)));
}

static pkv_status paged_mla_decode_impl(const pkv_tensor* q_lat_p, const pkv_tensor* q_pe_p,
                                        const pkv_tensor* ckv_cache_p, const pkv_tensor* kpe_cache_p,
                                        const pkv_tensor* block_tables_p, const pkv_tensor* seq_lens_p,
                                        float softmax_scale, int32_t num_splits, const pkv_tensor* out_partial_p,
                                        const pkv_tensor* lse_partial_p, const pkv_tensor* ckv_scale_p,
                                        int32_t* err_flag, pkv_stream_t stream,
                                        const pkv_tensor* splits_per_seq_p = nullptr,
                                        const pkv_tensor* work_p = nullptr) {
    const pkv_tensor& q_lat = arg(q_lat_p);
    const pkv_tensor& q_pe = arg(q_pe_p);
    const pkv_tensor& ckv_cache = arg(ckv_cache_p);
    const pkv_tensor& kpe_cache = arg(kpe_cache_p);
    const pkv_tensor& block_tables = arg(block_tables_p);
    const pkv_tensor& seq_lens = arg(seq_lens_p);
    const pkv_tensor& out_partial = arg(out_partial_p);
    const pkv_tensor& lse_partial = arg(lse_partial_p);
    const pkv_tensor& ckv_scale = arg(ckv_scale_p);
    int64_t num_pages;
    int P;
    pkv_status st = check_mla_caches(ckv_cache, kpe_cache, &num_pages, &P);
    if (st != PKV_OK) return st;
    if (!shape_ok(q_lat, 3, PKV_BF16) || q_lat.shape[2] != pkv::kMlaDc) return PKV_ERR_INVALID_ARG;
    const int64_t B = q_lat.shape[0];
    const int64_t H = q_lat.shape[1];
    if (!shape_ok(q_pe, 3, PKV_BF16) || q_pe.shape[0] != B || q_pe.shape[1] != H || q_pe.shape[2] != pkv::kMlaDr)
        return PKV_ERR_INVALID_ARG;
    if (H < 1 || num_splits < 1) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(block_tables, 2, PKV_I32) || block_tables.shape[0] != B) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(seq_lens, 1, PKV_I32) || seq_lens.shape[0] != B) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(out_partial, 4, PKV_F32) || out_partial.shape[0] != B || out_partial.shape[1] != num_splits ||
        out_partial.shape[2] != H || out_partial.shape[3] != pkv::kMlaDc)
        return PKV_ERR_INVALID_ARG;
    if (!shape_ok(lse_partial, 3, PKV_F32) || lse_partial.shape[0] != B || lse_partial.shape[1] != num_splits ||
        lse_partial.shape[2] != H)
        return PKV_ERR_INVALID_ARG;
    if (!ckv_scale.ptr || !shape_ok(ckv_scale, 1, PKV_F32) || ckv_scale.shape[0] != 1) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale)) return PKV_ERR_INVALID_ARG;
    if (P != pkv::kMlaPage) return PKV_ERR_UNSUPPORTED;
    if (H > 16) return PKV_ERR_UNSUPPORTED;
    if (num_splits > 4096 || B > 65535) return PKV_ERR_UNSUPPORTED;
    if (B == 0) return PKV_OK;
    if (!q_lat.ptr || !q_pe.ptr || !block_tables.ptr || !seq_lens.ptr || !out_partial.ptr || !lse_partial.ptr)
        return PKV_ERR_INVALID_ARG;
    const int64_t max_pages = block_tables.shape[1];
    if (max_pages < 1) return PKV_ERR_INVALID_ARG;
    if (max_pages > (int64_t{1} << 24)) return PKV_ERR_UNSUPPORTED;
    for (const pkv_tensor* q : {&q_lat, &q_pe})
        if (q->stride[2] != 1 || !aligned(q->ptr, 4) || (q->stride[0] % 2) || (q->stride[1] % 2))
            return PKV_ERR_UNSUPPORTED;
    if (block_tables.stride[1] != 1 || seq_lens.stride[0] != 1) return PKV_ERR_UNSUPPORTED;
    if (out_partial.stride[3] != 1 || lse_partial.stride[2] != 1) return PKV_ERR_UNSUPPORTED;
    if (!aligned(out_partial.ptr, 8) || (out_partial.stride[0] % 2) || (out_partial.stride[1] % 2) ||
        (out_partial.stride[2] % 2))
        return PKV_ERR_UNSUPPORTED;

    const bool planned = work_p != nullptr;
    int64_t n_work = 0;
    if (planned) {
        const pkv_tensor& sp = arg(splits_per_seq_p);
        const pkv_tensor& wk = arg(work_p);
        if (!shape_ok(sp, 1, PKV_I32) || sp.shape[0] != B || !sp.ptr) return PKV_ERR_INVALID_ARG;
        if (!shape_ok(wk, 2, PKV_I32) || wk.shape[1] != 2) return PKV_ERR_INVALID_ARG;
        n_work = wk.shape[0];
        if (n_work > 0 && !wk.ptr) return PKV_ERR_INVALID_ARG;
        if (sp.stride[0] != 1 || wk.stride[1] != 1 || wk.stride[0] != 2) return PKV_ERR_UNSUPPORTED;
        if (n_work > 0x7FFFFFFF || num_splits > 4095) return PKV_ERR_UNSUPPORTED;
    }

    CUtensorMap tckv, tkpe;
    if (!make_mla_map(&tckv, ckv_cache) || !make_mla_map(&tkpe, kpe_cache)) return PKV_ERR_CUDA;

    pkv::MlaDecodeArgs a{};
    if (planned) {
        a.splits_per_seq = static_cast<const int32_t*>(arg(splits_per_seq_p).ptr);
        a.work = static_cast<const int32_t*>(arg(work_p).ptr);
        a.n_work = n_work;
    }
    a.q_lat = static_cast<const uint16_t*>(q_lat.ptr);
    a.ql_s0 = q_lat.stride[0];
    a.ql_s1 = q_lat.stride[1];
    a.q_pe = static_cast<const uint16_t*>(q_pe.ptr);
    a.qp_s0 = q_pe.stride[0];
    a.qp_s1 = q_pe.stride[1];
    a.block_tables = static_cast<const int32_t*>(block_tables.ptr);
    a.bt_s0 = block_tables.stride[0];
    a.max_pages = static_cast<int32_t>(max_pages);
    a.seq_lens = static_cast<const int32_t*>(seq_lens.ptr);
    a.num_pages = num_pages;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.ckv_scale = static_cast<const float*>(ckv_scale.ptr);
    a.num_splits = num_splits;
    a.out_partial = static_cast<float*>(out_partial.ptr);
    a.op_s0 = out_partial.stride[0];
    a.op_s1 = out_partial.stride[1];
    a.op_s2 = out_partial.stride[2];
    a.lse_partial = static_cast<float*>(lse_partial.ptr);
    a.lp_s0 = lse_partial.stride[0];
    a.lp_s1 = lse_partial.stride[1];
    a.B = static_cast<int32_t>(B);
    a.H = static_cast<int32_t>(H);
    a.err = err_flag;
    return cuda_status(pkv::launch_mla_decode(a, tckv, tkpe, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_paged_mla_decode(const pkv_tensor* q_lat, const pkv_tensor* q_pe, const pkv_tensor* ckv_cache,
                                const pkv_tensor* kpe_cache, const pkv_tensor* block_tables,
                                const pkv_tensor* seq_lens, float softmax_scale, int32_t num_splits,
                                const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                const pkv_tensor* ckv_scale, int32_t* err_flag, pkv_stream_t stream) {
    return paged_mla_decode_impl(q_lat, q_pe, ckv_cache, kpe_cache, block_tables, seq_lens, softmax_scale,
                                 num_splits, out_partial, lse_partial, ckv_scale, err_flag, stream);
}

pkv_status pkv_paged_mla_decode_planned(const pkv_tensor* q_lat, const pkv_tensor* q_pe, const pkv_tensor* ckv_cache,
                                        const pkv_tensor* kpe_cache, const pkv_tensor* block_tables,
                                        const pkv_tensor* seq_lens, float softmax_scale,
                                        const pkv_tensor* splits_per_seq, const pkv_tensor* work,
                                        const pkv_tensor* out_partial, const pkv_tensor* lse_partial,
                                        const pkv_tensor* ckv_scale, int32_t* err_flag, pkv_stream_t stream) {
    if (!splits_per_seq || !work || !out_partial) return PKV_ERR_INVALID_ARG;
    const pkv_tensor& op = arg(out_partial);
    if (op.ndim != 4 || op.shape[1] < 1) return PKV_ERR_INVALID_ARG;
    if (op.shape[1] > 4095) return PKV_ERR_UNSUPPORTED;
    return paged_mla_decode_impl(q_lat, q_pe, ckv_cache, kpe_cache, block_tables, seq_lens, softmax_scale,
                                 static_cast<int32_t>(op.shape[1]), out_partial, lse_partial, ckv_scale, err_flag,
                                 stream, splits_per_seq, work);
}

int32_t pkv_choose_num_splits_mla(int32_t B, int32_t H, int64_t total_pages, int32_t max_pages, int32_t sm_count) {
    if (B <= 0 || H <= 0 || total_pages <= 0 || max_pages <= 0 || sm_count <= 0) return 1;
    const double sms = static_cast<double>(sm_count);
    const double slots = sms * pkv::mla_decode_ctas_per_sm(H);
    // GB300 constants, measured on the persistent decode: ~3 us per item
    // (query staging, epilogue) and ~2 us per 128-token chunk a CTA streams
    // alone, 60% more when two CTAs share every SM; the latent rows stream
    // at ~5 bytes/ns; 0.1 us per MB of partial records.
    const double e = 3.0, c = 2.0, share = 0.6, bw = 5.0e3;
    const double mx = static_cast<double>(max_pages);
    const double rest = B > 1 ? (static_cast<double>(total_pages) - mx) / (B - 1) : 0.0;  // a mean other sequence
    const double hbm = static_cast<double>(total_pages) * pkv::kMlaPage * (pkv::kMlaDc + 2 * pkv::kMlaDr) / (bw * 1e3);
    // items (splits with pages) and chunks of a sequence of n pages at S
    // splits of ceil(n / S) pages, and the chunks of its largest item
    auto split = [](double n, int S, double* items, double* chunks, double* cmax) {
        *items = *chunks = *cmax = 0.0;
        if (n <= 0.0) return;
        const double pps = std::ceil(n / S);
        const double full = std::floor(n / pps), r = n - full * pps;
        *items = full + (r > 0.0 ? 1.0 : 0.0);
        *chunks = full * std::ceil(pps / 2.0) + std::ceil(r / 2.0);
        *cmax = std::ceil(pps / 2.0);
    };
    int best = 1;
    double best_cost = 1e300;
    for (int S = 1; S <= 1024; ++S) {
        if (S > max_pages) break;
        double i1, c1, cmax, ir, cr, unused;
        split(mx, S, &i1, &c1, &cmax);
        split(rest, S, &ir, &cr, &unused);
        const double items = i1 + (B - 1) * ir, chunks = c1 + (B - 1) * cr;
        const double busy = std::fmin(items, slots);
        const double cc = c * (1.0 + share * std::fmax(0.0, busy - sms) / sms);
        const double stream = (items * e + chunks * cc) / busy;  // a CTA's share of the items
        const double crit = e + cc * cmax;                        // the largest item
        const double merge = 0.1 * 2.0 * B * S * static_cast<double>(H) * (pkv::kMlaDc + 1) * 4.0 / 1e6;
        const double cost = std::fmax(std::fmax(stream, crit), hbm) + merge;
        if (cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = S;
        }
    }
    // More splits that only add empty ones (the same items, the longest
    // split unchanged) up to the CTA slots: measured faster on one 800-page
    // sequence (26.0 us per step at 254 splits against 27.0 at 200, both
    // 200 four-page items), which the model above does not capture.
    auto same_items = [&](int S1, int S2) {
        double a1, b1, m1, a2, b2, m2, r1, q1, u1, r2, q2, u2;
        split(mx, S1, &a1, &b1, &m1);
        split(mx, S2, &a2, &b2, &m2);
        split(rest, S1, &r1, &q1, &u1);
        split(rest, S2, &r2, &q2, &u2);
        return a1 == a2 && b1 == b2 && r1 == r2 && q1 == q2;
    };
    while (best < 1024 && best + 1 <= max_pages && static_cast<double>(B) * (best + 1) <= slots &&
           same_items(best, best + 1))
        ++best;
    return best;
}

int32_t pkv_choose_num_splits(int32_t B, int32_t Hkv, int32_t Hq, int32_t D, int64_t total_pages,
                              int32_t max_pages, int32_t cache_dtype, int32_t sm_count) {
    if (B <= 0 || Hkv <= 0 || Hq <= 0 || D <= 0 || total_pages <= 0 || max_pages <= 0 || sm_count <= 0) return 1;
    const int kind = cache_dtype == PKV_FP4_E2M1X2 ? pkv::kFp4 : (cache_dtype == PKV_FP8_E4M3 ? pkv::kFp8 : pkv::kBf16);
    // bytes of one token row of one head: values (+ NVFP4 block scales)
    const double row = kind == pkv::kFp4 ? D / 2.0 + D / 16.0 : (kind == pkv::kFp8 ? D : 2.0 * D);
    const double page_bytes = 2.0 * kPageSize * row;                // K + V of one page, one kv head
    const double slots = static_cast<double>(sm_count) * pkv::decode_ctas_per_sm(D, kind, (Hq + Hkv - 1) / Hkv);
    // GB300 constants, measured: a CTA spends ~3 us on start-up and its
    // epilogue and streams a page in ~0.28 us per 8 KB (bf16) or ~0.55 us per
    // 8 KB of its bytes (FP8 / NVFP4: bound by instruction issue); HBM moves
    // ~7 bytes per ns.
    const double t0 = 3.0;
    const double tp = (kind == pkv::kBf16 ? 0.278 : 0.55) * page_bytes / 8192.0;
    const double bw = 7.0e3;  // bytes per ns (x 1e3 per us below)
    const double units = static_cast<double>(B) * Hkv;
    const double mean_pages = static_cast<double>(total_pages) / B;
    const double stream0 = static_cast<double>(Hkv) * static_cast<double>(total_pages) * page_bytes / (bw * 1e3);
    int best = 1;
    double best_cost = 1e300;
    for (int S = 1; S <= 1024; ++S) {
        if (S > max_pages) break;
        const double ncta = units * S;
        const bool waves = ncta > slots;
        const double t_mean = t0 + tp * mean_pages / S;                                // a mean CTA
        const double t_max = t0 + tp * std::ceil(static_cast<double>(max_pages) / S);  // the longest split
        // HBM time plus the CTAs' start-up where it does not overlap other
        // CTAs' streaming, plus, past one wave, part of the longest split's
        // excess (it may be dispatched last) ...
        const double stream = stream0 + 0.25 * ncta * t0 / slots + (waves ? 0.5 * (t_max - t_mean) : 0.0);
        // ... or the longest split itself (after a mean CTA's wait for a slot)
        const double crit = t_max + (waves ? t_mean : 0.0);
        // partial records written by the decode and read by the merge, and
        // past 32 splits the merge's two-level tree (measured ~2 us more
        // per step than its one-warp-per-row form)
        const double merge = 0.15 * 2.0 * B * S * static_cast<double>(Hq) * (D + 1) * 4.0 / 1e6 + (S > 32 ? 2.0 : 0.0);
        const double cost = std::fmax(stream, crit) + merge;
        if (cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = S;
        }
    }
    return best;
}

namespace {

// The split count of a sequence of n pages under a target of T pages per
// split, at most max_splits, reduced to the splits that hold pages when that
// keeps the same page ranges.
// Page counts and targets stay below 2^26 (the block-table width limit), so
// the arithmetic is done in 32 bits. The count does not grow with T.
int64_t plan_count(int64_t n64, int64_t T64, int max_splits) {
    if (n64 <= 0) return 1;
    const int32_t n = static_cast<int32_t>(n64), T = static_cast<int32_t>(std::min<int64_t>(T64, n64));
    const int32_t S = std::min<int32_t>((n + T - 1) / T, max_splits);
    const int32_t pps = (n + S - 1) / S;
    const int32_t k = (n + pps - 1) / pps;
    return ((n + k - 1) / k == pps) ? k : S;
}

// Pages of each sequence (seq_lens clamped to [0, page * max_pages]).
std::vector<int64_t> plan_pages(const int32_t* seq_lens, int32_t B, int64_t page, int32_t max_pages, int64_t* max_np,
                                int64_t* total) {
    std::vector<int64_t> np(B);
    *max_np = 0;
    *total = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t L = std::min<int64_t>(std::max<int32_t>(seq_lens[b], 0), page * max_pages);
        np[b] = (L + page - 1) / page;
        *max_np = std::max(*max_np, np[b]);
        *total += np[b];
    }
    return np;
}

// The plan's outputs for a page target T: split counts, record count and
// the work list, items in order of decreasing page count (ties by sequence
// then split).
pkv_status plan_emit(const std::vector<int64_t>& np, int64_t T, int max_splits, int32_t* splits_per_seq,
                     int32_t* num_records, int32_t* work, int64_t work_capacity, int64_t* num_work) {
    const int B = static_cast<int>(np.size());
    int64_t n_items = 0;
    int32_t recs = 1;
    for (int b = 0; b < B; ++b) {
        const int64_t S = plan_count(np[b], T, max_splits);
        splits_per_seq[b] = static_cast<int32_t>(S);
        recs = std::max<int32_t>(recs, static_cast<int32_t>(S));
        n_items += S;
    }
    *num_records = recs;
    *num_work = n_items;
    if (!work) return PKV_OK;
    if (work_capacity < n_items) return PKV_ERR_INVALID_ARG;
    struct It { int64_t pages; int32_t b, s, p0; };
    std::vector<It> items;
    items.reserve(static_cast<size_t>(n_items));
    for (int b = 0; b < B; ++b) {
        const int64_t S = splits_per_seq[b];
        const int64_t pps = np[b] > 0 ? (np[b] + S - 1) / S : 0;
        for (int64_t sp = 0; sp < S; ++sp) {
            const int64_t p0 = std::min(sp * pps, np[b]);
            items.push_back({std::min(pps, np[b] - p0), b, static_cast<int32_t>(sp), static_cast<int32_t>(p0)});
        }
    }
    std::stable_sort(items.begin(), items.end(), [](const It& x, const It& y) { return x.pages > y.pages; });
    for (int64_t i = 0; i < n_items; ++i) {
        work[2 * i] = (items[i].b << 12) | items[i].s;
        work[2 * i + 1] = items[i].p0;
    }
    return PKV_OK;
}

pkv_status plan_check(const int32_t* seq_lens, int32_t B, int32_t max_pages, int32_t sm_count, int32_t max_splits,
                      int32_t target_pages, const int32_t* splits_per_seq, const int32_t* num_records,
                      const int32_t* work, int64_t work_capacity, const int64_t* num_work) {
    if (B < 0 || max_pages < 1 || sm_count < 1) return PKV_ERR_INVALID_ARG;
    if (max_splits < 1 || max_splits > 4095 || target_pages < 0 || work_capacity < 0) return PKV_ERR_INVALID_ARG;
    if (B > (1 << 19) || max_pages > (1 << 26)) return PKV_ERR_UNSUPPORTED;
    if ((B > 0 && (!seq_lens || !splits_per_seq)) || !num_records || !num_work) return PKV_ERR_INVALID_ARG;
    if (work_capacity > 0 && !work) return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

}  // namespace

// The split plan: a split count per sequence so that every CTA streams
// about the same number of pages, and the work list of (sequence, split)
// items, longest first. Host only; no CUDA call.
pkv_status pkv_plan_splits(const int32_t* seq_lens, int32_t B, int32_t Hkv, int32_t Hq, int32_t D,
                           int32_t max_pages, int32_t cache_dtype, int32_t sm_count, int32_t max_splits,
                           int32_t target_pages, int32_t* splits_per_seq, int32_t* num_records, int32_t* work,
                           int64_t work_capacity, int64_t* num_work) {
    if (Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || D < 1) return PKV_ERR_INVALID_ARG;
    pkv_status st = plan_check(seq_lens, B, max_pages, sm_count, max_splits, target_pages, splits_per_seq,
                               num_records, work, work_capacity, num_work);
    if (st != PKV_OK) return st;
    int64_t max_np = 0, total = 0;
    const std::vector<int64_t> np = plan_pages(seq_lens, B, kPageSize, max_pages, &max_np, &total);
    int64_t T = target_pages;
    if (T == 0) {
        // When every sequence and kv head can have a CTA of its own within
        // one wave, the plan fills that wave with items of nearly equal
        // length, chosen with a model of the decode on GB300 (fitted to sweeps
        // of the page target on the qwen, longctx, fp8 and fp4 workloads): a
        // CTA spends ~3 us on start-up and its epilogue, then streams its
        // page-heads at its share of HBM (~7 bytes/ns over the CTAs running
        // at once), at most at the ~30 bytes/ns one CTA keeps in flight, or,
        // for FP8 / NVFP4, at the ~0.36 us per page-head its dequantisation
        // takes when that is slower; the step ends with the longest item.
        // Past one wave (many short sequences) the uniform heuristic's
        // longest split is the target: measured on the ragged workload, no
        // other target did better by more than the run-to-run spread.
        const int kind = cache_dtype == PKV_FP4_E2M1X2 ? pkv::kFp4 : (cache_dtype == PKV_FP8_E4M3 ? pkv::kFp8 : pkv::kBf16);
        const double row = kind == pkv::kFp4 ? D / 2.0 + D / 16.0 : (kind == pkv::kFp8 ? D : 2.0 * D);
        const double page_bytes = 2.0 * kPageSize * row;
        const double slots = static_cast<double>(sm_count) * pkv::decode_ctas_per_sm(D, kind, Hq / Hkv);
        const double t0 = 3.0, bw = 7.0e6, bw_cta = 2.95e4;  // us; bytes per us
        const double tc = std::max(kind == pkv::kBf16 ? 0.0 : 0.36, page_bytes / bw_cta);
        const int64_t top = std::max<int64_t>(max_np, 1);
        if (static_cast<double>(B) * Hkv > slots) {
            const int32_t S_u = pkv_choose_num_splits(B, Hkv, Hq, D, std::max<int64_t>(total, 1),
                                                      static_cast<int32_t>(top), cache_dtype, sm_count);
            T = (top + S_u - 1) / S_u;
        } else {
            // The targets whose CTAs exceed one wave are skipped: the item
            // count does not grow with the target, so the smallest target that
            // fits is found by bisection and the search starts there.
            const int64_t cap = static_cast<int64_t>(slots) / Hkv;
            auto fits = [&](int64_t Tc) {
                int64_t it = 0;
                for (int b = 0; b < B && it <= cap; ++b) it += plan_count(np[b], Tc, max_splits);
                return it <= cap;
            };
            int64_t lo = 0, hi = top;  // fits(top): B items, and B * Hkv <= slots here
            while (hi - lo > 1) {
                const int64_t mid = lo + (hi - lo) / 2;
                if (fits(mid))
                    hi = mid;
                else
                    lo = mid;
            }
            const int64_t T_fit = hi;
            double best_cost = 1e300;
            int64_t best_T = top;
            for (int64_t Tc = 1; Tc <= top; Tc = Tc < 64 ? Tc + 1 : std::max<int64_t>(Tc + 1, static_cast<int64_t>(Tc * 1.05))) {
                if (Tc < T_fit) continue;
                double items = 0, p_max = 0;
                int64_t recs = 1;
                for (int b = 0; b < B; ++b) {
                    const int64_t S = plan_count(np[b], Tc, max_splits);
                    items += static_cast<double>(S);
                    p_max = std::max(p_max, static_cast<double>(np[b] > 0 ? (np[b] + S - 1) / S : 0));
                    recs = std::max(recs, S);
                }
                const double n = items * Hkv;  // CTAs
                if (n > slots) continue;
                const double cost = t0 + p_max * std::max(page_bytes * n / bw, tc) +
                                    0.15 * 2.0 * items * static_cast<double>(Hq) * (D + 1) * 4.0 / 1e6 +
                                    (recs > 32 ? 2.0 : 0.0);
                if (cost < best_cost * (1.0 - 1e-9)) {
                    best_cost = cost;
                    best_T = Tc;
                }
            }
            T = best_T;
        }
    }
    return plan_emit(np, T, max_splits, splits_per_seq, num_records, work, work_capacity, num_work);
}

// The split plan of the MLA decode: persistent CTAs (two per SM) take the
// items in the plan's order. When every sequence can have a CTA of its own,
// the plan makes at most one item per CTA, of nearly equal length: the
// smallest page target (whole 128-token chunks: an even page count) whose
// items fit the CTAs; else the uniform heuristic's longest split. Host only.
pkv_status pkv_plan_splits_mla(const int32_t* seq_lens, int32_t B, int32_t H, int32_t max_pages, int32_t sm_count,
                               int32_t max_splits, int32_t target_pages, int32_t* splits_per_seq,
                               int32_t* num_records, int32_t* work, int64_t work_capacity, int64_t* num_work) {
    if (H < 1) return PKV_ERR_INVALID_ARG;
    pkv_status st = plan_check(seq_lens, B, max_pages, sm_count, max_splits, target_pages, splits_per_seq,
                               num_records, work, work_capacity, num_work);
    if (st != PKV_OK) return st;
    int64_t max_np = 0, total = 0;
    const std::vector<int64_t> np = plan_pages(seq_lens, B, pkv::kMlaPage, max_pages, &max_np, &total);
    int64_t T = target_pages;
    if (T == 0) {
        const int64_t ctas = static_cast<int64_t>(sm_count) * pkv::mla_decode_ctas_per_sm(H);
        const int64_t top = std::max<int64_t>(max_np, 1);
        if (static_cast<int64_t>(B) > ctas) {
            const int32_t S_u = pkv_choose_num_splits_mla(B, H, std::max<int64_t>(total, 1), static_cast<int32_t>(top),
                                                          sm_count);
            T = (top + S_u - 1) / S_u;
        } else {
            // The item count does not grow with the target: bisect over the
            // even targets below the longest sequence (T = top gives B items).
            auto fits = [&](int64_t Tc) {
                int64_t items = 0;
                for (int b = 0; b < B && items <= ctas; ++b) items += plan_count(np[b], Tc, max_splits);
                return items <= ctas;
            };
            int64_t lo = 1, hi = (top + 1) / 2;  // even targets 2 lo .. 2 hi; 2 hi >= top fits
            if (fits(2)) hi = 1;
            while (hi - lo > 1) {  // fits(2 hi) holds, fits(2 lo) does not
                const int64_t mid = lo + (hi - lo) / 2;
                if (fits(2 * mid))
                    hi = mid;
                else
                    lo = mid;
            }
            T = std::min<int64_t>(2 * hi, top);
        }
    }
    return plan_emit(np, T, max_splits, splits_per_seq, num_records, work, work_capacity, num_work);
}

pkv_status pkv_validate_indices(const pkv_tensor* block_tables_p, const pkv_tensor* seq_lens_p, const pkv_tensor* slot_mapping_p,
                                int64_t num_pages, const pkv_tensor* slot_bitmap_p, int32_t* err_flag, pkv_stream_t stream) {
    const pkv_tensor& block_tables = arg(block_tables_p);
    const pkv_tensor& seq_lens = arg(seq_lens_p);
    const pkv_tensor& slot_mapping = arg(slot_mapping_p);
    const pkv_tensor& slot_bitmap = arg(slot_bitmap_p);
    if (!err_flag) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(block_tables, 2, PKV_I32) || !shape_ok(seq_lens, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
    if (seq_lens.shape[0] != block_tables.shape[0]) return PKV_ERR_INVALID_ARG;
    if (num_pages < 0) return PKV_ERR_INVALID_ARG;
    if (num_pages > 0x7FFFFFFF / kPageSize) return PKV_ERR_UNSUPPORTED;
    pkv::ValidateArgs a{};
    if (slot_mapping.ptr) {
        if (!shape_ok(slot_mapping, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
        a.slots = static_cast<const int32_t*>(slot_mapping.ptr);
        a.sm_s0 = slot_mapping.stride[0];
        a.T = slot_mapping.shape[0];
    }
    if (slot_bitmap.ptr) {
        if (!shape_ok(slot_bitmap, 1, PKV_I32) || slot_bitmap.stride[0] != 1) return PKV_ERR_INVALID_ARG;
        const int64_t words = (num_pages * kPageSize + 31) / 32;
        if (slot_bitmap.shape[0] < words) return PKV_ERR_INVALID_ARG;
        a.bitmap = static_cast<uint32_t*>(slot_bitmap.ptr);
        a.bitmap_words = words;
    }
    if (block_tables.shape[0] > 0x7FFFFFFF / 32 || block_tables.shape[1] > (int64_t{1} << 26))
        return PKV_ERR_UNSUPPORTED;
    if (block_tables.shape[0] > 0 && (!block_tables.ptr || !seq_lens.ptr)) return PKV_ERR_INVALID_ARG;
    a.block_tables = static_cast<const int32_t*>(block_tables.ptr);
    a.bt_s0 = block_tables.stride[0];
    a.bt_s1 = block_tables.stride[1];
    a.max_pages = static_cast<int32_t>(block_tables.shape[1]);
    a.seq_lens = static_cast<const int32_t*>(seq_lens.ptr);
    a.sl_s0 = seq_lens.stride[0];
    a.B = static_cast<int32_t>(block_tables.shape[0]);
    a.num_pages = num_pages;
    a.err = err_flag;
    return cuda_status(pkv::launch_validate(a, reinterpret_cast<cudaStream_t>(stream)));
}

// Same checks as pkv_validate_indices; the bitmap is the library's static
// device array instead of a caller buffer, so nothing is allocated.
pkv_status pkv_validate_indices_static(const pkv_tensor* block_tables_p, const pkv_tensor* seq_lens_p,
                                       const pkv_tensor* slot_mapping_p, int64_t num_pages, int32_t* err_flag,
                                       pkv_stream_t stream) {
    const pkv_tensor& block_tables = arg(block_tables_p);
    const pkv_tensor& seq_lens = arg(seq_lens_p);
    const pkv_tensor& slot_mapping = arg(slot_mapping_p);
    if (!err_flag) return PKV_ERR_INVALID_ARG;
    if (!shape_ok(block_tables, 2, PKV_I32) || !shape_ok(seq_lens, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
    if (seq_lens.shape[0] != block_tables.shape[0]) return PKV_ERR_INVALID_ARG;
    if (num_pages < 0) return PKV_ERR_INVALID_ARG;
    // compared before any product, so no num_pages can overflow the check
    if (num_pages > PKV_STATIC_VALIDATE_MAX_SLOTS / kPageSize) return PKV_ERR_UNSUPPORTED;
    pkv::ValidateArgs a{};
    if (slot_mapping.ptr) {
        if (!shape_ok(slot_mapping, 1, PKV_I32)) return PKV_ERR_INVALID_ARG;
        a.slots = static_cast<const int32_t*>(slot_mapping.ptr);
        a.sm_s0 = slot_mapping.stride[0];
        a.T = slot_mapping.shape[0];
    }
    if (block_tables.shape[0] > 0x7FFFFFFF / 32 || block_tables.shape[1] > (int64_t{1} << 26))
        return PKV_ERR_UNSUPPORTED;
    if (block_tables.shape[0] > 0 && (!block_tables.ptr || !seq_lens.ptr)) return PKV_ERR_INVALID_ARG;
    uint32_t* bitmap = nullptr;
    int64_t words = 0;
    cudaError_t e = pkv::static_slot_bitmap(&bitmap, &words);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    a.bitmap = bitmap;
    a.bitmap_words = (num_pages * kPageSize + 31) / 32;  // only the part this call uses is cleared
    a.block_tables = static_cast<const int32_t*>(block_tables.ptr);
    a.bt_s0 = block_tables.stride[0];
    a.bt_s1 = block_tables.stride[1];
    a.max_pages = static_cast<int32_t>(block_tables.shape[1]);
    a.seq_lens = static_cast<const int32_t*>(seq_lens.ptr);
    a.sl_s0 = seq_lens.stride[0];
    a.B = static_cast<int32_t>(block_tables.shape[0]);
    a.num_pages = num_pages;
    a.err = err_flag;
    return cuda_status(pkv::launch_validate(a, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_selftest_bounded_wait(int64_t limit_ns, int32_t* err_flag, uint64_t* elapsed_ns,
                                     pkv_stream_t stream) {
    if (limit_ns < 100000 || limit_ns > 10000000 || !err_flag || !elapsed_ns) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_selftest_wait(static_cast<uint64_t>(limit_ns), err_flag, elapsed_ns,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

// A pointer the SMs of the current device can address: its own device
// memory, managed memory, or host memory page-locked by CUDA and mapped at
// the same address (unified addressing). Another GPU's memory is refused
// (it would need peer access).
static bool device_accessible(const void* p) {
    cudaPointerAttributes at{};
    int cur = -1;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess || cudaGetDevice(&cur) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
            return at.device == cur;
        case cudaMemoryTypeManaged:
            return true;
        case cudaMemoryTypeHost:
            return at.devicePointer == p;
        default:
            return false;
    }
}

pkv_status pkv_copy(void* dst, const void* src, int64_t bytes, pkv_stream_t stream) {
    if (bytes < 0) return PKV_ERR_INVALID_ARG;
    if (bytes == 0) return PKV_OK;
    if (!dst || !src) return PKV_ERR_INVALID_ARG;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + static_cast<uintptr_t>(bytes) && s < d + static_cast<uintptr_t>(bytes)) return PKV_ERR_INVALID_ARG;
    if (!device_accessible(dst) || !device_accessible(src)) return PKV_ERR_UNSUPPORTED;
    return cuda_status(pkv::launch_copy(dst, src, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status pkv_stream_read(const void* buf, int64_t bytes, uint32_t* sink, int32_t ctas, pkv_stream_t stream) {
    if (bytes < 0 || bytes % 16 != 0 || ctas < 1 || ctas > 65535) return PKV_ERR_INVALID_ARG;
    if (bytes == 0) return PKV_OK;
    if (!buf || !sink || !aligned(buf, 16)) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_stream_read(buf, bytes, sink, ctas, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
