"""Thin ctypes binding of the C ABI in include/pkv.h (libpkv.so).

Argument marshalling only: each function turns torch tensors into pkv_tensor
descriptors (pointer, dtype, shape, strides) and calls the library on the
current CUDA stream. Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU implementation behind these names, and a
missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA = 0, 1, 2, 3
LAYOUTS = {"NHD": 0, "HND": 1}
STYLES = {"neox": 0, "interleaved": 1}
FLAG_SLOT_RANGE = 0x01
FLAG_POSITION_RANGE = 0x02
FLAG_PAGE_RANGE = 0x04
FLAG_SEQ_LEN_RANGE = 0x08
FLAG_DUPLICATE_SLOT = 0x10
FLAG_WAIT_TIMEOUT = 0x20
FLAG_PLAN_RANGE = 0x40

_DTYPES = {
    torch.bfloat16: 0,
    torch.float8_e4m3fn: 1,
    torch.uint8: 1,
    torch.float32: 2,
    torch.int32: 3,
}
PKV_FP4_E2M1X2 = 4    # uint8 bytes of two E2M1 values (NVFP4 value caches)
_CACHE_DTYPE = {"bf16": 0, "fp8": 1, "nvfp4": PKV_FP4_E2M1X2}

EXPORTED = ("pkv_rope_kv_write", "pkv_paged_gqa_decode", "pkv_lse_merge", "pkv_choose_num_splits",
            "pkv_validate_indices", "pkv_status_string", "pkv_abi_version", "pkv_stream_read",
            "pkv_validate_indices_static", "pkv_rope_kv_write_nvfp4", "pkv_paged_gqa_decode_nvfp4",
            "pkv_mla_cache_write", "pkv_paged_mla_decode", "pkv_choose_num_splits_mla",
            "pkv_selftest_bounded_wait", "pkv_copy", "pkv_plan_splits", "pkv_paged_gqa_decode_planned",
            "pkv_lse_merge_planned", "pkv_plan_splits_mla", "pkv_paged_mla_decode_planned")


class PkvTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        T = ctypes.POINTER(PkvTensor)
        P = ctypes.c_void_p
        i32 = ctypes.c_int32
        L.pkv_rope_kv_write.argtypes = [T, T, T, T, T, T, T, T, T, T, i32, i32, P, P]
        L.pkv_paged_gqa_decode.argtypes = [T, T, T, T, T, ctypes.c_float, i32, T, T, T, T, i32, P, P]
        L.pkv_rope_kv_write_nvfp4.argtypes = [T, T, T, T, T, T, T, T, T, T, T, T, i32, i32, P, P]
        L.pkv_paged_gqa_decode_nvfp4.argtypes = [T, T, T, T, T, T, T, ctypes.c_float, i32, T, T, T, T, i32, P, P]
        L.pkv_mla_cache_write.argtypes = [T, T, T, T, T, T, T, T, T, i32, P, P]
        L.pkv_paged_mla_decode.argtypes = [T, T, T, T, T, T, ctypes.c_float, i32, T, T, T, P, P]
        L.pkv_choose_num_splits_mla.argtypes = [i32, i32, ctypes.c_int64, i32, i32]
        L.pkv_lse_merge.argtypes = [T, T, T, T, P]
        L.pkv_choose_num_splits.argtypes = [i32, i32, i32, i32, ctypes.c_int64, i32, i32, i32]
        L.pkv_validate_indices.argtypes = [T, T, T, ctypes.c_int64, T, P, P]
        L.pkv_stream_read.argtypes = [P, ctypes.c_int64, P, i32, P]
        L.pkv_selftest_bounded_wait.argtypes = [ctypes.c_int64, P, P, P]
        L.pkv_copy.argtypes = [P, P, ctypes.c_int64, P]
        L.pkv_validate_indices_static.argtypes = [T, T, T, ctypes.c_int64, P, P]
        L.pkv_plan_splits.argtypes = [P, i32, i32, i32, i32, i32, i32, i32, i32, i32, P, P, P, ctypes.c_int64, P]
        L.pkv_paged_gqa_decode_planned.argtypes = [T, T, T, T, T, T, T, ctypes.c_float, T, T, T, T, T, T, i32, P,
                                                   P]
        L.pkv_lse_merge_planned.argtypes = [T, T, T, T, T, P]
        L.pkv_plan_splits_mla.argtypes = [P, i32, i32, i32, i32, i32, i32, P, P, P, ctypes.c_int64, P]
        L.pkv_paged_mla_decode_planned.argtypes = [T, T, T, T, T, T, ctypes.c_float, T, T, T, T, T, P, P]
        L.pkv_status_string.argtypes = [i32]
        L.pkv_status_string.restype = ctypes.c_char_p
        for name in ("pkv_rope_kv_write", "pkv_paged_gqa_decode", "pkv_lse_merge", "pkv_validate_indices",
                     "pkv_choose_num_splits", "pkv_abi_version", "pkv_stream_read", "pkv_validate_indices_static",
                     "pkv_rope_kv_write_nvfp4", "pkv_paged_gqa_decode_nvfp4", "pkv_mla_cache_write",
                     "pkv_paged_mla_decode", "pkv_choose_num_splits_mla", "pkv_selftest_bounded_wait", "pkv_copy",
                     "pkv_plan_splits", "pkv_paged_gqa_decode_planned", "pkv_lse_merge_planned",
                     "pkv_plan_splits_mla", "pkv_paged_mla_decode_planned"):
            getattr(L, name).restype = ctypes.c_int32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def _desc(t: Optional[torch.Tensor], dtype: Optional[int] = None):
    """Pointer to a descriptor of t (NULL for None); `dtype` overrides the
    pkv_dtype taken from t.dtype (uint8 NVFP4 value caches)."""
    if t is None:
        return None
    d = PkvTensor()
    if t.dim() > 4:
        raise ValueError("tensors of more than 4 dims are not part of the ABI")
    if t.dtype not in _DTYPES:
        raise TypeError(f"dtype {t.dtype} is not part of the ABI")
    if t.numel() and not t.is_cuda:
        raise ValueError("the C ABI takes device tensors; copy host data to the GPU first")
    d.ptr = t.data_ptr() if t.numel() else None
    d.dtype = _DTYPES[t.dtype] if dtype is None else dtype
    d.ndim = t.dim()
    for i, (n, s) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = n
        d.stride[i] = s
    return ctypes.pointer(d)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _check(fn: str, status: int) -> None:
    if status != PKV_OK:
        raise PkvError(fn, status)


def rope_kv_write(q, k, v, positions, cos_sin, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                  layout: str = "HND", rope_style: str = "neox", err_flag=None, stream=None) -> None:
    """Fused RoPE + paged-KV write (pkv_rope_kv_write): q (or None) rotated
    in place, rotated k and v written into the caches at slot_mapping."""
    _check("pkv_rope_kv_write", lib().pkv_rope_kv_write(
        _desc(q), _desc(k), _desc(v), _desc(positions), _desc(cos_sin), _desc(k_cache), _desc(v_cache),
        _desc(slot_mapping), _desc(k_scale), _desc(v_scale), LAYOUTS[layout], STYLES[rope_style],
        _ptr(err_flag), _stream(stream)))


def paged_gqa_decode(q, k_cache, v_cache, block_tables, seq_lens, softmax_scale: float, num_splits: int,
                     out_partial, lse_partial, k_scale=None, v_scale=None, layout: str = "HND", err_flag=None,
                     stream=None) -> None:
    """Paged GQA split-K decode (pkv_paged_gqa_decode) into out_partial
    [B,S,Hq,D] and lse_partial [B,S,Hq]."""
    _check("pkv_paged_gqa_decode", lib().pkv_paged_gqa_decode(
        _desc(q), _desc(k_cache), _desc(v_cache), _desc(block_tables), _desc(seq_lens), float(softmax_scale),
        int(num_splits), _desc(out_partial), _desc(lse_partial), _desc(k_scale), _desc(v_scale), LAYOUTS[layout],
        _ptr(err_flag), _stream(stream)))


def _fp4(t):
    if t is not None and t.dtype != torch.uint8:
        raise TypeError("NVFP4 value caches are uint8 tensors of packed E2M1 pairs")
    return _desc(t, PKV_FP4_E2M1X2)


def rope_kv_write_nvfp4(q, k, v, positions, cos_sin, k_cache, v_cache, k_block_scale, v_block_scale,
                        slot_mapping, k_scale, v_scale, layout: str = "HND", rope_style: str = "neox",
                        err_flag=None, stream=None) -> None:
    """pkv_rope_kv_write_nvfp4: as rope_kv_write into NVFP4 caches -- value
    caches uint8 [.., D/2] (packed E2M1 pairs), block-scale caches uint8 or
    float8_e4m3fn [.., D/16], static scales [1] or [Hkv] float32."""
    _check("pkv_rope_kv_write_nvfp4", lib().pkv_rope_kv_write_nvfp4(
        _desc(q), _desc(k), _desc(v), _desc(positions), _desc(cos_sin), _fp4(k_cache), _fp4(v_cache),
        _desc(k_block_scale), _desc(v_block_scale), _desc(slot_mapping), _desc(k_scale), _desc(v_scale),
        LAYOUTS[layout], STYLES[rope_style], _ptr(err_flag), _stream(stream)))


def paged_gqa_decode_nvfp4(q, k_cache, v_cache, k_block_scale, v_block_scale, block_tables, seq_lens,
                           softmax_scale: float, num_splits: int, out_partial, lse_partial, k_scale, v_scale,
                           layout: str = "HND", err_flag=None, stream=None) -> None:
    """pkv_paged_gqa_decode_nvfp4: paged GQA split-K decode over NVFP4
    caches (HND) into out_partial [B,S,Hq,D] and lse_partial [B,S,Hq]."""
    _check("pkv_paged_gqa_decode_nvfp4", lib().pkv_paged_gqa_decode_nvfp4(
        _desc(q), _fp4(k_cache), _fp4(v_cache), _desc(k_block_scale), _desc(v_block_scale), _desc(block_tables),
        _desc(seq_lens), float(softmax_scale), int(num_splits), _desc(out_partial), _desc(lse_partial),
        _desc(k_scale), _desc(v_scale), LAYOUTS[layout], _ptr(err_flag), _stream(stream)))


def mla_cache_write(q_pe, ckv, kpe, positions, cos_sin, ckv_cache, kpe_cache, slot_mapping, ckv_scale,
                    rope_style: str = "interleaved", err_flag=None, stream=None) -> None:
    """pkv_mla_cache_write: ckv [T,512] bf16 -> E4M3 bytes of ckv_cache
    [pages,P,512] (uint8 or float8_e4m3fn), RoPE(kpe [T,64]) -> kpe_cache
    [pages,P,64] bf16, q_pe [T,H,64] (or None) rotated in place."""
    _check("pkv_mla_cache_write", lib().pkv_mla_cache_write(
        _desc(q_pe), _desc(ckv), _desc(kpe), _desc(positions), _desc(cos_sin), _desc(ckv_cache), _desc(kpe_cache),
        _desc(slot_mapping), _desc(ckv_scale), STYLES[rope_style], _ptr(err_flag), _stream(stream)))


def paged_mla_decode(q_lat, q_pe, ckv_cache, kpe_cache, block_tables, seq_lens, softmax_scale: float,
                     num_splits: int, out_partial, lse_partial, ckv_scale, err_flag=None, stream=None) -> None:
    """pkv_paged_mla_decode: q_lat [B,H,512], q_pe [B,H,64] over the latent
    cache into out_partial [B,S,H,512] and lse_partial [B,S,H]."""
    _check("pkv_paged_mla_decode", lib().pkv_paged_mla_decode(
        _desc(q_lat), _desc(q_pe), _desc(ckv_cache), _desc(kpe_cache), _desc(block_tables), _desc(seq_lens),
        float(softmax_scale), int(num_splits), _desc(out_partial), _desc(lse_partial), _desc(ckv_scale),
        _ptr(err_flag), _stream(stream)))


def choose_num_splits_mla(B: int, H: int, total_pages: int, max_pages: int, sm_count: int) -> int:
    """Split count for the MLA decode from the library's heuristic (host only)."""
    return int(lib().pkv_choose_num_splits_mla(B, H, int(total_pages), max_pages, sm_count))


def lse_merge(out_partial, lse_partial, out, lse_out=None, stream=None) -> None:
    """LSE merge of the split partials into out [B,Hq,D] bf16 (pkv_lse_merge)."""
    _check("pkv_lse_merge", lib().pkv_lse_merge(_desc(out_partial), _desc(lse_partial), _desc(out),
                                                 _desc(lse_out), _stream(stream)))


def choose_num_splits(B: int, Hkv: int, Hq: int, D: int, total_pages: int, max_pages: int, cache_dtype: str,
                      sm_count: int) -> int:
    """Split count from the library's heuristic (host only)."""
    return int(lib().pkv_choose_num_splits(B, Hkv, Hq, D, int(total_pages), max_pages,
                                           _CACHE_DTYPE[cache_dtype], sm_count))


def plan_splits(seq_lens, Hkv: int, Hq: int, D: int, max_pages: int, cache_dtype: str, sm_count: int,
                max_splits: int = 4095, target_pages: int = 0):
    """pkv_plan_splits (host only): (splits_per_seq int32 [B], num_records,
    work int32 [W, 2]) for the planned decode and merge."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = int(sl.size)
    sp = np.zeros(max(B, 1), np.int32)
    nrec = ctypes.c_int32(0)
    nwork = ctypes.c_int64(0)
    f = lib().pkv_plan_splits
    args = (sl.ctypes.data if B else None, B, Hkv, Hq, D, max_pages, _CACHE_DTYPE[cache_dtype], sm_count,
            max_splits, target_pages, sp.ctypes.data)
    _check("pkv_plan_splits", f(*args, ctypes.byref(nrec), None, 0, ctypes.byref(nwork)))
    work = np.zeros((max(int(nwork.value), 1), 2), np.int32)
    _check("pkv_plan_splits", f(*args, ctypes.byref(nrec), work.ctypes.data, int(nwork.value), ctypes.byref(nwork)))
    return sp[:B], int(nrec.value), work[:int(nwork.value)]


def paged_gqa_decode_planned(q, k_cache, v_cache, block_tables, seq_lens, softmax_scale: float, splits_per_seq,
                             work, out_partial, lse_partial, k_scale=None, v_scale=None, layout: str = "HND",
                             err_flag=None, stream=None, k_block_scale=None, v_block_scale=None) -> None:
    """pkv_paged_gqa_decode_planned: the decode under a split plan (device
    splits_per_seq [B] and work [W, 2] int32 from plan_splits); NVFP4 caches
    when the block-scale caches are given."""
    fp4 = k_block_scale is not None
    kc, vc = (_fp4(k_cache), _fp4(v_cache)) if fp4 else (_desc(k_cache), _desc(v_cache))
    _check("pkv_paged_gqa_decode_planned", lib().pkv_paged_gqa_decode_planned(
        _desc(q), kc, vc, _desc(k_block_scale), _desc(v_block_scale), _desc(block_tables), _desc(seq_lens),
        float(softmax_scale), _desc(splits_per_seq), _desc(work), _desc(out_partial), _desc(lse_partial),
        _desc(k_scale), _desc(v_scale), LAYOUTS[layout], _ptr(err_flag), _stream(stream)))


def plan_splits_mla(seq_lens, H: int, max_pages: int, sm_count: int, max_splits: int = 4095, target_pages: int = 0):
    """pkv_plan_splits_mla (host only): (splits_per_seq int32 [B],
    num_records, work int32 [W, 2]) for the planned MLA decode."""
    import numpy as np
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = int(sl.size)
    sp = np.zeros(max(B, 1), np.int32)
    nrec = ctypes.c_int32(0)
    nwork = ctypes.c_int64(0)
    f = lib().pkv_plan_splits_mla
    args = (sl.ctypes.data if B else None, B, H, max_pages, sm_count, max_splits, target_pages, sp.ctypes.data)
    _check("pkv_plan_splits_mla", f(*args, ctypes.byref(nrec), None, 0, ctypes.byref(nwork)))
    work = np.zeros((max(int(nwork.value), 1), 2), np.int32)
    _check("pkv_plan_splits_mla", f(*args, ctypes.byref(nrec), work.ctypes.data, int(nwork.value),
                                    ctypes.byref(nwork)))
    return sp[:B], int(nrec.value), work[:int(nwork.value)]


def paged_mla_decode_planned(q_lat, q_pe, ckv_cache, kpe_cache, block_tables, seq_lens, softmax_scale: float,
                             splits_per_seq, work, out_partial, lse_partial, ckv_scale, err_flag=None,
                             stream=None) -> None:
    """pkv_paged_mla_decode_planned: the MLA decode under a split plan."""
    _check("pkv_paged_mla_decode_planned", lib().pkv_paged_mla_decode_planned(
        _desc(q_lat), _desc(q_pe), _desc(ckv_cache), _desc(kpe_cache), _desc(block_tables), _desc(seq_lens),
        float(softmax_scale), _desc(splits_per_seq), _desc(work), _desc(out_partial), _desc(lse_partial),
        _desc(ckv_scale), _ptr(err_flag), _stream(stream)))


def lse_merge_planned(out_partial, lse_partial, splits_per_seq, out, lse_out=None, stream=None) -> None:
    """pkv_lse_merge_planned: each sequence's own records [0, S_b)."""
    _check("pkv_lse_merge_planned", lib().pkv_lse_merge_planned(
        _desc(out_partial), _desc(lse_partial), _desc(splits_per_seq), _desc(out), _desc(lse_out), _stream(stream)))


def validate_indices(block_tables, seq_lens, slot_mapping, num_pages: int, err_flag, slot_bitmap=None,
                     stream=None) -> None:
    """Device check of seq_lens, block tables and slots (pkv_validate_indices)."""
    _check("pkv_validate_indices", lib().pkv_validate_indices(
        _desc(block_tables), _desc(seq_lens), _desc(slot_mapping), int(num_pages), _desc(slot_bitmap),
        _ptr(err_flag), _stream(stream)))


def validate_indices_static(block_tables, seq_lens, slot_mapping, num_pages: int, err_flag, stream=None) -> None:
    """pkv_validate_indices_static: the same check as validate_indices
    (duplicates included) for callers that cannot allocate device memory --
    e.g. an engine whose allocator already holds all free memory for its KV
    pool, or a path that must not call cudaMalloc/cudaFree because they can
    synchronise the device. The bitmap is a fixed 1 MiB device array in the
    library (at most 2**23 cache slots); calls overlapping on the GPU race on
    it, and the first call on a device should come before any stream
    capture."""
    _check("pkv_validate_indices_static", lib().pkv_validate_indices_static(
        _desc(block_tables), _desc(seq_lens), _desc(slot_mapping), int(num_pages), _ptr(err_flag),
        _stream(stream)))


def selftest_bounded_wait(limit_ns: int, err_flag: torch.Tensor, elapsed_ns: torch.Tensor, stream=None) -> None:
    """Self-test of the bounded in-kernel waits (pkv_selftest_bounded_wait):
    err_flag an int32 device word, elapsed_ns two int64 device words."""
    if not (err_flag.is_cuda and err_flag.dtype == torch.int32 and elapsed_ns.is_cuda
            and elapsed_ns.dtype == torch.int64 and elapsed_ns.numel() >= 2):
        raise ValueError("int32 device flag and two int64 device words expected")
    _check("pkv_selftest_bounded_wait",
           lib().pkv_selftest_bounded_wait(int(limit_ns), err_flag.data_ptr(), elapsed_ns.data_ptr(), _stream(stream)))


def copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """pkv_copy: dst <- src byte for byte by the SMs; each a contiguous tensor
    in device memory or in pinned host memory (e.g. from pin_memory()), the
    same number of bytes."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy: dst and src must be contiguous")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("copy: dst and src differ in size")
    _check("pkv_copy", lib().pkv_copy(_ptr(dst), _ptr(src), n, _stream(stream)))


def stream_read(buf: torch.Tensor, sink: torch.Tensor, stream=None) -> None:
    """Streaming-read ceiling (pkv_stream_read): read all of `buf` once in
    one launch of sink.numel() CTAs."""
    if not (buf.is_cuda and sink.is_cuda and sink.dtype == torch.int32):
        raise ValueError("device buffer and int32 device sink expected")
    _check("pkv_stream_read", lib().pkv_stream_read(buf.data_ptr(), buf.numel() * buf.element_size(),
                                                     sink.data_ptr(), sink.numel(), _stream(stream)))
