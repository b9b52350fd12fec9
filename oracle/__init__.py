"""Float64 CPU oracle of the paged-KV decode step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product (the CUDA library and its Python
binding) never imports, loads or calls it, and it imports nothing from the
product: the two share only the seeded input generators.

The arithmetic lives in ``oracle.c`` (plain C, float64, built with
``-ffp-contract=off``); this module builds it with gcc and marshals numpy
arrays. Each function names the passage it follows; see ``oracle.h``.

Pins: every function here is pinned by ``tests/test_oracle_*.py`` against
closed forms, invariants, library routines (torch's bf16 and e4m3fn casts,
torch's float64 scaled-dot-product attention) and hand-worked examples.
No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

LAYOUT = {"NHD": 0, "HND": 1}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no GPU needed)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_bf16_rne_n.argtypes = [P, P, i64]
        lib.orc_e4m3_sat_rne_n.argtypes = [P, P, i64]
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f64.restype = dbl
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_f64.restype = dbl
        lib.orc_rope_rotate_f64.argtypes = [P, P, i32, dbl, dbl, i32]
        lib.orc_rope_row_f32.argtypes = [P, P, P, i32, i32]
        lib.orc_rope_kv_write.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, i64, P, P, i64, i32,
                                          i32, i32, P, P, i32, P]
        lib.orc_rope_kv_write.restype = i64
        lib.orc_decode_head.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, i64, i32, i32, P, P, i32,
                                        P, i32, P, dbl, i32, P, P]
        lib.orc_paged_decode.argtypes = [i32, i32, i32, i32, i32, P, P, P, i64, i32, i32, P, P, i32, P,
                                         i32, P, dbl, i32, P, P]
        lib.orc_lse_merge.argtypes = [i32, i32, i32, i32, P, P, P, P]
        lib.orc_e2m1_sat_rne_n.argtypes = [P, P, i64]
        lib.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e2m1_to_f64.restype = dbl
        lib.orc_nvfp4_block.argtypes = [P, ctypes.c_float, P, P]
        lib.orc_rope_kv_write_nvfp4.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, i64, P, P, P, P, i64,
                                                i32, i32, P, P, i32, P]
        lib.orc_rope_kv_write_nvfp4.restype = i64
        lib.orc_paged_decode_nvfp4.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, i64, i32, P, P, i32, P,
                                               i32, P, dbl, i32, P, P]
        lib.orc_paged_decode_splits.argtypes = [i32, i32, i32, i32, i32, P, P, P, i64, i32, i32, P, P, i32, P,
                                                i32, P, dbl, i32, P, P, P]
        lib.orc_paged_decode_nvfp4_splits.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, i64, i32, P, P, i32,
                                                      P, i32, P, dbl, i32, P, P, P]
        lib.orc_mla_cache_write.argtypes = [i64, i32, i32, i32, i32, P, P, P, P, P, i64, P, P, i64, i32,
                                            ctypes.c_float, P]
        lib.orc_mla_cache_write.restype = i64
        lib.orc_mla_decode.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, i64, ctypes.c_float, P, i32, P,
                                       dbl, i32, P, P]
        lib.orc_mla_decode_splits.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, i64, ctypes.c_float, P, i32, P,
                                              dbl, i32, P, P, P]
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---- encoders ----------------------------------------------------------------
def bf16_rne(x) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (own bit-level definition)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _L().orc_bf16_rne_n(_p(x), _p(out), x.size)
    return out


def e4m3_sat_rne(x) -> np.ndarray:
    """float32 -> OCP E4M3 bytes, saturating to +-448, ties to even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().orc_e4m3_sat_rne_n(_p(x), _p(out), x.size)
    return out


def e4m3_to_f64(b) -> np.ndarray:
    """E4M3 bytes -> float64 from the OCP definition."""
    b = np.asarray(b, np.uint8)
    f = _L().orc_e4m3_to_f64
    return np.array([f(int(v)) for v in b.reshape(-1)], np.float64).reshape(b.shape)


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_table() -> np.ndarray:
    """float64 value of each of the 256 E4M3 codes (NaN for 0x7F / 0xFF)."""
    return e4m3_to_f64(np.arange(256, dtype=np.uint8))


# ---- RoPE --------------------------------------------------------------------
def rope_rotate_f64(x, pos: float, base: float, interleaved: bool) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _L().orc_rope_rotate_f64(_p(x), _p(y), x.shape[-1], float(pos), float(base), int(interleaved))
    return y


def rope_row_f32(x_bits, cs_row, interleaved: bool) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    cs = _c(cs_row, np.float32)
    y = np.empty(x.shape, np.float32)
    _L().orc_rope_row_f32(_p(x), _p(cs), _p(y), x.shape[-1], int(interleaved))
    return y


def rope_kv_write(q, k, v, positions, cos_sin, k_cache, v_cache, slot_mapping, layout: str,
                  style: str, k_scale=None, v_scale=None, page_size: int = 16) -> int:
    """In place on numpy arrays: q [T,Hq,D] uint16 (or None), caches uint16
    (bf16) or uint8 (fp8) of shape NHD [pages,P,Hkv,D] / HND [pages,Hkv,P,D].
    Returns the number of tokens skipped for a bad slot or position."""
    k = _c(k, np.uint16); v = _c(v, np.uint16)
    T, Hkv, D = k.shape
    Hq = 0 if q is None else q.shape[1]
    if q is not None:
        assert q.dtype == np.uint16 and q.flags.c_contiguous
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    fp8 = k_cache.dtype == np.uint8
    pos = _c(positions, np.int32); slot = _c(slot_mapping, np.int32)
    cs = _c(cos_sin, np.float32)
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    n_scale = 0 if ks is None else ks.size
    if fp8 and ks is None:
        raise ValueError("fp8 cache needs scales")
    return int(_L().orc_rope_kv_write(T, Hq, Hkv, D, page_size, _p(q), _p(k), _p(v), _p(pos), _p(cs),
                                      cs.shape[0], _p(k_cache), _p(v_cache), k_cache.shape[0],
                                      LAYOUT[layout], int(style == "interleaved"), int(fp8), _p(ks),
                                      _p(vs), n_scale, _p(slot)))


# ---- attention ---------------------------------------------------------------
def _cache_args(k_cache, layout):
    if layout == "HND":
        num_pages, Hkv, P, D = k_cache.shape
    else:
        num_pages, P, Hkv, D = k_cache.shape
    return num_pages, Hkv, P, D


def decode_head(b: int, h: int, Hq: int, q_row, k_cache, v_cache, block_tables, seq_lens,
                softmax_scale: float, num_splits: int, layout: str, k_scale=None, v_scale=None):
    """Partials (out [S,D] float64, lse [S] float64) of query head h of
    sequence b."""
    num_pages, Hkv, P, D = _cache_args(k_cache, layout)
    fp8 = k_cache.dtype == np.uint8
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32); sl = _c(seq_lens, np.int32)
    qr = _c(q_row, np.uint16)
    o = np.empty((num_splits, D), np.float64)
    l = np.empty(num_splits, np.float64)
    _L().orc_decode_head(b, h, Hq, Hkv, D, P, _p(qr), _p(_c(k_cache, k_cache.dtype)),
                         _p(_c(v_cache, v_cache.dtype)), num_pages, LAYOUT[layout], int(fp8), _p(ks),
                         _p(vs), 0 if ks is None else ks.size, _p(bt), bt.shape[1], _p(sl),
                         float(softmax_scale), num_splits, _p(o), _p(l))
    return o, l


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, softmax_scale: float, num_splits: int,
                 layout: str, k_scale=None, v_scale=None, splits_per_seq=None):
    """q [B,Hq,D] uint16 -> (out_partial [B,S,Hq,D], lse_partial [B,S,Hq]) float64.

    splits_per_seq (int32 [B], optional): the number of splits each
    sequence's pages are dealt into (clamped to [1, num_splits]); its
    records past that count are empty. None = num_splits for every one."""
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = _cache_args(k_cache, layout)
    assert D == D2
    fp8 = k_cache.dtype == np.uint8
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32); sl = _c(seq_lens, np.int32)
    sp = None if splits_per_seq is None else _c(splits_per_seq, np.int32)
    assert sp is None or sp.shape == (B,)
    o = np.empty((B, num_splits, Hq, D), np.float64)
    l = np.empty((B, num_splits, Hq), np.float64)
    _L().orc_paged_decode_splits(B, Hq, Hkv, D, P, _p(q), _p(_c(k_cache, k_cache.dtype)),
                                 _p(_c(v_cache, v_cache.dtype)), num_pages, LAYOUT[layout], int(fp8), _p(ks),
                                 _p(vs), 0 if ks is None else ks.size, _p(bt), bt.shape[1], _p(sl),
                                 float(softmax_scale), num_splits, _p(sp), _p(o), _p(l))
    return o, l


def lse_merge(out_partial, lse_partial):
    """(out_partial [B,S,Hq,D], lse_partial [B,S,Hq]) -> (out [B,Hq,D], lse [B,Hq]) float64."""
    op = _c(out_partial, np.float64); lp = _c(lse_partial, np.float64)
    B, S, Hq, D = op.shape
    out = np.empty((B, Hq, D), np.float64)
    lse = np.empty((B, Hq), np.float64)
    _L().orc_lse_merge(B, S, Hq, D, _p(op), _p(lp), _p(out), _p(lse))
    return out, lse


def empty_cache(shape, cache_dtype: str) -> np.ndarray:
    return np.zeros(shape, np.uint8 if cache_dtype in ("fp8", "nvfp4") else np.uint16)


# ---- NVFP4 (E2M1 values + an E4M3 scale per 16 elements) --------------------
def e2m1_sat_rne(x) -> np.ndarray:
    """float32 -> 4-bit E2M1 codes (uint8, 0..15), saturating to +-6, ties to even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().orc_e2m1_sat_rne_n(_p(x), _p(out), x.size)
    return out


def e2m1_table() -> np.ndarray:
    """float64 value of each of the 16 E2M1 codes."""
    f = _L().orc_e2m1_to_f64
    return np.array([f(c) for c in range(16)], np.float64)


def nvfp4_block(y, g: float):
    """One block of 16 float32 values -> (8 packed bytes, scale byte)."""
    y = _c(y, np.float32)
    assert y.size == 16
    packed = np.empty(8, np.uint8)
    sb = np.empty(1, np.uint8)
    _L().orc_nvfp4_block(_p(y), float(g), _p(packed), _p(sb))
    return packed, int(sb[0])


def rope_kv_write_nvfp4(q, k, v, positions, cos_sin, k_cache, v_cache, k_block_scale, v_block_scale,
                        slot_mapping, layout: str, style: str, k_scale, v_scale, page_size: int = 16) -> int:
    """In place on numpy arrays: value caches uint8 [.., D/2] (packed E2M1
    pairs), scale caches uint8 [.., D/16] (E4M3), both in the given layout."""
    k = _c(k, np.uint16); v = _c(v, np.uint16)
    T, Hkv, D = k.shape
    Hq = 0 if q is None else q.shape[1]
    for a in (k_cache, v_cache, k_block_scale, v_block_scale):
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    pos = _c(positions, np.int32); slot = _c(slot_mapping, np.int32)
    cs = _c(cos_sin, np.float32)
    ks = _c(k_scale, np.float32); vs = _c(v_scale, np.float32)
    return int(_L().orc_rope_kv_write_nvfp4(T, Hq, Hkv, D, page_size, _p(q), _p(k), _p(v), _p(pos), _p(cs),
                                            cs.shape[0], _p(k_cache), _p(v_cache), _p(k_block_scale),
                                            _p(v_block_scale), k_cache.shape[0], LAYOUT[layout],
                                            int(style == "interleaved"), _p(ks), _p(vs), ks.size, _p(slot)))


def paged_decode_nvfp4(q, k_cache, v_cache, k_block_scale, v_block_scale, block_tables, seq_lens,
                       softmax_scale: float, num_splits: int, layout: str, k_scale, v_scale, splits_per_seq=None):
    """As paged_decode, for NVFP4 caches (value caches [.., D/2] bytes)."""
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    if layout == "HND":
        num_pages, Hkv, P, _ = k_cache.shape
    else:
        num_pages, P, Hkv, _ = k_cache.shape
    ks = _c(k_scale, np.float32); vs = _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32); sl = _c(seq_lens, np.int32)
    sp = None if splits_per_seq is None else _c(splits_per_seq, np.int32)
    assert sp is None or sp.shape == (B,)
    o = np.empty((B, num_splits, Hq, D), np.float64)
    l = np.empty((B, num_splits, Hq), np.float64)
    _L().orc_paged_decode_nvfp4_splits(B, Hq, Hkv, D, P, _p(q), _p(_c(k_cache, np.uint8)),
                                       _p(_c(v_cache, np.uint8)), _p(_c(k_block_scale, np.uint8)),
                                       _p(_c(v_block_scale, np.uint8)), num_pages, LAYOUT[layout], _p(ks), _p(vs),
                                       ks.size, _p(bt), bt.shape[1], _p(sl), float(softmax_scale), num_splits,
                                       _p(sp), _p(o), _p(l))
    return o, l


# ---- MLA (absorbed decode form) -----------------------------------------------
def mla_cache_write(q_pe, ckv, kpe, positions, cos_sin, ckv_cache, kpe_cache, slot_mapping, ckv_scale: float,
                    style: str = "interleaved") -> int:
    """In place on numpy arrays: ckv_cache uint8 [pages, P, Dc] (E4M3),
    kpe_cache uint16 [pages, P, Dr] (bf16 bits), q_pe [T, H, Dr] (or None)
    rotated in place. ckv [T, Dc], kpe [T, Dr] bf16 bits."""
    ckv = _c(ckv, np.uint16); kpe = _c(kpe, np.uint16)
    T, Dc = ckv.shape
    Dr = kpe.shape[1]
    H = 0 if q_pe is None else q_pe.shape[1]
    assert ckv_cache.dtype == np.uint8 and kpe_cache.dtype == np.uint16
    assert ckv_cache.flags.c_contiguous and kpe_cache.flags.c_contiguous
    if q_pe is not None:
        assert q_pe.dtype == np.uint16 and q_pe.flags.c_contiguous
    pos = _c(positions, np.int32); slot = _c(slot_mapping, np.int32)
    cs = _c(cos_sin, np.float32)
    return int(_L().orc_mla_cache_write(T, H, Dc, Dr, ckv_cache.shape[1], _p(q_pe), _p(ckv), _p(kpe), _p(pos),
                                        _p(cs), cs.shape[0], _p(ckv_cache), _p(kpe_cache), ckv_cache.shape[0],
                                        int(style == "interleaved"), float(ckv_scale), _p(slot)))


def mla_decode(q_lat, q_pe, ckv_cache, kpe_cache, block_tables, seq_lens, softmax_scale: float, num_splits: int,
               ckv_scale: float, splits_per_seq=None):
    """(out_partial [B,S,H,Dc], lse_partial [B,S,H]) float64. splits_per_seq
    (int32 [B], optional): a split count per sequence, as for paged_decode."""
    q_lat = _c(q_lat, np.uint16); q_pe = _c(q_pe, np.uint16)
    B, H, Dc = q_lat.shape
    Dr = q_pe.shape[2]
    num_pages, P, _ = ckv_cache.shape
    bt = _c(block_tables, np.int32); sl = _c(seq_lens, np.int32)
    sp = None if splits_per_seq is None else _c(splits_per_seq, np.int32)
    assert sp is None or sp.shape == (B,)
    o = np.empty((B, num_splits, H, Dc), np.float64)
    l = np.empty((B, num_splits, H), np.float64)
    _L().orc_mla_decode_splits(B, H, Dc, Dr, P, _p(q_lat), _p(q_pe), _p(_c(ckv_cache, np.uint8)),
                               _p(_c(kpe_cache, np.uint16)), num_pages, float(ckv_scale), _p(bt), bt.shape[1],
                               _p(sl), float(softmax_scale), num_splits, _p(sp), _p(o), _p(l))
    return o, l
