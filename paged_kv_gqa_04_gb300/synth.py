"""Seeded synthetic inputs for the paged-KV decode step.

This module draws random numbers and lays out the shapes, page pools, block
tables and slot mappings of the decode workloads. It holds none of the
method's own arithmetic (no rotation, rounding, quantisation or attention):
the cos/sin table it builds is an input of the cache write, and bf16 input
values are made by truncating float32 bits, which is input synthesis and not
the round-to-nearest-even conversion the cache write performs.

Both sides of every parity check (the CUDA path and the float64 oracle) take
their inputs from here; this module imports neither of them.

Random numbers come from a counter-based generator: output i of stream
(seed, name, index) is the splitmix64 finaliser applied to
key + (i + 1) * 0x9E3779B97F4A7C15, so any sequence's values can be drawn on
their own, in any order. (Normals go through float32 transcendental
functions, whose last bits may differ between CPUs; both sides of a parity
check always draw their inputs in the same process.)

Workload shapes follow the decode regimes the pages describe:
  * Loom Kernels, "Supported operator paths" table, rows "Position and KV"
    (NeoX/interleaved RoPE, NHD/HND views, static per-tensor/per-head FP8
    E4M3 scales) and "Attention" (paged MQA/GQA decode, split-K/LSE merge);
  * mainarch, decode-attention section (long KV, low batch, shuffled page
    layout, Gaussian data with outliers);
  * microLLM-rocm, optimisation checkpoints (Qwen2.5 / DeepSeek-Distill
    1.5B-class cached decode).
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

PAGE_SIZE = 16


def _mix64(x: np.ndarray) -> np.ndarray:
    x = x ^ (x >> np.uint64(30))
    x = x * _M1
    x = x ^ (x >> np.uint64(27))
    x = x * _M2
    return x ^ (x >> np.uint64(31))


def stream_key(seed: int, name: str, index: int = 0) -> np.uint64:
    """64-bit key of one named substream, built from three mixed words so
    that nearby (seed, name, index) triples give unrelated streams."""
    w = np.array([seed & 0xFFFFFFFFFFFFFFFF, zlib.crc32(name.encode()), index & 0xFFFFFFFFFFFFFFFF],
                 dtype=np.uint64)
    with np.errstate(over="ignore"):
        k = _mix64(w[0:1] + _GAMMA)
        k = _mix64(k ^ (w[1:2] * _GAMMA))
        k = _mix64(k ^ (w[2:3] + _GAMMA * np.uint64(3)))
    return k[0]


def raw_u64(key: np.uint64, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of the stream with this key."""
    out = np.empty(n, dtype=np.uint64)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = _raw_chunk(key, start + c0, c1 - c0)
    return out


def _raw_chunk(key: np.uint64, start: int, n: int) -> np.ndarray:
    # splitmix64 of key + (i + 1) * gamma, computed in place
    x = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    t = np.empty_like(x)
    with np.errstate(over="ignore"):
        np.multiply(x, _GAMMA, out=x)
        np.add(x, np.uint64(key), out=x)
        np.right_shift(x, np.uint64(30), out=t); np.bitwise_xor(x, t, out=x); np.multiply(x, _M1, out=x)
        np.right_shift(x, np.uint64(27), out=t); np.bitwise_xor(x, t, out=x); np.multiply(x, _M2, out=x)
        np.right_shift(x, np.uint64(31), out=t); np.bitwise_xor(x, t, out=x)
    return x


def uniform(key: np.uint64, n: int, start: int = 0) -> np.ndarray:
    """float64 uniforms in the open interval (0, 1)."""
    u = raw_u64(key, start, n)
    return ((u >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal_f32(key: np.uint64, n: int) -> np.ndarray:
    """n standard normals (float32), Box-Muller in float32 on pairs of
    uniforms: each 64-bit output gives two 24-bit uniforms, each uniform
    pair gives two normals (cos and sin branch)."""
    npair = (n + 1) // 2
    out = np.empty(2 * npair, dtype=np.float32)
    inv = np.float32(1.0 / 16777216.0)
    half = np.float32(0.5)
    for c0 in range(0, npair, _CHUNK):
        c1 = min(npair, c0 + _CHUNK)
        u = _raw_chunk(key, c0, c1 - c0)
        u1 = ((u >> np.uint64(40)).astype(np.float32) + half) * inv
        u2 = (((u >> np.uint64(8)) & np.uint64(0xFFFFFF)).astype(np.float32) + half) * inv
        r = np.sqrt(np.float32(-2.0) * np.log(u1))
        th = np.float32(2.0 * math.pi) * u2
        out[2 * c0:2 * c1:2] = r * np.cos(th)
        out[2 * c0 + 1:2 * c1:2] = r * np.sin(th)
    return out[:n]


def f32_to_bf16_trunc(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) made by dropping the low 16 bits of float32.

    Input synthesis only: the values are simply random bf16 numbers."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a bit shift)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def cos_sin_table(max_pos: int, head_dim: int, base: float) -> np.ndarray:
    """RoPE table input: float32 [max_pos, head_dim]; columns [0, D/2) hold
    cos(pos * base^(-2i/D)) and [D/2, D) hold the matching sin, each computed
    in float64 and stored as float32."""
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / head_dim)
    pos = np.arange(max_pos, dtype=np.float64)[:, None]
    ang = pos * inv_freq[None, :]
    tab = np.empty((max_pos, head_dim), dtype=np.float32)
    tab[:, :half] = np.cos(ang).astype(np.float32)
    tab[:, half:] = np.sin(ang).astype(np.float32)
    return tab


LAYOUTS = ("NHD", "HND")
STYLES = ("neox", "interleaved")
CACHE_DTYPES = ("bf16", "fp8")
ALL_CACHE_DTYPES = ("bf16", "fp8", "nvfp4")


@dataclasses.dataclass
class Workload:
    """One decode workload: shapes, lengths, page pool and block tables.

    Token values are drawn on demand, per sequence, so that large workloads
    need not be materialised on the host to check a sample of them."""
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    layout: str
    style: str
    cache_dtype: str
    rope_base: float
    seq_lens: np.ndarray            # int32 [B]
    num_pages: int                  # physical pages in the pool
    block_tables: np.ndarray        # int32 [B, max_pages], -1 padded
    k_scale: Optional[np.ndarray]   # float32 [1] or [Hkv] (fp8 only)
    v_scale: Optional[np.ndarray]
    k_mult: float = 1.0             # K values scaled by this before bf16
    outlier_p: float = 0.0          # probability that a K row is scaled x8
    num_splits: tuple = ()
    page_size: int = PAGE_SIZE

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_pages(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_pos(self) -> int:
        return int(self.seq_lens.max()) if self.B else 1

    @property
    def elem_bytes(self) -> float:
        """Bytes per cached value in the value cache (NVFP4: half a byte)."""
        return {"fp8": 1, "nvfp4": 0.5}.get(self.cache_dtype, 2)

    @property
    def cache_bytes_per_value(self) -> float:
        """Value-cache bytes plus block-scale bytes per cached value (NVFP4:
        1/2 + 1/16)."""
        return self.elem_bytes + (1.0 / 16 if self.cache_dtype == "nvfp4" else 0.0)

    @property
    def pages_per_seq(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.page_size - 1) // self.page_size

    def cache_shape(self) -> tuple:
        """Shape of the value cache in storage units (bf16 / E4M3 values, or
        bytes of packed E2M1 pairs for NVFP4)."""
        P = self.page_size
        last = self.D // 2 if self.cache_dtype == "nvfp4" else self.D
        if self.layout == "HND":
            return (self.num_pages, self.Hkv, P, last)
        return (self.num_pages, P, self.Hkv, last)

    def scale_shape(self) -> tuple:
        """NVFP4 block-scale cache: one E4M3 byte per 16 values."""
        P = self.page_size
        if self.layout == "HND":
            return (self.num_pages, self.Hkv, P, self.D // 16)
        return (self.num_pages, P, self.Hkv, self.D // 16)

    def cos_sin(self) -> np.ndarray:
        return cos_sin_table(max(self.max_pos, 1), self.D, self.rope_base)

    # ---- per-sequence token data -------------------------------------
    def seq_kv(self, b: int):
        """bf16 bits of K and V for positions 0..L-1 of sequence b,
        each uint16 [L, Hkv, D] (K before rotation)."""
        L = int(self.seq_lens[b])
        n = L * self.Hkv * self.D
        k = normal_f32(stream_key(self.seed, "k", b), n)
        v = normal_f32(stream_key(self.seed, "v", b), n)
        if self.k_mult != 1.0:
            k = k * np.float32(self.k_mult)
        if self.outlier_p > 0.0:
            u = uniform(stream_key(self.seed, "outlier", b), L * self.Hkv)
            rows = np.where(u < self.outlier_p, np.float32(8.0), np.float32(1.0))
            k = (k.reshape(L * self.Hkv, self.D) * rows[:, None]).reshape(-1)
        k = f32_to_bf16_trunc(k).reshape(L, self.Hkv, self.D)
        v = f32_to_bf16_trunc(v).reshape(L, self.Hkv, self.D)
        return k, v

    def seq_q(self, b: int) -> np.ndarray:
        """bf16 bits of the new token's q for sequence b: uint16 [Hq, D]."""
        q = normal_f32(stream_key(self.seed, "q", b), self.Hq * self.D)
        return f32_to_bf16_trunc(q).reshape(self.Hq, self.D)

    def slots(self, b: int, positions: np.ndarray) -> np.ndarray:
        """Cache slot (page * page_size + offset) of the given positions."""
        pos = np.asarray(positions, dtype=np.int64)
        page = self.block_tables[b, pos // self.page_size].astype(np.int64)
        return (page * self.page_size + pos % self.page_size).astype(np.int32)

    # ---- batched calls ------------------------------------------------
    def fill_batch(self, seqs=None):
        """Context tokens 0..L-2 of each sequence, as one cache-write call
        with no q: dict(k, v [T,Hkv,D] uint16, positions [T], slot_mapping [T])."""
        seqs = range(self.B) if seqs is None else seqs
        ks, vs, ps, ss = [], [], [], []
        for b in seqs:
            L = int(self.seq_lens[b])
            if L <= 1:
                continue
            k, v = self.seq_kv(b)
            pos = np.arange(L - 1, dtype=np.int32)
            ks.append(k[:L - 1]); vs.append(v[:L - 1]); ps.append(pos)
            ss.append(self.slots(b, pos))
        if not ks:
            z = np.zeros((0, self.Hkv, self.D), np.uint16)
            return dict(k=z, v=z.copy(), positions=np.zeros(0, np.int32), slot_mapping=np.zeros(0, np.int32))
        return dict(k=np.concatenate(ks), v=np.concatenate(vs),
                    positions=np.concatenate(ps), slot_mapping=np.concatenate(ss))

    def decode_batch(self):
        """The new token (position L-1) of every sequence, as one cache-write
        call with q: dict(q [B,Hq,D], k, v [B,Hkv,D] uint16, positions [B],
        slot_mapping [B])."""
        q = np.zeros((self.B, self.Hq, self.D), np.uint16)
        k = np.zeros((self.B, self.Hkv, self.D), np.uint16)
        v = np.zeros((self.B, self.Hkv, self.D), np.uint16)
        pos = np.zeros(self.B, np.int32)
        slot = np.full(self.B, -1, np.int32)
        for b in range(self.B):
            L = int(self.seq_lens[b])
            q[b] = self.seq_q(b)
            if L >= 1:
                kk, vv = self.seq_kv(b)
                k[b] = kk[L - 1]; v[b] = vv[L - 1]
                pos[b] = L - 1
                slot[b] = self.slots(b, np.array([L - 1]))[0]
        return dict(q=q, k=k, v=v, positions=pos, slot_mapping=slot)


def _pool_tables(seed: int, seq_lens: np.ndarray, num_pages: int, page_size: int = PAGE_SIZE):
    """Block tables drawn from a shuffled pool: each sequence takes the next
    ceil(L/page_size) entries of a seeded permutation of the pool."""
    need = (seq_lens.astype(np.int64) + page_size - 1) // page_size
    total = int(need.sum())
    if total > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {total}")
    perm = np.argsort(uniform(stream_key(seed, "pool"), num_pages), kind="stable").astype(np.int32)
    width = max(1, int(need.max()) if len(need) else 1)
    bt = np.full((len(seq_lens), width), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return bt


def _uniform_int(seed: int, name: str, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive."""
    u = uniform(stream_key(seed, name), n)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


def make_workload(name: str, seed: Optional[int] = None) -> Workload:
    """The decode workloads:

    tiny        B2, L {37,100}, 4/2 heads, D64, HND, NeoX base 1e4, 16 pages
    qwen        B32, L ~ U[512,4096], 12/2, D128, HND, K x0.5, 12000-page pool
    longctx     B2, L 32768, 28/4, D128, HND, 8192-page pool
    ragged      B256, L lognormal (median 1024, sigma 1, clip [1,8192]),
                32/8, D128, NHD, interleaved base 5e5, 1% K rows x8
    fp8         B64, L ~ U[2048,16384], 12/2, D128, HND, E4M3 cache,
                per-head K/V scales ~ U[0.01, 0.1]
    fp4         the fp8 workload's shapes with an NVFP4 cache: packed E2M1
                values, an E4M3 scale per 16 values, static per-head scales
                ~ U[0.5, 1.5]
    million     B1, L = 2^20, 8/1 (GQA 8), D128, HND, NeoX base 1e6,
                a 65536-page shuffled pool (the 1M-token regime of the
                mainarch decode-attention tables)
    """
    idx = {"tiny": 0, "qwen": 1, "longctx": 2, "ragged": 3, "fp8": 4, "million": 5, "fp4": 6}[name]
    seed = 1000 + idx if seed is None else seed
    if name == "tiny":
        L = np.array([37, 100], np.int32)
        bt = _pool_tables(seed, L, 16)
        return Workload(name, seed, 2, 4, 2, 64, "HND", "neox", "bf16", 1e4, L, 16, bt, None, None,
                        num_splits=(1, 2))
    if name == "qwen":
        L = _uniform_int(seed, "lens", 32, 512, 4096)
        return Workload(name, seed, 32, 12, 2, 128, "HND", "neox", "bf16", 1e6, L, 12000,
                        _pool_tables(seed, L, 12000), None, None, k_mult=0.5)
    if name == "longctx":
        L = np.full(2, 32768, np.int32)
        return Workload(name, seed, 2, 28, 4, 128, "HND", "neox", "bf16", 1e6, L, 8192,
                        _pool_tables(seed, L, 8192), None, None, num_splits=(16, 32, 48, 64))
    if name == "ragged":
        z = normal_f32(stream_key(seed, "lens"), 256).astype(np.float64)
        L = np.clip(np.rint(1024.0 * np.exp(z)), 1, 8192).astype(np.int32)
        pool = int(((L.astype(np.int64) + 15) // 16).sum())
        return Workload(name, seed, 256, 32, 8, 128, "NHD", "interleaved", "bf16", 5e5, L, pool,
                        _pool_tables(seed, L, pool), None, None, outlier_p=0.01)
    if name == "fp4":
        L = _uniform_int(seed, "lens", 64, 2048, 16384)
        pool = int(((L.astype(np.int64) + 15) // 16).sum())
        ks = (0.5 + uniform(stream_key(seed, "kscale"), 2)).astype(np.float32)
        vs = (0.5 + uniform(stream_key(seed, "vscale"), 2)).astype(np.float32)
        return Workload(name, seed, 64, 12, 2, 128, "HND", "neox", "nvfp4", 1e6, L, pool,
                        _pool_tables(seed, L, pool), ks, vs)
    if name == "million":
        L = np.full(1, 1 << 20, np.int32)
        return Workload(name, seed, 1, 8, 1, 128, "HND", "neox", "bf16", 1e6, L, 1 << 16,
                        _pool_tables(seed, L, 1 << 16), None, None)
    # fp8
    L = _uniform_int(seed, "lens", 64, 2048, 16384)
    pool = int(((L.astype(np.int64) + 15) // 16).sum())
    ks = (0.01 + 0.09 * uniform(stream_key(seed, "kscale"), 2)).astype(np.float32)
    vs = (0.01 + 0.09 * uniform(stream_key(seed, "vscale"), 2)).astype(np.float32)
    return Workload(name, seed, 64, 12, 2, 128, "HND", "neox", "fp8", 1e6, L, pool,
                    _pool_tables(seed, L, pool), ks, vs)


WORKLOADS = ("tiny", "qwen", "longctx", "ragged", "fp8", "million", "fp4")


def custom_workload(name: str, seed: int, seq_lens, Hq: int, Hkv: int, D: int, layout: str = "HND",
                    style: str = "neox", cache_dtype: str = "bf16", rope_base: float = 1e4,
                    num_pages: Optional[int] = None, per_head_scale: bool = True,
                    k_mult: float = 1.0, outlier_p: float = 0.0, width: Optional[int] = None) -> Workload:
    """A small workload of any shape, for edge cases (empty, ragged tails,
    one-token contexts, maximum group size)."""
    L = np.asarray(seq_lens, np.int32)
    need = int(((L.astype(np.int64) + 15) // 16).sum())
    pool = max(need, 1) if num_pages is None else num_pages
    bt = _pool_tables(seed, L, pool)
    if width is not None and width > bt.shape[1]:
        bt = np.concatenate([bt, np.full((bt.shape[0], width - bt.shape[1]), -1, np.int32)], axis=1)
    ks = vs = None
    if cache_dtype == "fp8":
        n = Hkv if per_head_scale else 1
        ks = (0.01 + 0.09 * uniform(stream_key(seed, "kscale"), n)).astype(np.float32)
        vs = (0.01 + 0.09 * uniform(stream_key(seed, "vscale"), n)).astype(np.float32)
    elif cache_dtype == "nvfp4":
        n = Hkv if per_head_scale else 1
        ks = (0.5 + uniform(stream_key(seed, "kscale"), n)).astype(np.float32)
        vs = (0.5 + uniform(stream_key(seed, "vscale"), n)).astype(np.float32)
    return Workload(name, seed, len(L), Hq, Hkv, D, layout, style, cache_dtype, rope_base, L, pool, bt,
                    ks, vs, k_mult=k_mult, outlier_p=outlier_p)


# ---- multi-head latent attention (MLA) workloads ---------------------------------
MLA_PAGE_SIZE = 64   # tokens per page of the latent cache (mainarch's MLA run: 51,200 tokens in 800 pages)
MLA_DC = 512         # compressed latent (ckv) values per token
MLA_DR = 64          # positional (kpe) values per token


@dataclasses.dataclass
class MlaWorkload:
    """One MLA decode workload: B sequences, H query heads sharing one latent
    cache of Dc-value ckv rows (FP8 E4M3, static per-tensor scale) and
    Dr-value kpe rows (bf16), pages of page_size tokens."""
    name: str
    seed: int
    B: int
    H: int
    seq_lens: np.ndarray            # int32 [B]
    num_pages: int
    block_tables: np.ndarray        # int32 [B, max_pages], -1 padded
    ckv_scale: float                # float32-representable (the call takes a float32)
    rope_base: float = 1e4
    style: str = "interleaved"
    Dc: int = MLA_DC
    Dr: int = MLA_DR
    page_size: int = MLA_PAGE_SIZE

    @property
    def softmax_scale(self) -> float:
        # the query/key head width of the absorbed form: 128 no-position
        # values (as in the per-head projections) + Dr positional values
        return 1.0 / math.sqrt(128 + self.Dr)

    @property
    def pages_per_seq(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.page_size - 1) // self.page_size

    @property
    def max_pos(self) -> int:
        return int(self.seq_lens.max()) if self.B else 1

    def cos_sin(self) -> np.ndarray:
        return cos_sin_table(max(self.max_pos, 1), self.Dr, self.rope_base)

    def seq_latent(self, b: int):
        """bf16 bits of ckv [L, Dc] and kpe [L, Dr] (kpe before rotation) of
        sequence b."""
        L = int(self.seq_lens[b])
        ckv = normal_f32(stream_key(self.seed, "ckv", b), L * self.Dc)
        kpe = normal_f32(stream_key(self.seed, "kpe", b), L * self.Dr)
        return f32_to_bf16_trunc(ckv).reshape(L, self.Dc), f32_to_bf16_trunc(kpe).reshape(L, self.Dr)

    def seq_q(self, b: int):
        """bf16 bits of the new token's q_lat [H, Dc] and q_pe [H, Dr] (q_pe
        before rotation)."""
        ql = normal_f32(stream_key(self.seed, "qlat", b), self.H * self.Dc)
        qp = normal_f32(stream_key(self.seed, "qpe", b), self.H * self.Dr)
        return f32_to_bf16_trunc(ql).reshape(self.H, self.Dc), f32_to_bf16_trunc(qp).reshape(self.H, self.Dr)

    def slots(self, b: int, positions: np.ndarray) -> np.ndarray:
        pos = np.asarray(positions, dtype=np.int64)
        page = self.block_tables[b, pos // self.page_size].astype(np.int64)
        return (page * self.page_size + pos % self.page_size).astype(np.int32)

    def fill_batch(self, seqs=None):
        """Context tokens 0..L-2 of each sequence as one cache-write call with
        no q: dict(ckv [T,Dc], kpe [T,Dr] uint16, positions [T], slot_mapping [T])."""
        seqs = range(self.B) if seqs is None else seqs
        cs, ks, ps, ss = [], [], [], []
        for b in seqs:
            L = int(self.seq_lens[b])
            if L <= 1:
                continue
            c, k = self.seq_latent(b)
            pos = np.arange(L - 1, dtype=np.int32)
            cs.append(c[:L - 1]); ks.append(k[:L - 1]); ps.append(pos); ss.append(self.slots(b, pos))
        if not cs:
            return dict(ckv=np.zeros((0, self.Dc), np.uint16), kpe=np.zeros((0, self.Dr), np.uint16),
                        positions=np.zeros(0, np.int32), slot_mapping=np.zeros(0, np.int32))
        return dict(ckv=np.concatenate(cs), kpe=np.concatenate(ks), positions=np.concatenate(ps),
                    slot_mapping=np.concatenate(ss))

    def decode_batch(self):
        """The new token (position L-1) of every sequence: dict(q_lat [B,H,Dc],
        q_pe [B,H,Dr], ckv [B,Dc], kpe [B,Dr], positions [B], slot_mapping [B])."""
        ql = np.zeros((self.B, self.H, self.Dc), np.uint16)
        qp = np.zeros((self.B, self.H, self.Dr), np.uint16)
        ckv = np.zeros((self.B, self.Dc), np.uint16)
        kpe = np.zeros((self.B, self.Dr), np.uint16)
        pos = np.zeros(self.B, np.int32)
        slot = np.full(self.B, -1, np.int32)
        for b in range(self.B):
            L = int(self.seq_lens[b])
            ql[b], qp[b] = self.seq_q(b)
            if L >= 1:
                c, k = self.seq_latent(b)
                ckv[b] = c[L - 1]; kpe[b] = k[L - 1]
                pos[b] = L - 1
                slot[b] = self.slots(b, np.array([L - 1]))[0]
        return dict(q_lat=ql, q_pe=qp, ckv=ckv, kpe=kpe, positions=pos, slot_mapping=slot)


def make_mla_workload(name: str, seed: Optional[int] = None) -> MlaWorkload:
    """The MLA decode workloads (latent 512 FP8 + positional 64 bf16, pages of
    64 tokens, interleaved RoPE base 1e4 on the positional part):

    mla_tiny   B2, L {100, 300} (7 pages), 8 heads, an 11-page shuffled pool
    mla        B1, L 51,200 (800 pages), 8 heads, 1024-page shuffled pool:
               mainarch's MLA decode run (51,200 tokens across 800 pages,
               8 heads)
    mla_batch  B32, L ~ U[4096, 16384], 16 heads (a 128-head model over 8
               GPUs), pool = the pages needed, shuffled
    """
    idx = {"mla_tiny": 0, "mla": 1, "mla_batch": 2}[name]
    seed = 2000 + idx if seed is None else seed
    cs = float(np.float32(0.01 + 0.04 * uniform(stream_key(seed, "ckvscale"), 1)[0]))  # a float32 input
    if name == "mla_tiny":
        L = np.array([100, 300], np.int32)
        return MlaWorkload(name, seed, 2, 8, L, 11, _pool_tables(seed, L, 11, MLA_PAGE_SIZE), cs)
    if name == "mla":
        L = np.array([51200], np.int32)
        return MlaWorkload(name, seed, 1, 8, L, 1024, _pool_tables(seed, L, 1024, MLA_PAGE_SIZE), cs)
    L = _uniform_int(seed, "lens", 32, 4096, 16384)
    pool = int(((L.astype(np.int64) + MLA_PAGE_SIZE - 1) // MLA_PAGE_SIZE).sum())
    return MlaWorkload(name, seed, 32, 16, L, pool, _pool_tables(seed, L, pool, MLA_PAGE_SIZE), cs)


MLA_WORKLOADS = ("mla_tiny", "mla", "mla_batch")


def custom_mla_workload(name: str, seed: int, seq_lens, H: int, style: str = "interleaved",
                        num_pages: Optional[int] = None, rope_base: float = 1e4,
                        ckv_scale: Optional[float] = None) -> MlaWorkload:
    """A small MLA workload of any batch and head count (edge cases)."""
    L = np.asarray(seq_lens, np.int32)
    need = int(((L.astype(np.int64) + MLA_PAGE_SIZE - 1) // MLA_PAGE_SIZE).sum())
    pool = max(need, 1) if num_pages is None else num_pages
    cs = float(np.float32(0.01 + 0.04 * uniform(stream_key(seed, "ckvscale"), 1)[0]) if ckv_scale is None
               else np.float32(ckv_scale))
    return MlaWorkload(name, seed, len(L), H, L, pool, _pool_tables(seed, L, pool, MLA_PAGE_SIZE), cs,
                       rope_base=rope_base, style=style)
