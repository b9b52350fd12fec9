"""Pins of the oracle's 4-bit KV path (CPU): the E2M1 encoder, the NVFP4
block quantiser, the NVFP4 cache write and the decode over NVFP4 caches.

E2M1 is the 4-bit element the decode-attention section of the mainarch page
stores its FP4 KV in ("4-bit E2M1 KV with ... block scales"); the block form
here is NVFP4 (E2M1 values, one E4M3 scale per 16 values, a static scale per
head), the form Blackwell converts natively. Pins: the element table as the
OCP Microscaling definition lists it, nearest-value rounding by brute force
(ties to the even code, saturation at 6), a worked block by hand, the
quantiser's error bound and its amax-to-6 invariant, placement in the cache
against a numpy float32 rotation, and the decode against torch's float64
scaled-dot-product attention on K/V decoded with the literal table."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import synth
from tests._pipeline import E2M1_VALUES, nvfp4_values_f64, oracle_step


# ---- E2M1 element -----------------------------------------------------------
def test_e2m1_table_is_the_ocp_element_set():
    assert np.array_equal(oracle.e2m1_table(), E2M1_VALUES)
    # the sign bit is bit 3
    t = oracle.e2m1_table()
    assert all(math.copysign(1, t[c]) == -1 for c in range(8, 16))


def _nearest_code(x: float) -> int:
    """Brute force: the E2M1 code nearest to x, ties to the even code,
    magnitudes above 6 to 6, the sign kept."""
    sign = 8 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= 6.0:
        return sign | 7
    mags = E2M1_VALUES[:8]
    d = np.abs(mags - a)
    best = np.flatnonzero(d == d.min())
    code = int(best[0]) if len(best) == 1 else int([c for c in best if c % 2 == 0][0])
    return sign | code


def test_e2m1_rounding_by_brute_force():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    pts = [0.0, 1e-30, 0.1, 6.0, 6.5, 7.0, 100.0, 1e30, float(np.finfo(np.float32).max)]
    for m in mids + [0.5, 1.0, 1.5, 2.0, 3.0, 4.0]:
        f = np.float32(m)
        pts += [float(f), float(np.nextafter(f, np.float32(0))), float(np.nextafter(f, np.float32(10)))]
    grid = np.linspace(-8, 8, 64001, dtype=np.float32)
    xs = np.concatenate([np.array(pts, np.float32), -np.array(pts, np.float32), grid])
    got = oracle.e2m1_sat_rne(xs)
    want = np.array([_nearest_code(float(x)) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_e2m1_worked_ties_and_saturation():
    # each tie goes to the neighbour with the even code
    cases = [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
             (-0.25, 0x8), (-5.0, 0xE), (6.0, 0x7), (7.0, 0x7), (1e9, 0x7), (-1e9, 0xF),
             (-0.0, 0x8), (-0.1, 0x8), (0.26, 0x1), (5.01, 0x7)]
    got = oracle.e2m1_sat_rne(np.array([c[0] for c in cases], np.float32))
    assert [int(g) for g in got] == [c[1] for c in cases]


def test_e2m1_monotone_and_odd():
    x = np.linspace(0, 10, 20001, dtype=np.float32)
    v = E2M1_VALUES[oracle.e2m1_sat_rne(x)]
    assert np.all(np.diff(v) >= 0)
    assert np.array_equal(oracle.e2m1_sat_rne(-x[1:]), oracle.e2m1_sat_rne(x[1:]) | 8)


# ---- NVFP4 block -------------------------------------------------------------
def test_nvfp4_worked_block():
    """amax 12 with g = 1: s = E4M3(12 / 6) = 2 (byte 0x40); y / 2 =
    0.25, -0.5, 0.75, 1.5, 3, 6 -> codes 0 (tie, even), 0x9, 2 (tie, even),
    3, 5, 7; element 2i in the low nibble of byte i."""
    y = np.zeros(16, np.float32)
    y[:6] = [0.5, -1.0, 1.5, 3.0, 6.0, 12.0]
    packed, sb = oracle.nvfp4_block(y, 1.0)
    assert sb == 0x40
    assert list(packed) == [0x90, 0x32, 0x75, 0, 0, 0, 0, 0]
    # the static scale divides out: g = 4 gives s = 0.5 (byte 0x30) and the same codes
    packed4, sb4 = oracle.nvfp4_block(y, 4.0)
    assert sb4 == 0x30 and np.array_equal(packed4, packed)


def test_nvfp4_degenerate_blocks():
    # all zero: scale 0, codes 0
    p, sb = oracle.nvfp4_block(np.zeros(16, np.float32), 1.0)
    assert sb == 0 and not p.any()
    # amax / 6 below half of E4M3's smallest subnormal (2^-10): scale 0, codes 0
    p, sb = oracle.nvfp4_block(np.full(16, 1e-4, np.float32), 1.0)
    assert sb == 0 and not p.any()
    # amax / 6 above E4M3's largest value: scale 448 (0x7E), codes saturate to 6
    y = np.full(16, 6000.0, np.float32)
    y[1] = -6000.0
    p, sb = oracle.nvfp4_block(y, 1.0)
    assert sb == 0x7E
    assert p[0] == 0xF7 and all(b == 0x77 for b in p[1:])   # element 1 (-6000) is the high nibble of byte 0


def test_nvfp4_error_bound_and_amax_invariant():
    """For blocks whose scale lands in E4M3's normal range: every element's
    code is within half an E2M1 step of y / (g s) (or clipped to 6 from at
    most 6 / (1 - 2^-4)), and the largest magnitude takes code 7 (|6|)."""
    rng_key = synth.stream_key(4242, "fp4block")
    n = 4000
    y = synth.normal_f32(rng_key, 16 * n).reshape(n, 16)
    sig = np.exp(np.linspace(-3, 3, n)).astype(np.float32)
    y = (y * sig[:, None]).astype(np.float32)
    g = (0.25 + 2 * synth.uniform(synth.stream_key(4242, "g"), n)).astype(np.float32)
    e4 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    checked = 0
    for i in range(n):
        p, sb = oracle.nvfp4_block(y[i], float(g[i]))
        s = e4[sb]
        if not (2.0 ** -6 <= s < 448.0):
            continue
        checked += 1
        codes = np.stack([p & 0xF, p >> 4], axis=-1).reshape(16)
        z = y[i].astype(np.float64) / (np.float64(g[i]) * s)
        q = E2M1_VALUES[codes]
        az = np.abs(z)
        half_step = np.where(az < 2, 0.25, np.where(az < 4, 0.5, 1.0))
        lim = np.where(az <= 6, half_step, az - 6)
        assert np.all(np.abs(z - q) <= lim * (1 + 1e-6) + 1e-12), i
        assert np.all(az <= 6 / (1 - 2.0 ** -4) + 1e-9)
        j = int(np.argmax(np.abs(y[i])))
        assert codes[j] & 7 == 7, i
    assert checked > 3000


# ---- NVFP4 cache write ---------------------------------------------------------
def _rotate_f32(x: np.ndarray, cs: np.ndarray, interleaved: bool) -> np.ndarray:
    """RoPE in numpy float32, each product and sum rounded to float32."""
    D = x.shape[-1]
    c, s = cs[: D // 2], cs[D // 2:]
    if interleaved:
        x1, x2 = x[..., 0::2], x[..., 1::2]
    else:
        x1, x2 = x[..., : D // 2], x[..., D // 2:]
    y1 = (x1 * c) - (x2 * s)
    y2 = (x2 * c) + (x1 * s)
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = y1, y2
    else:
        out[..., : D // 2], out[..., D // 2:] = y1, y2
    return out


@pytest.mark.parametrize("layout,style,per_head", [("HND", "neox", True), ("NHD", "interleaved", False)])
def test_nvfp4_write_places_blocks(layout, style, per_head):
    w = synth.custom_workload("fp4w", 31, [1, 17, 40], 6, 2, 64, layout=layout, style=style,
                              cache_dtype="nvfp4", per_head_scale=per_head, rope_base=5e5)
    st = oracle_step(w)
    cs = w.cos_sin()
    P = w.page_size
    for i in range(w.B):
        k, v = w.seq_kv(i)
        for t in range(int(w.seq_lens[i])):
            page = st["block_tables"][i, t // P]
            kf = synth.bf16_bits_to_f32(k[t])
            yk = _rotate_f32(kf, cs[t], style == "interleaved")
            yv = synth.bf16_bits_to_f32(v[t])
            for h in range(w.Hkv):
                for y, g, vals, scl in ((yk[h], w.k_scale, st["k_cache"], st["k_block_scale"]),
                                        (yv[h], w.v_scale, st["v_cache"], st["v_block_scale"])):
                    gh = float(g[0] if g.size == 1 else g[h])
                    row = vals[page, h, t % P] if layout == "HND" else vals[page, t % P, h]
                    srow = scl[page, h, t % P] if layout == "HND" else scl[page, t % P, h]
                    for blk in range(w.D // 16):
                        p, sb = oracle.nvfp4_block(y[16 * blk:16 * blk + 16], gh)
                        assert np.array_equal(row[8 * blk:8 * blk + 8], p)
                        assert srow[blk] == sb


def test_nvfp4_write_skips_and_counts_bad_slots():
    D, Hkv = 32, 1
    k = np.full((3, Hkv, D), 0x3F80, np.uint16)   # 1.0
    cs = synth.cos_sin_table(4, D, 1e4)
    kc = np.zeros((2, Hkv, 16, D // 2), np.uint8); vc = np.zeros_like(kc)
    ks = np.zeros((2, Hkv, 16, D // 16), np.uint8); vs = np.zeros_like(ks)
    g = np.ones(1, np.float32)
    bad = oracle.rope_kv_write_nvfp4(None, k, k, np.array([0, 1, 9], np.int32), cs, kc, vc, ks, vs,
                                     np.array([-1, 32, 3], np.int32), "HND", "neox", g, g)
    assert bad == 2          # slot 32 is past the pool; position 9 is past the table
    assert not kc.any() and not ks.any()


# ---- decode over NVFP4 caches ---------------------------------------------------
def _gather_fp4(st, w, i, kvh):
    L = int(st["seq_lens"][i])
    P = w.page_size
    out = []
    for vals, scl, g in ((st["k_cache"], st["k_block_scale"], w.k_scale),
                         (st["v_cache"], st["v_block_scale"], w.v_scale)):
        full = nvfp4_values_f64(vals, scl)
        rows = []
        for t in range(L):
            page = st["block_tables"][i, t // P]
            rows.append(full[page, kvh, t % P] if w.layout == "HND" else full[page, t % P, kvh])
        out.append(np.array(rows).reshape(L, w.D) * float(g[0] if g.size == 1 else g[kvh]))
    return out


FP4_CASES = [
    ("hnd_g6", dict(seq_lens=[1, 16, 33, 90], Hq=12, Hkv=2, D=128)),
    ("nhd_interleaved", dict(seq_lens=[7, 40], Hq=4, Hkv=2, D=64, layout="NHD", style="interleaved")),
    ("tensor_scale_g8", dict(seq_lens=[50], Hq=8, Hkv=1, D=128, per_head_scale=False)),
]


@pytest.mark.parametrize("name,kw", FP4_CASES, ids=[c[0] for c in FP4_CASES])
def test_nvfp4_decode_against_torch_sdpa(name, kw):
    w = synth.custom_workload(name, 78, cache_dtype="nvfp4", **kw)
    st = oracle_step(w, num_splits=1)
    for i in range(w.B):
        for h in range(w.Hq):
            k, v = _gather_fp4(st, w, i, h // w.G)
            q = synth.bf16_bits_to_f32(st["q_rot"][i, h]).astype(np.float64)
            qt = torch.from_numpy(q).reshape(1, 1, 1, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None],
                scale=w.softmax_scale).reshape(-1).numpy()
            ref_lse = torch.logsumexp(torch.from_numpy(w.softmax_scale * (k @ q)), 0).item()
            assert np.allclose(st["out"][i, h], ref, rtol=1e-12, atol=1e-12)
            assert abs(st["lse"][i, h] - ref_lse) < 1e-12


def test_nvfp4_split_merge_equals_single_pass():
    w = synth.custom_workload("fp4s", 79, [1, 15, 16, 17, 200], 6, 2, 64, cache_dtype="nvfp4")
    one = oracle_step(w, num_splits=1)
    for S in (2, 5, 13):
        op, lp = oracle.paged_decode_nvfp4(one["q_rot"], one["k_cache"], one["v_cache"], one["k_block_scale"],
                                           one["v_block_scale"], one["block_tables"], one["seq_lens"],
                                           w.softmax_scale, S, w.layout, w.k_scale, w.v_scale)
        out, lse = oracle.lse_merge(op, lp)
        assert np.allclose(out, one["out"], rtol=1e-12, atol=1e-13)
        assert np.allclose(lse, one["lse"], rtol=0, atol=1e-12)


def test_nvfp4_per_sequence_splits_merge_to_the_single_pass():
    w = synth.custom_workload("fp4v", 81, [1, 15, 16, 17, 200], 6, 2, 64, cache_dtype="nvfp4")
    one = oracle_step(w, num_splits=1)
    sp = np.array([1, 4, 2, 6, 3], np.int32)
    op, lp = oracle.paged_decode_nvfp4(one["q_rot"], one["k_cache"], one["v_cache"], one["k_block_scale"],
                                       one["v_block_scale"], one["block_tables"], one["seq_lens"],
                                       w.softmax_scale, 6, w.layout, w.k_scale, w.v_scale, splits_per_seq=sp)
    out, lse = oracle.lse_merge(op, lp)
    assert np.allclose(out, one["out"], rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, one["lse"], rtol=0, atol=1e-12)
    for b, sb in enumerate(sp):
        assert np.all(lp[b, sb:] == -np.inf) and not op[b, sb:].any()


def test_nvfp4_v_scale_enters_linearly():
    w = synth.custom_workload("fp4l", 80, [20, 45], 4, 2, 64, cache_dtype="nvfp4")
    st = oracle_step(w)
    args = (st["q_rot"], st["k_cache"], st["v_cache"], st["k_block_scale"], st["v_block_scale"],
            st["block_tables"], st["seq_lens"], w.softmax_scale, 1, w.layout)
    o1, l1 = oracle.paged_decode_nvfp4(*args, w.k_scale, w.v_scale)
    o2, l2 = oracle.paged_decode_nvfp4(*args, w.k_scale, w.v_scale * np.float32(2.0))
    assert np.array_equal(o2, 2 * o1) and np.array_equal(l1, l2)
