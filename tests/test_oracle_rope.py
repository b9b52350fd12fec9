"""Pins of the oracle's RoPE + paged-cache write (CPU).

Checked against hand-worked examples (tests/golden/rope_worked.json), the
rotation's invariants (identity at position 0, norm preservation, dependence
of <R_m q, R_n k> on m - n only), the NeoX/interleaved relation, and the
slot -> (page, offset) placement in both cache layouts.
(Loom Kernels, "Supported operator paths" table, row "Position and KV";
microLLM-rocm, optimisation checkpoints: split-half RoPE.)"""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_gqa_04_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "rope_worked.json")))


def _bf16(x):
    # Inputs of the worked examples are exact bf16 values; truncation is exact for them.
    b = synth.f32_to_bf16_trunc(np.asarray(x, np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(b), np.asarray(x, np.float32))
    return b


def _write_one(x_bits, cs_row, style, q=None, v_bits=None, cache_dtype="bf16", scale=None, layout="HND"):
    """Run the oracle cache write on one token, one kv head, a one-page pool,
    slot 5; return (q_after, k_bytes, v_bytes)."""
    D = len(x_bits)
    k = np.asarray(x_bits, np.uint16).reshape(1, 1, D)
    v = (np.zeros_like(k) if v_bits is None else np.asarray(v_bits, np.uint16).reshape(1, 1, D))
    cs = np.asarray(cs_row, np.float32).reshape(1, D)
    kc = oracle.empty_cache((1, 1, 16, D) if layout == "HND" else (1, 16, 1, D), cache_dtype)
    vc = np.zeros_like(kc)
    qq = None if q is None else np.asarray(q, np.uint16).reshape(1, 1, D).copy()
    sc = None if scale is None else np.array([scale], np.float32)
    bad = oracle.rope_kv_write(qq, k, v, np.array([0], np.int32), cs, kc, vc, np.array([5], np.int32),
                               layout, style, sc, sc)
    assert bad == 0
    slot = (0, 0, 5) if layout == "HND" else (0, 5, 0)
    return qq, kc[slot], vc[slot]


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: c["name"])
def test_worked_rotation(case):
    xb = np.asarray(case["x_bf16_bits"], np.uint16) if "x_bf16_bits" in case else _bf16(case["x"])
    cs = (np.asarray(case["cs_row_f32_bits"], np.uint32).view(np.float32) if "cs_row_f32_bits" in case
          else np.asarray(case["cs_row"], np.float32))
    inter = case["style"] == "interleaved"
    y = oracle.rope_row_f32(xb, cs, inter)
    if "y" in case:
        assert np.array_equal(y, np.asarray(case["y"], np.float32))
    if "y_f32_bits" in case:
        assert np.array_equal(y.view(np.uint32), np.asarray(case["y_f32_bits"], np.uint32))
    qq, kb, _ = _write_one(xb, cs, case["style"], q=xb)
    assert np.array_equal(kb, np.asarray(case["y_bf16_bits"], np.uint16))
    assert np.array_equal(qq.reshape(-1), np.asarray(case["y_bf16_bits"], np.uint16))


@pytest.mark.parametrize("case", GOLD["fp8_cases"], ids=lambda c: c["name"])
@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_worked_fp8_write(case, layout):
    _, kb, vb = _write_one(_bf16(case["k"]), case["cs_row"], case["style"], v_bits=_bf16(case["v"]),
                           cache_dtype="fp8", scale=case["scale"], layout=layout)
    assert [int(b) for b in kb] == case["k_bytes"]
    assert [int(b) for b in vb] == case["v_bytes"]


@pytest.mark.parametrize("style", synth.STYLES)
def test_position_zero_is_identity(style):
    """Row 0 of the table is cos = 1, sin = 0: the cache holds k unchanged
    and q is unchanged, bit for bit."""
    D, T, Hq, Hkv = 64, 5, 4, 2
    rng_k = synth.normal_f32(synth.stream_key(7, "k"), T * Hkv * D)
    rng_q = synth.normal_f32(synth.stream_key(7, "q"), T * Hq * D)
    k = synth.f32_to_bf16_trunc(rng_k).reshape(T, Hkv, D)
    q = synth.f32_to_bf16_trunc(rng_q).reshape(T, Hq, D)
    v = k[::-1].copy()
    cs = synth.cos_sin_table(4, D, 1e4)
    kc = oracle.empty_cache((2, Hkv, 16, D), "bf16")
    vc = np.zeros_like(kc)
    q2 = q.copy()
    slots = np.array([0, 3, 16, 17, 31], np.int32)
    oracle.rope_kv_write(q2, k, v, np.zeros(T, np.int32), cs, kc, vc, slots, "HND", style)
    assert np.array_equal(q2, q)
    for t, s in enumerate(slots):
        assert np.array_equal(kc[s // 16, :, s % 16, :], k[t])
        assert np.array_equal(vc[s // 16, :, s % 16, :], v[t])


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotation_preserves_norm(interleaved):
    x = synth.normal_f32(synth.stream_key(3, "x"), 128).astype(np.float64)
    for pos in (1, 17, 1000, 123456):
        y = oracle.rope_rotate_f64(x, pos, 1e6, interleaved)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)


@pytest.mark.parametrize("interleaved", [False, True])
def test_relative_position(interleaved):
    """<R_m q, R_n k> depends only on m - n."""
    q = synth.normal_f32(synth.stream_key(4, "q"), 128).astype(np.float64)
    k = synth.normal_f32(synth.stream_key(4, "k"), 128).astype(np.float64)
    base = 1e4
    for m, n, j in ((5, 2, 7), (100, 300, 1000), (0, 0, 12345)):
        a = oracle.rope_rotate_f64(q, m, base, interleaved) @ oracle.rope_rotate_f64(k, n, base, interleaved)
        b = oracle.rope_rotate_f64(q, m + j, base, interleaved) @ oracle.rope_rotate_f64(k, n + j, base, interleaved)
        assert abs(a - b) <= 1e-10 * (np.abs(q).sum() * np.abs(k).sum())


def test_rotation_by_quarter_turn():
    """An angle of pi/2 on one pair maps (x1, x2) to (-x2, x1)."""
    D = 2
    x = np.array([0.3, -1.7])
    # pos * base^0 = pi/2 for the single frequency of D = 2
    y = oracle.rope_rotate_f64(x, np.pi / 2, 10.0, False)
    assert np.allclose(y, [1.7, 0.3], atol=1e-15)


def test_neox_equals_interleaved_under_permutation():
    """Interleaved RoPE of x equals NeoX RoPE of x with element 2i moved to
    i and 2i+1 moved to i + D/2 (and the result moved back), bit for bit."""
    D = 128
    xb = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(5, "x"), D))
    cs = synth.cos_sin_table(50, D, 5e5)[37]
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])   # neox index -> interleaved index
    y_int = oracle.rope_row_f32(xb, cs, True)
    y_neox = oracle.rope_row_f32(xb[perm], cs, False)
    back = np.empty_like(y_neox)
    back[perm] = y_neox
    assert np.array_equal(back.view(np.uint32), y_int.view(np.uint32))


def test_table_rows_match_analytic_rotation():
    """The byte-exact rotation with the float32 table agrees with the
    float64 analytic rotation to float32 accuracy."""
    D = 128
    xb = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(6, "x"), D))
    tab = synth.cos_sin_table(4096, D, 1e6)
    for pos in (1, 2047, 4095):
        for inter in (False, True):
            y = oracle.rope_row_f32(xb, tab[pos], inter).astype(np.float64)
            ref = oracle.rope_rotate_f64(synth.bf16_bits_to_f32(xb).astype(np.float64), pos, 1e6, inter)
            assert np.max(np.abs(y - ref)) < 1e-5


@pytest.mark.parametrize("layout", synth.LAYOUTS)
def test_slot_placement_and_skips(layout):
    """slot = page * 16 + offset lands in the right page row in either
    layout; negative slots are skipped silently; slots beyond the pool and
    positions outside the table are skipped and counted."""
    D, Hkv = 64, 3
    T = 6
    k = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(8, "k"), T * Hkv * D)).reshape(T, Hkv, D)
    v = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(8, "v"), T * Hkv * D)).reshape(T, Hkv, D)
    cs = synth.cos_sin_table(10, D, 1e4)
    shape = (4, Hkv, 16, D) if layout == "HND" else (4, 16, Hkv, D)
    kc = oracle.empty_cache(shape, "bf16"); vc = np.zeros_like(kc)
    slots = np.array([63, -1, 0, 64, 20, 33], np.int32)
    pos = np.array([1, 2, 3, 4, 11, 9], np.int32)
    bad = oracle.rope_kv_write(None, k, v, pos, cs, kc, vc, slots, layout, "neox")
    assert bad == 2  # slot 64 (pool has 64 slots) and position 11 (table has 10 rows)
    written = {63: 0, 0: 2, 33: 5}
    for s in range(64):
        page, off = divmod(s, 16)
        row_v = vc[page, :, off, :] if layout == "HND" else vc[page, off, :, :]
        if s in written:
            assert np.array_equal(row_v, v[written[s]])
        else:
            assert not row_v.any()
