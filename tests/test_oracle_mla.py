"""Pins of the oracle's MLA path (CPU): the latent-cache write and the
absorbed-form decode (mainarch, MLA decode section: FP8 E4M3 ckv of 512
values beside BF16 kpe of 64 values per token, per-head scores, local
softmax with exported LSE, softmax-weighted latent outputs, split-K and a
stage-2 merge).

The decode is checked against torch's float64 scaled-dot-product attention
with keys [ckv * scale | kpe] (576 values) and values ckv * scale (512),
decoded through torch's float8_e4m3fn and bfloat16 views; and by closed
forms and invariants (one-token context returns the latent, split-K + merge
= one pass, physical page permutation). The write is checked against
torch's float8 / bfloat16 casts of a numpy float32 computation."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import synth
from tests._pipeline import mla_oracle_step


def _f64_e4m3(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _f64_bf16(u):
    return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _gather(st, w, i):
    L = int(st["seq_lens"][i])
    P = w.page_size
    rows = [st["block_tables"][i, t // P] * P + t % P for t in range(L)]
    ckv = _f64_e4m3(st["ckv_cache"].reshape(-1, w.Dc)[rows]) * w.ckv_scale
    kpe = _f64_bf16(st["kpe_cache"].reshape(-1, w.Dr)[rows])
    return ckv, kpe


MLA_CASES = [
    ("tiny", dict()),
    ("ragged_h16_neox", dict(seq_lens=[1, 63, 64, 65, 200], H=16, style="neox")),
    ("h1", dict(seq_lens=[130], H=1)),
]


def _workload(name, kw):
    return synth.make_mla_workload("mla_tiny") if name == "tiny" else synth.custom_mla_workload(name, 91, **kw)


@pytest.mark.parametrize("name,kw", MLA_CASES, ids=[c[0] for c in MLA_CASES])
def test_mla_decode_against_torch_sdpa(name, kw):
    w = _workload(name, kw)
    st = mla_oracle_step(w, num_splits=1)
    for i in range(w.B):
        ckv, kpe = _gather(st, w, i)
        k = np.concatenate([ckv, kpe], axis=1)
        for h in range(w.H):
            q = np.concatenate([_f64_bf16(st["q_lat"][i, h]), _f64_bf16(st["q_pe_rot"][i, h])])
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q).reshape(1, 1, 1, -1), torch.from_numpy(k)[None, None],
                torch.from_numpy(ckv)[None, None], scale=w.softmax_scale).reshape(-1).numpy()
            ref_lse = torch.logsumexp(torch.from_numpy(w.softmax_scale * (k @ q)), 0).item()
            assert np.allclose(st["out"][i, h], ref, rtol=1e-12, atol=1e-12)
            assert abs(st["lse"][i, h] - ref_lse) < 1e-12


def test_mla_one_token_returns_the_latent():
    w = synth.custom_mla_workload("one", 5, [1, 1], 4)
    st = mla_oracle_step(w, num_splits=3)
    for i in range(2):
        ckv, _ = _gather(st, w, i)
        for h in range(4):
            assert np.array_equal(st["out"][i, h], ckv[0])
            assert np.array_equal(st["out_partial"][i, 0, h], ckv[0])
            assert np.all(st["lse_partial"][i, 1:, h] == -np.inf)


@pytest.mark.parametrize("S", [2, 3, 7])
def test_mla_split_merge_equals_single_pass(S):
    w = synth.custom_mla_workload("split", 7, [1, 64, 65, 500], 8)
    one = mla_oracle_step(w, num_splits=1)
    op, lp = oracle.mla_decode(one["q_lat"], one["q_pe_rot"], one["ckv_cache"], one["kpe_cache"],
                               one["block_tables"], one["seq_lens"], w.softmax_scale, S, w.ckv_scale)
    out, lse = oracle.lse_merge(op, lp)
    assert np.allclose(out, one["out"], rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, one["lse"], rtol=0, atol=1e-12)


def test_mla_per_sequence_splits_merge_to_the_single_pass_and_partition_the_pages():
    """A split count per sequence (reading of the local split-K): merged, it
    is the single pass; under equal scores (zero queries) a split's LSE is
    the log of its token count, the counts fill a prefix of the sequence's
    records, add up to its length and are whole 64-token pages but the last."""
    lens = [1, 64, 65, 500, 130]
    w = synth.custom_mla_workload("vsplit", 11, lens, 8)
    one = mla_oracle_step(w, num_splits=1)
    sp = np.array([1, 3, 2, 6, 0], np.int32)           # the last is clamped to 1
    S = 6
    args = (one["ckv_cache"], one["kpe_cache"], one["block_tables"], one["seq_lens"], w.softmax_scale, S,
            w.ckv_scale)
    op, lp = oracle.mla_decode(one["q_lat"], one["q_pe_rot"], *args, splits_per_seq=sp)
    out, lse = oracle.lse_merge(op, lp)
    assert np.allclose(out, one["out"], rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, one["lse"], rtol=0, atol=1e-12)
    z_lat, z_pe = np.zeros_like(one["q_lat"]), np.zeros_like(one["q_pe_rot"])
    _, lz = oracle.mla_decode(z_lat, z_pe, *args, splits_per_seq=sp)
    for b, L in enumerate(lens):
        sb = max(1, int(sp[b]))
        counts = [round(np.exp(x)) if x != -np.inf else 0 for x in lz[b, :, 0]]
        nz = [c for c in counts if c]
        assert sum(counts) == L and counts[:len(nz)] == nz and len(nz) <= sb
        assert all(c % 64 == 0 for c in nz[:-1])
        assert np.all(lz[b, sb:] == -np.inf)


def test_mla_page_permutation_invariance():
    w = synth.custom_mla_workload("perm", 9, [70, 200], 4)
    st = mla_oracle_step(w, num_splits=2)
    pool = st["ckv_cache"].shape[0]
    perm = np.argsort(synth.uniform(synth.stream_key(9, "perm2"), pool))
    c2 = np.empty_like(st["ckv_cache"]); k2 = np.empty_like(st["kpe_cache"])
    c2[perm] = st["ckv_cache"]; k2[perm] = st["kpe_cache"]
    bt2 = np.where(st["block_tables"] >= 0, perm[np.maximum(st["block_tables"], 0)], -1).astype(np.int32)
    op, lp = oracle.mla_decode(st["q_lat"], st["q_pe_rot"], c2, k2, bt2, st["seq_lens"], w.softmax_scale, 2,
                               w.ckv_scale)
    assert np.array_equal(op, st["out_partial"]) and np.array_equal(lp, st["lse_partial"])


def _rotate_f32(x, cs, interleaved):
    D = x.shape[-1]
    c, s = cs[: D // 2], cs[D // 2:]
    x1, x2 = (x[..., 0::2], x[..., 1::2]) if interleaved else (x[..., : D // 2], x[..., D // 2:])
    y1 = (x1 * c) - (x2 * s)
    y2 = (x2 * c) + (x1 * s)
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = y1, y2
    else:
        out[..., : D // 2], out[..., D // 2:] = y1, y2
    return out


def _bf16_bits(x32):
    return torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("style", ["interleaved", "neox"])
def test_mla_cache_write_bytes(style):
    w = synth.custom_mla_workload("wr", 13, [90], 3, style=style, rope_base=1e4)
    ckv, kpe = w.seq_latent(0)
    qlat, qpe = w.seq_q(0)
    L = 90
    pos = np.arange(L, dtype=np.int32)[::-1].copy()          # out of order
    slots = w.slots(0, np.arange(L))
    cs = w.cos_sin()
    cc = np.zeros((w.num_pages, w.page_size, w.Dc), np.uint8)
    kc = np.zeros((w.num_pages, w.page_size, w.Dr), np.uint16)
    q = np.broadcast_to(qpe, (L, w.H, w.Dr)).copy()
    assert oracle.mla_cache_write(q, ckv, kpe, pos, cs, cc, kc, slots, w.ckv_scale, style) == 0
    inter = style == "interleaved"
    # ckv: E4M3 of the float32 quotient (torch's float8 cast; |x / scale| < 448 here)
    z = (synth.bf16_bits_to_f32(ckv) / np.float32(w.ckv_scale)).astype(np.float32)
    assert np.abs(z).max() < 448
    want_c = torch.from_numpy(z).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    flat_c = cc.reshape(-1, w.Dc)
    flat_k = kc.reshape(-1, w.Dr)
    for t in range(L):
        assert np.array_equal(flat_c[slots[t]], want_c[t])
        yk = _rotate_f32(synth.bf16_bits_to_f32(kpe[t]), cs[pos[t]], inter)
        assert np.array_equal(flat_k[slots[t]], _bf16_bits(yk))
        yq = _rotate_f32(synth.bf16_bits_to_f32(qpe), cs[pos[t]], inter)
        assert np.array_equal(q[t], _bf16_bits(yq))
    # untouched slots stay zero
    used = np.zeros(flat_c.shape[0], bool); used[slots] = True
    assert not flat_c[~used].any() and not flat_k[~used].any()


def test_mla_cache_write_skips_bad_slots_and_positions():
    Dc, Dr = 512, 64
    ckv = np.full((3, Dc), 0x3F80, np.uint16)
    kpe = np.full((3, Dr), 0x3F80, np.uint16)
    cs = synth.cos_sin_table(4, Dr, 1e4)
    cc = np.zeros((2, 64, Dc), np.uint8); kc = np.zeros((2, 64, Dr), np.uint16)
    q = np.full((3, 2, Dr), 0x3F80, np.uint16)
    bad = oracle.mla_cache_write(q, ckv, kpe, np.array([0, 1, 9], np.int32), cs, cc, kc,
                                 np.array([-1, 128, 3], np.int32), 0.5)
    assert bad == 2
    assert not cc.any() and not kc.any()
    assert (q == 0x3F80).all()          # skipped tokens leave q_pe as it was
