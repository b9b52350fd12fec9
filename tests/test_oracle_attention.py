"""Pins of the oracle's paged decode attention and LSE merge (CPU).

Checked against torch's float64 scaled-dot-product attention on gathered
contiguous K/V (a library routine), closed forms (a one-token context returns
V; equal scores return the mean of V with LSE = ln L; a split's LSE under
equal scores is the log of its token count), and invariants (physical page
permutation, split-K + merge = one pass, GQA = MHA with repeated K/V, NHD =
HND). (mainarch, decode-attention section: split-KV online softmax, tree
combine, paged KV with a deliberately shuffled layout, GQA sharing one KV
head; Loom Kernels, "Attention" row: paged MQA/GQA decode, local split-K/LSE
merge.)"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import synth
from tests._pipeline import cache_values_f64, oracle_step


def _gather(st, w, i, kvh):
    """Contiguous K, V (float64, dequantised) of sequence i, kv head kvh."""
    L = int(st["seq_lens"][i])
    P = w.page_size
    kv = []
    for cache, sc in ((st["k_cache"], w.k_scale), (st["v_cache"], w.v_scale)):
        vals = cache_values_f64(cache, w.cache_dtype)
        rows = []
        for t in range(L):
            page = st["block_tables"][i, t // P]
            rows.append(vals[page, kvh, t % P] if w.layout == "HND" else vals[page, t % P, kvh])
        a = np.array(rows).reshape(L, w.D)
        if sc is not None:
            a = a * float(sc[0] if sc.size == 1 else sc[kvh])
        kv.append(a)
    return kv


def _sdpa(q, k, v, scale):
    qt = torch.from_numpy(q).reshape(1, 1, 1, -1)
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).reshape(-1).numpy()
    lse = torch.logsumexp(torch.from_numpy(scale * (k @ q)), 0).item()
    return out, lse


CASES = [
    ("tiny", dict()),
    ("fp8_nhd", dict(seq_lens=[1, 17, 40], Hq=6, Hkv=2, D=64, layout="NHD", cache_dtype="fp8")),
    ("fp8_tensor_scale", dict(seq_lens=[33], Hq=4, Hkv=1, D=128, cache_dtype="fp8", per_head_scale=False)),
    ("interleaved_g7", dict(seq_lens=[16, 31, 50], Hq=14, Hkv=2, D=128, style="interleaved", rope_base=5e5)),
    ("mqa_g16", dict(seq_lens=[20, 3], Hq=16, Hkv=1, D=64, layout="NHD")),
]


def _workload(name, kw):
    if name == "tiny":
        return synth.make_workload("tiny")
    return synth.custom_workload(name, 77, **kw)


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_bruteforce_against_torch_sdpa(name, kw):
    w = _workload(name, kw)
    st = oracle_step(w, num_splits=1)
    for i in range(w.B):
        for h in range(w.Hq):
            k, v = _gather(st, w, i, h // w.G)
            q = synth.bf16_bits_to_f32(st["q_rot"][i, h]).astype(np.float64)
            ref, ref_lse = _sdpa(q, k, v, w.softmax_scale)
            assert np.allclose(st["out"][i, h], ref, rtol=1e-12, atol=1e-12)
            assert abs(st["lse"][i, h] - ref_lse) < 1e-12
            assert abs(st["lse_partial"][i, 0, h] - ref_lse) < 1e-12


def test_one_token_context_returns_v():
    for dt in ("bf16", "fp8"):
        w = synth.custom_workload("one", 5, [1, 1], 4, 2, 64, cache_dtype=dt)
        st = oracle_step(w, num_splits=3)
        for i in range(2):
            for h in range(4):
                _, v = _gather(st, w, i, h // 2)
                assert np.array_equal(st["out"][i, h], v[0])
                # split 0 holds the only page; the others are empty
                assert np.array_equal(st["out_partial"][i, 0, h], v[0])
                assert np.all(st["lse_partial"][i, 1:, h] == -np.inf)
                assert not st["out_partial"][i, 1:, h].any()


def test_equal_scores_give_mean_of_v_and_log_length():
    w = synth.custom_workload("eq", 6, [1, 15, 16, 17, 100], 4, 2, 64)
    st = oracle_step(w, num_splits=1)
    q0 = np.zeros_like(st["q_rot"])
    for S in (1, 2, 5):
        op, lp = oracle.paged_decode(q0, st["k_cache"], st["v_cache"], st["block_tables"], st["seq_lens"],
                                     w.softmax_scale, S, w.layout)
        out, lse = oracle.lse_merge(op, lp)
        for i, L in enumerate(st["seq_lens"]):
            for h in range(4):
                _, v = _gather(st, w, i, h // 2)
                assert np.allclose(out[i, h], v.mean(axis=0), rtol=1e-13, atol=1e-14)
                assert abs(lse[i, h] - math.log(L)) < 1e-13
                # a split's LSE is the log of its token count
                npages = -(-int(L) // 16)
                pps = -(-npages // S)
                for s in range(S):
                    n_s = max(0, min(int(L), (s + 1) * pps * 16) - s * pps * 16)
                    exp_l = math.log(n_s) if n_s else -np.inf
                    assert lp[i, s, h] == pytest.approx(exp_l, abs=1e-13) if n_s else lp[i, s, h] == -np.inf


def test_page_permutation_invariance():
    """Moving pages to other physical slots (block table rewritten) leaves
    the output bit-for-bit unchanged."""
    w = synth.custom_workload("perm", 9, [37, 100, 16], 4, 2, 64, layout="NHD")
    st = oracle_step(w, num_splits=2)
    pool = st["k_cache"].shape[0]
    perm = np.argsort(synth.uniform(synth.stream_key(9, "perm2"), pool))
    kc2 = np.empty_like(st["k_cache"]); vc2 = np.empty_like(st["v_cache"])
    kc2[perm] = st["k_cache"]; vc2[perm] = st["v_cache"]
    bt2 = np.where(st["block_tables"] >= 0, perm[np.maximum(st["block_tables"], 0)], -1).astype(np.int32)
    op, lp = oracle.paged_decode(st["q_rot"], kc2, vc2, bt2, st["seq_lens"], w.softmax_scale, 2, w.layout)
    assert np.array_equal(op, st["out_partial"]) and np.array_equal(lp, st["lse_partial"])


@pytest.mark.parametrize("S", [2, 3, 7, 64])
def test_split_merge_equals_single_pass(S):
    w = synth.custom_workload("split", 10, [1, 16, 17, 200, 333], 8, 2, 128, style="interleaved")
    st1 = oracle_step(w, num_splits=1)
    stS = oracle_step(w, num_splits=S)
    assert np.allclose(stS["out"], st1["out"], rtol=1e-12, atol=1e-13)
    assert np.allclose(stS["lse"], st1["lse"], rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv():
    G = 4
    w = synth.custom_workload("gqa", 11, [40, 77], 8, 2, 64)
    st = oracle_step(w, num_splits=2)
    kc, vc = st["k_cache"], st["v_cache"]          # HND [pages, Hkv, P, D]
    kc_m = np.repeat(kc, G, axis=1); vc_m = np.repeat(vc, G, axis=1)
    op, lp = oracle.paged_decode(st["q_rot"], kc_m, vc_m, st["block_tables"], st["seq_lens"], w.softmax_scale,
                                 2, "HND")
    assert np.array_equal(op, st["out_partial"]) and np.array_equal(lp, st["lse_partial"])


def test_layouts_agree():
    kw = dict(seq_lens=[5, 60], Hq=6, Hkv=3, D=64)
    a = oracle_step(synth.custom_workload("lay", 12, layout="HND", **kw), num_splits=2)
    b = oracle_step(synth.custom_workload("lay", 12, layout="NHD", **kw), num_splits=2)
    assert np.array_equal(a["k_cache"], b["k_cache"].transpose(0, 2, 1, 3))
    assert np.array_equal(a["out_partial"], b["out_partial"]) and np.array_equal(a["lse"], b["lse"])


def test_fp8_scale_enters_linearly():
    """Doubling k_scale doubles every score (LSE of scaled scores moves
    accordingly); doubling v_scale doubles the output."""
    w = synth.custom_workload("sc", 13, [45], 2, 1, 64, cache_dtype="fp8")
    st = oracle_step(w, num_splits=1)
    args = (st["q_rot"], st["k_cache"], st["v_cache"], st["block_tables"], st["seq_lens"], w.softmax_scale, 1,
            w.layout)
    o1, l1 = oracle.paged_decode(*args, k_scale=w.k_scale, v_scale=w.v_scale)
    o2, _ = oracle.paged_decode(*args, k_scale=w.k_scale, v_scale=2 * w.v_scale)
    assert np.allclose(o2, 2 * o1, rtol=1e-14, atol=0)
    # scores of one token: compare to the brute-force product
    k, _ = _gather(st, w, 0, 0)
    q = synth.bf16_bits_to_f32(st["q_rot"][0, 0]).astype(np.float64)
    _, lse_ref = _sdpa(q, k, k, w.softmax_scale)
    assert abs(l1[0, 0, 0] - lse_ref) < 1e-12


def test_merge_closed_forms():
    rng_o = synth.normal_f32(synth.stream_key(14, "o"), 2 * 4 * 3 * 8).astype(np.float64).reshape(2, 4, 3, 8)
    lse = np.log(np.array([1.0, 2.0, 3.0, 4.0]))[None, :, None] * np.ones((2, 4, 3))
    out, l = oracle.lse_merge(rng_o, lse)
    wts = np.array([1, 2, 3, 4]) / 10.0
    assert np.allclose(out, np.einsum("s,bshd->bhd", wts, rng_o), rtol=1e-14, atol=1e-15)
    assert np.allclose(l, math.log(10.0), atol=1e-15)
    # -inf splits contribute nothing; an all -inf row gives 0 and -inf
    lse2 = lse.copy(); lse2[:, 1:] = -np.inf
    out2, l2 = oracle.lse_merge(rng_o, lse2)
    assert np.array_equal(out2, rng_o[:, 0]) and np.allclose(l2, 0.0)
    out3, l3 = oracle.lse_merge(rng_o, np.full_like(lse, -np.inf))
    assert not out3.any() and np.all(l3 == -np.inf)


def test_bad_block_table_entry_is_left_out():
    w = synth.custom_workload("bad", 15, [48], 2, 1, 64)
    st = oracle_step(w, num_splits=1)
    bt = st["block_tables"].copy()
    bt[0, 1] = 10 ** 6          # page 1 (tokens 16..31) points outside the pool
    op, lp = oracle.paged_decode(st["q_rot"], st["k_cache"], st["v_cache"], bt, st["seq_lens"], w.softmax_scale,
                                 1, w.layout)
    k, v = _gather(st, w, 0, 0)
    keep = np.r_[0:16, 32:48]
    q = synth.bf16_bits_to_f32(st["q_rot"][0, 0]).astype(np.float64)
    ref, ref_lse = _sdpa(q, k[keep], v[keep], w.softmax_scale)
    assert np.allclose(op[0, 0, 0], ref, rtol=1e-12, atol=1e-13) and abs(lp[0, 0, 0] - ref_lse) < 1e-12


def test_empty_sequence():
    w = synth.custom_workload("empty", 16, [0, 5], 2, 1, 64)
    st = oracle_step(w, num_splits=2)
    assert not st["out"][0].any() and np.all(st["lse"][0] == -np.inf)
    assert np.all(np.isfinite(st["out"][1]))


# ---- a split count per sequence ------------------------------------------------------
# Loom Kernels, "Evidence" table, row "Local split-K paged decode": the split
# is local to each sequence. Reading: sequence b's pages are dealt into its
# own count S_b of page-granular splits (at most the call's record count S);
# its records past S_b are empty.

def test_per_sequence_splits_merge_to_the_single_pass():
    w = synth.custom_workload("vsplit", 21, [1, 16, 17, 200, 333, 64, 5], 8, 2, 128, style="interleaved")
    st1 = oracle_step(w, num_splits=1)
    S = 9
    sp = np.array([1, 3, 9, 5, 9, 2, 4], np.int32)
    op, lp = oracle.paged_decode(st1["q_rot"], st1["k_cache"], st1["v_cache"], st1["block_tables"],
                                 st1["seq_lens"], w.softmax_scale, S, w.layout, splits_per_seq=sp)
    out, lse = oracle.lse_merge(op, lp)
    assert np.allclose(out, st1["out"], rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, st1["lse"], rtol=0, atol=1e-12)
    # records past a sequence's own count are empty
    for b, sb in enumerate(sp):
        assert np.all(lp[b, sb:] == -np.inf) and not op[b, sb:].any()
    # a count of S for every sequence is the uniform call, bit for bit
    opu, lpu = oracle.paged_decode(st1["q_rot"], st1["k_cache"], st1["v_cache"], st1["block_tables"],
                                   st1["seq_lens"], w.softmax_scale, S, w.layout)
    opS, lpS = oracle.paged_decode(st1["q_rot"], st1["k_cache"], st1["v_cache"], st1["block_tables"],
                                   st1["seq_lens"], w.softmax_scale, S, w.layout,
                                   splits_per_seq=np.full(w.B, S, np.int32))
    assert np.array_equal(opu, opS) and np.array_equal(lpu, lpS)


def test_per_sequence_splits_partition_the_pages():
    """Under equal scores (q = 0) a split's LSE is the log of its token
    count. For every sequence the counts must: add up to L; be whole pages
    except in the last non-empty split; fill a prefix of at most S_b
    records; be equal except the last; and use the smallest equal page
    count with which S_b splits cover the sequence."""
    lens = [1, 15, 16, 17, 100, 160, 161, 333]
    w = synth.custom_workload("vpart", 22, lens, 4, 2, 64)
    st = oracle_step(w, num_splits=1)
    q0 = np.zeros_like(st["q_rot"])
    S = 7
    for sp in (np.array([1, 2, 7, 3, 7, 4, 6, 5], np.int32), np.array([0, 9, -3, 100, 1, 7, 2, 3], np.int32)):
        op, lp = oracle.paged_decode(q0, st["k_cache"], st["v_cache"], st["block_tables"], st["seq_lens"],
                                     w.softmax_scale, S, w.layout, splits_per_seq=sp)
        for b, L in enumerate(lens):
            sb = min(max(int(sp[b]), 1), S)   # the stated clamp
            counts = [round(math.exp(x)) if x != -np.inf else 0 for x in lp[b, :, 0]]
            for x, c in zip(lp[b, :, 0], counts):
                if c:
                    assert x == pytest.approx(math.log(c), abs=1e-12)
            assert sum(counts) == L
            nz = [c for c in counts if c]
            k = len(nz)
            assert counts[:k] == nz and not any(counts[k:])          # a prefix of the records
            assert k <= sb and k <= -(-L // 16)
            assert all(c % 16 == 0 for c in nz[:-1])                # whole pages but the last
            if k > 1:
                p = nz[0] // 16                                     # pages per split
                assert all(c == 16 * p for c in nz[:-1])
                npages = -(-L // 16)
                assert (p - 1) * sb < npages <= p * sb              # the smallest such count
