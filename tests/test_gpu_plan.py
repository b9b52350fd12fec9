"""GPU parity of the decode under a split plan (a split count per
sequence: pkv_plan_splits, pkv_paged_gqa_decode_planned,
pkv_lse_merge_planned) against the float64 oracle with the same per-sequence
counts (oracle.paged_decode(..., splits_per_seq=...)).

Each written record (sequence b, split s < S_b) is compared element by
element, then the merged output and LSE, within tests/_compare.py's
tolerance. Plans are the library's own (automatic and with fixed page
targets), so sequences split into 1 to many splits, ragged last pages and
single-page splits all occur; bf16, FP8 and NVFP4 caches, both layouts,
groups of 1 to 16. (Loom Kernels, "Evidence" table, row "Local split-K
paged decode".)"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import _abi, harness, synth
from tests._compare import assert_close_lse, assert_close_out, bf16_u16_to_f64
from tests._pipeline import oracle_step

pytestmark = pytest.mark.gpu


def _case(name, targets, **kw):
    return pytest.param(name, targets, kw, id=name)


CASES = [
    _case("bf16_hnd_d128_g6_mixed", (0, 1, 3, 7), seq_lens=[1, 16, 17, 31, 33, 100, 257, 600], Hq=12, Hkv=2,
          D=128, rope_base=1e6, k_mult=0.5),
    _case("bf16_nhd_d128_g4_interleaved", (0, 2, 5), seq_lens=[5, 48, 130, 700, 2], Hq=16, Hkv=4, D=128,
          layout="NHD", style="interleaved", rope_base=5e5, outlier_p=0.05),
    _case("fp8_hnd_d128_g6", (0, 4), seq_lens=[15, 16, 17, 200, 999], Hq=12, Hkv=2, D=128, cache_dtype="fp8",
          rope_base=1e6),
    _case("fp8_nhd_d64_g2", (0, 1), seq_lens=[3, 70, 300], Hq=4, Hkv=2, D=64, layout="NHD", cache_dtype="fp8",
          per_head_scale=False),
    _case("bf16_hnd_d64_g16", (0, 3), seq_lens=[40, 9, 400], Hq=16, Hkv=1, D=64),
    _case("empty_and_short", (0, 2), seq_lens=[0, 1, 20, 0], Hq=8, Hkv=2, D=128),
    _case("nvfp4_hnd_d128_g6", (0, 1, 3), seq_lens=[1, 15, 16, 17, 33, 257, 800], Hq=12, Hkv=2, D=128,
          cache_dtype="nvfp4", rope_base=1e6),
    _case("nvfp4_hnd_d64_g16", (0, 2), seq_lens=[40, 9, 300], Hq=16, Hkv=1, D=64, cache_dtype="nvfp4"),
]


def _oracle_planned(w, st, sp, nrec):
    args = (st["q_rot"], st["k_cache"], st["v_cache"])
    if w.cache_dtype == "nvfp4":
        op, lp = oracle.paged_decode_nvfp4(*args, st["k_block_scale"], st["v_block_scale"], st["block_tables"],
                                           st["seq_lens"], w.softmax_scale, nrec, w.layout, w.k_scale, w.v_scale,
                                           splits_per_seq=sp)
    else:
        op, lp = oracle.paged_decode(*args, st["block_tables"], st["seq_lens"], w.softmax_scale, nrec, w.layout,
                                     w.k_scale, w.v_scale, splits_per_seq=sp)
    return op, lp


def _check_planned(w, dw, seqs=None):
    """Compare the planned step's records and merged output with the oracle
    for the given sequences (all by default)."""
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    sp_all, _ = dw.plan_host
    st = oracle_step(w, seqs=seqs, num_splits=1)
    sp = sp_all[seqs]
    nrec = dw.num_splits
    op, lp = _oracle_planned(w, st, sp, nrec)
    out, lse = oracle.lse_merge(op, lp)
    gop = dw.out_partial.cpu().numpy()
    glp = dw.lse_partial.cpu().numpy()
    for i, b in enumerate(seqs):
        n = int(sp[i])
        assert_close_out(gop[b, :n], op[i, :n], f"out_partial of sequence {b}")
        assert_close_lse(glp[b, :n], lp[i, :n], f"lse_partial of sequence {b}")
    gout = bf16_u16_to_f64(dw.bf16_u16(dw.out))[seqs]
    assert_close_out(gout, out, "out")
    assert_close_lse(dw.lse.cpu().numpy()[seqs], lse, "lse")


@pytest.mark.parametrize("name,targets,kw", CASES)
def test_planned_decode_parity(name, targets, kw):
    w = synth.custom_workload(name, 131, **kw)
    dw = harness.DeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    d = dw.decode_inputs
    for T in targets:
        dw.set_plan(target_pages=T)
        sp, work = dw.plan_host
        # the plan itself: every (b, s < S_b) once, longest items first
        items = sorted((int(e) >> 12, int(e) & 0xFFF) for e in work[:, 0])
        assert items == [(b, s) for b in range(w.B) for s in range(int(sp[b]))]
        d["q"].copy_(d["q0"])
        dw.err.zero_()
        dw.step()
        torch.cuda.synchronize()
        assert int(dw.err.item()) == 0
        _check_planned(w, dw)


@pytest.mark.parametrize("name", ["qwen", "ragged", "fp8", "fp4"])
def test_planned_decode_full_size_sampled(name):
    """The library's automatic plan on a full-size workload; sequences at
    evenly spaced length quantiles (the longest included) checked."""
    w = synth.make_workload(name)
    dw = harness.DeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    dw.set_plan()
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    order = np.argsort(w.seq_lens, kind="stable")
    seqs = sorted({int(order[int(q * (w.B - 1))]) for q in (0.0, 0.3, 0.7, 1.0)})
    _check_planned(w, dw, seqs)


def test_plan_from_other_lengths_stays_correct():
    """A plan made from other lengths than the device's seq_lens: the page
    ranges follow the device lengths, so the merged output is still the
    attention over every token."""
    w = synth.custom_workload("stale", 132, [300, 40, 1000], 8, 2, 128)
    dw = harness.DeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    props = torch.cuda.get_device_properties(0)
    sp, nrec, work = _abi.plan_splits(np.array([20, 900, 16], np.int32), w.Hkv, w.Hq, w.D, w.max_pages, "bf16",
                                      props.multi_processor_count, 4095, 4)
    dw.set_splits(nrec)
    dw.plan_host = (sp, work)
    dw.splits_per_seq = torch.from_numpy(sp).cuda()
    dw.work = torch.from_numpy(np.ascontiguousarray(work)).cuda()
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    _check_planned(w, dw)


def test_bad_plan_entries_are_flagged_and_skipped():
    """Work items outside the batch or the records, and split counts outside
    [1, S], set PKV_FLAG_PLAN_RANGE; nothing faults and the valid items are
    still computed (the merge clamps the counts)."""
    w = synth.custom_workload("badplan", 133, [100, 50], 4, 2, 64)
    dw = harness.DeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    dw.set_plan(target_pages=2)
    sp, work = dw.plan_host
    bad = np.concatenate([work, np.array([[(7 << 12) | 0, 0], [(0 << 12) | 4000, 0], [-5, -9]], np.int32)])
    dw.work = torch.from_numpy(bad).cuda()
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == _abi.FLAG_PLAN_RANGE
    _check_planned(w, dw)
    # a split count of 0 is taken as 1 (and flagged)
    sp0 = sp.copy()
    sp0[1] = 0
    dw.splits_per_seq = torch.from_numpy(sp0).cuda()
    dw.err.zero_()
    dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) & _abi.FLAG_PLAN_RANGE


def test_planned_steps_back_to_back_and_as_graphs_match_one_step():
    """Planned steps issued back to back, and the CUDA-graph forms of the
    planned step (device inputs, and host inputs with the plan copied in
    with them), give results bit-identical to one synchronised step."""
    w = synth.custom_workload("b2bplan", 134, [700, 33, 1500, 250, 2], 12, 2, 128, rope_base=1e6)
    dw = harness.DeviceWorkload(w)
    dw.fill()
    d = dw.upload_decode()
    dw.set_plan(target_pages=9)
    dw.step()
    torch.cuda.synchronize()
    nrec = dw.splits_per_seq.cpu().numpy()
    ref_out, ref_lse = dw.bf16_u16(dw.out), dw.lse.cpu().numpy()
    ref_op = [dw.out_partial[b, :int(nrec[b])].cpu().numpy() for b in range(w.B)]

    def same():
        assert np.array_equal(dw.bf16_u16(dw.out), ref_out)
        assert np.array_equal(dw.lse.cpu().numpy(), ref_lse)
        for b in range(w.B):
            assert np.array_equal(dw.out_partial[b, :int(nrec[b])].cpu().numpy(), ref_op[b])

    for _ in range(5):
        d["q"].copy_(d["q0"])
        dw.step()
    torch.cuda.synchronize()
    same()
    g = harness.StepGraph(dw)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    same()
    dw.out.zero_()
    g2 = harness.StepGraph(dw, host_io=True)
    g2.replay()
    torch.cuda.synchronize()
    same()
    assert np.array_equal(g2.out_h.view(torch.int16).numpy().view(np.uint16), ref_out)
    assert int(dw.err.item()) == 0


# ---- split plans of the MLA decode -----------------------------------------------------
from tests._pipeline import mla_oracle_step  # noqa: E402

MLA_CASES = [
    pytest.param("mla_tiny", (0, 2, 4), {}, id="mla_tiny"),
    pytest.param("ragged_h16", (0, 2, 6), dict(seq_lens=[1, 63, 64, 65, 200, 900, 0], H=16, style="neox"),
                 id="ragged_h16"),
    pytest.param("h5", (0, 4), dict(seq_lens=[100, 257, 1500], H=5), id="h5"),
]


def _check_mla_planned(w, dw, seqs=None):
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    sp_all, _ = dw.plan_host
    st = mla_oracle_step(w, seqs=seqs, num_splits=1)
    sp = sp_all[seqs]
    op, lp = oracle.mla_decode(st["q_lat"], st["q_pe_rot"], st["ckv_cache"], st["kpe_cache"], st["block_tables"],
                               st["seq_lens"], w.softmax_scale, dw.num_splits, w.ckv_scale, splits_per_seq=sp)
    out, lse = oracle.lse_merge(op, lp)
    gop = dw.out_partial.cpu().numpy()
    glp = dw.lse_partial.cpu().numpy()
    for i, b in enumerate(seqs):
        n = int(sp[i])
        assert_close_out(gop[b, :n], op[i, :n], f"out_partial of sequence {b}")
        assert_close_lse(glp[b, :n], lp[i, :n], f"lse_partial of sequence {b}")
    assert_close_out(bf16_u16_to_f64(dw.bf16_u16(dw.out))[seqs], out, "out")
    assert_close_lse(dw.lse.cpu().numpy()[seqs], lse, "lse")


@pytest.mark.parametrize("name,targets,kw", MLA_CASES)
def test_planned_mla_decode_parity(name, targets, kw):
    w = synth.make_mla_workload("mla_tiny") if name == "mla_tiny" else synth.custom_mla_workload(name, 135, **kw)
    dw = harness.MlaDeviceWorkload(w, num_splits=1)
    dw.fill()
    dw.upload_decode()
    d = dw.decode_inputs
    for T in targets:
        dw.set_plan(target_pages=T)
        sp, work = dw.plan_host
        items = sorted((int(e) >> 12, int(e) & 0xFFF) for e in work[:, 0])
        assert items == [(b, s) for b in range(w.B) for s in range(int(sp[b]))]
        d["q"].copy_(d["q0"])
        dw.err.zero_()
        dw.step()
        torch.cuda.synchronize()
        assert int(dw.err.item()) == 0
        _check_mla_planned(w, dw)


@pytest.mark.parametrize("name", ["mla", "mla_batch"])
def test_planned_mla_decode_full_size_sampled(name):
    """The automatic MLA plan on a full-size workload (mla: 200 records of
    one sequence, merged by the two-level tree)."""
    w = synth.make_mla_workload(name)
    dw = harness.MlaDeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    dw.set_plan()
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    L = w.seq_lens
    _check_mla_planned(w, dw, sorted({int(np.argmax(L)), int(np.argmin(L)), int(w.B // 2)}))


def test_bad_mla_plan_entries_are_flagged_and_skipped():
    w = synth.custom_mla_workload("badmla", 136, [300, 100], 4)
    dw = harness.MlaDeviceWorkload(w, num_splits=1)
    dw.fill()
    dw.upload_decode()
    dw.set_plan(target_pages=2)
    sp, work = dw.plan_host
    bad = np.concatenate([work, np.array([[(9 << 12) | 0, 0], [(1 << 12) | 4000, 0], [-7, 0]], np.int32)])
    dw.work = torch.from_numpy(bad).cuda()
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == _abi.FLAG_PLAN_RANGE
    _check_mla_planned(w, dw)
    # a split count of 0 is taken as 1 (and flagged)
    sp0 = sp.copy()
    sp0[1] = 0
    dw.splits_per_seq = torch.from_numpy(sp0).cuda()
    dw.err.zero_()
    dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) & _abi.FLAG_PLAN_RANGE


def test_large_batch_of_short_sequences_uniform_and_planned():
    """8,192 sequences of 0 to 80 tokens (grids of 8,192 x S x Hkv CTAs for
    the uniform launch and a work list of about 8,000 items under a plan):
    sampled sequences, including empty and one-token ones, against the
    oracle in both forms."""
    rng = np.random.default_rng(137)
    lens = rng.integers(0, 81, 8192).astype(np.int32)
    lens[:4] = [0, 1, 16, 17]
    w = synth.custom_workload("bigbatch", 137, lens, 8, 2, 128)
    dw = harness.DeviceWorkload(w, num_splits=2)
    dw.fill()
    d = dw.upload_decode()
    seqs = sorted({0, 1, 2, 3, 4097, 8191, int(np.argmax(lens))})
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    st = oracle_step(w, seqs=seqs, num_splits=2)
    out = bf16_u16_to_f64(dw.bf16_u16(dw.out))
    assert_close_out(out[seqs], st["out"], "out (uniform)")
    assert_close_lse(dw.lse.cpu().numpy()[seqs], st["lse"], "lse (uniform)")
    dw.set_plan(target_pages=2)
    d["q"].copy_(d["q0"])
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    _check_planned(w, dw, seqs)
