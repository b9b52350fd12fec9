"""GPU parity of the MLA decode step (latent-cache write, paged MLA decode,
D = 512 merge) against the float64 oracle, through the C ABI.

Compared: rotated q_pe and every ckv / kpe cache byte bit for bit; partial
outputs, merged output and LSE within the tolerance of tests/_compare.py.
Cases span ragged last pages and chunks (a page is two 32-token chunks),
empty sequences and splits, 1 to 16 heads (one and two head tiles, counts
that are not multiples of 8), both RoPE styles, split counts past 32 (the
merge's tree path at D = 512), and the full-size workloads on sampled
sequences."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_04_gb300 import _abi, harness, synth
from tests._compare import assert_close_lse, assert_close_out, bf16_u16_to_f64
from tests._pipeline import mla_oracle_step

pytestmark = pytest.mark.gpu


def _case(name, S_list, **kw):
    return pytest.param(name, S_list, kw, id=name)


CASES = [
    _case("mla_tiny", (1, 2, 5)),
    _case("ragged_h16_neox", (1, 3), seq_lens=[1, 31, 32, 33, 63, 64, 65, 200], H=16, style="neox"),
    _case("h1", (1, 4), seq_lens=[130, 7], H=1),
    _case("h5_h13", (2,), seq_lens=[100, 257], H=5),
    _case("h13", (3,), seq_lens=[100, 257], H=13),
    _case("empty_and_short", (4,), seq_lens=[0, 1, 2, 33], H=8),
    _case("many_splits_tree_merge", (40, 64), seq_lens=[4100], H=8),
    # the schedule: batches up to 64 are ordered by length (B > 32: two rank
    # keys per lane, with ties and empty sequences), larger ones round-robin
    _case("b40_length_order", (1, 3), seq_lens=[(37 * i) % 400 if i % 7 else 200 for i in range(40)], H=4),
    _case("b70_round_robin", (2,), seq_lens=[(53 * i) % 300 for i in range(70)], H=2),
]


def _workload(name, kw):
    return synth.make_mla_workload("mla_tiny") if name == "mla_tiny" else synth.custom_mla_workload(name, 303, **kw)


def _compare(w, dw, st, seqs):
    q = dw.bf16_u16(dw.decode_inputs["q"])
    out = bf16_u16_to_f64(dw.bf16_u16(dw.out))
    lse = dw.lse.cpu().numpy()
    op = dw.out_partial.cpu().numpy()
    lp = dw.lse_partial.cpu().numpy()
    for i, b in enumerate(seqs):
        assert np.array_equal(q[b], st["q_pe_rot"][i]), f"q_pe bytes of sequence {b}"
        n = int(w.pages_per_seq[b])
        if n:
            for gc, oc in ((dw.ckv_cache, st["ckv_cache"]), (dw.kpe_cache, st["kpe_cache"])):
                got = dw.cache_pages_u(gc, w.block_tables[b, :n])
                want = oc[st["block_tables"][i, :n]]
                # only the rows the sequence wrote are defined (a page's tail past L is not)
                L = int(w.seq_lens[b])
                got = got.reshape(n * w.page_size, -1)[:L]
                want = want.reshape(n * w.page_size, -1)[:L]
                assert np.array_equal(got, want), f"cache bytes of sequence {b}"
        assert_close_out(op[b], st["out_partial"][i], f"out_partial[{b}]")
        assert_close_lse(lp[b], st["lse_partial"][i], f"lse_partial[{b}]")
        assert_close_out(out[b], st["out"][i], f"out[{b}]")
        assert_close_lse(lse[b], st["lse"][i], f"lse[{b}]")
    assert np.isfinite(out).all()
    assert int(dw.err.item()) == 0


@pytest.mark.parametrize("name,S_list,kw", CASES)
def test_mla_step_parity(name, S_list, kw):
    w = _workload(name, kw)
    dw = harness.MlaDeviceWorkload(w, num_splits=S_list[0])
    dw.fill()
    dw.upload_decode()
    for S in S_list:
        dw.set_splits(S)
        dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
        dw.err.zero_()
        dw.step()
        torch.cuda.synchronize()
        _compare(w, dw, mla_oracle_step(w, num_splits=S), list(range(w.B)))


@pytest.mark.parametrize("name", ["mla", "mla_batch"])
def test_mla_full_size_sampled(name):
    w = synth.make_mla_workload(name)
    dw = harness.MlaDeviceWorkload(w)
    dw.fill()
    dw.upload_decode()
    dw.step()
    torch.cuda.synchronize()
    L = w.seq_lens
    seqs = sorted({int(np.argmax(L)), int(np.argmin(L)), int(w.B // 2)})
    _compare(w, dw, mla_oracle_step(w, seqs=seqs, num_splits=dw.num_splits), seqs)


def test_mla_fill_in_one_call_two_tokens_per_thread():
    """One cache-write call over every context token of the mla_batch
    workload (319,783 tokens: from 131,072 tokens on, the launcher gives each
    thread two tokens) writes the oracle's bytes; sampled sequences include
    the last one (the ragged end of the grid)."""
    w = synth.make_mla_workload("mla_batch")
    dw = harness.MlaDeviceWorkload(w)
    fi = dw.fill_inputs()
    assert int(fi["positions"].numel()) >= 131072
    dw.err.zero_()
    dw.write_fill(fi)
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    L = w.seq_lens
    seqs = sorted({0, int(w.B // 2), int(w.B - 1), int(np.argmax(L))})
    st = mla_oracle_step(w, seqs=seqs, num_splits=1)
    for i, b in enumerate(seqs):
        n = int(w.pages_per_seq[b])
        for gc, oc in ((dw.ckv_cache, st["ckv_cache"]), (dw.kpe_cache, st["kpe_cache"])):
            got = dw.cache_pages_u(gc, w.block_tables[b, :n]).reshape(n * w.page_size, -1)[:int(L[b]) - 1]
            want = oc[st["block_tables"][i, :n]].reshape(n * w.page_size, -1)[:int(L[b]) - 1]
            assert np.array_equal(got, want), f"cache bytes of sequence {b}"


def test_mla_bad_page_and_seq_len_are_flagged():
    w = synth.custom_mla_workload("bad", 17, [200, 100], 8, num_pages=8)
    dw = harness.MlaDeviceWorkload(w, num_splits=2)
    dw.fill()
    dw.upload_decode()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    bt = dw.block_tables.clone()
    bt[0, 1] = w.num_pages + 3           # a page the first sequence needs
    dw.block_tables.copy_(bt)
    dw.err.zero_()
    dw.decode(dw.decode_inputs["q"])
    torch.cuda.synchronize()
    assert int(dw.err.item()) == _abi.FLAG_PAGE_RANGE
    dw.block_tables.copy_(torch.from_numpy(w.block_tables).cuda())
    sl = dw.seq_lens.clone()
    sl[1] = 64 * w.block_tables.shape[1] + 1
    dw.seq_lens.copy_(sl)
    dw.err.zero_()
    dw.decode(dw.decode_inputs["q"])
    torch.cuda.synchronize()
    assert int(dw.err.item()) & _abi.FLAG_SEQ_LEN_RANGE
    assert torch.isfinite(dw.out_partial).all()


@pytest.mark.parametrize("pad_lat,pad_pe", [(2, 0), (0, 2), (2, 2)])
def test_mla_padded_query_rows(pad_lat, pad_pe):
    """Query rows padded by two elements are 4-byte but not 16-byte aligned,
    which sends the kernel's query staging to its word-load path: the
    partial outputs equal those of contiguous queries bit for bit (and the
    oracle, checked on the contiguous run)."""
    w = synth.custom_mla_workload("padded_q", 305, [300, 129, 64], 12)
    dw = harness.MlaDeviceWorkload(w, num_splits=2)
    dw.fill()
    dw.upload_decode()
    dw.step()
    torch.cuda.synchronize()
    _compare(w, dw, mla_oracle_step(w, num_splits=2), list(range(w.B)))
    op0, lp0 = dw.out_partial.clone(), dw.lse_partial.clone()

    def padded(t, pad):
        if pad == 0:
            return t
        p = torch.zeros(*t.shape[:-1], t.shape[-1] + pad, dtype=t.dtype, device=t.device)
        p[..., :t.shape[-1]] = t
        return p[..., :t.shape[-1]]

    ql, qp = dw.decode_inputs["q_lat"], dw.decode_inputs["q"]  # q_pe as rotated by the write
    dw.decode_inputs["q_lat"] = padded(ql, pad_lat)
    q_pe = padded(qp, pad_pe)
    assert dw.decode_inputs["q_lat"].stride(1) % 8 == pad_lat % 8 and q_pe.stride(1) % 8 == pad_pe % 8
    dw.out_partial.fill_(float("nan"))
    dw.lse_partial.fill_(float("nan"))
    dw.decode(q_pe)
    torch.cuda.synchronize()
    dw.decode_inputs["q_lat"] = ql
    assert torch.equal(dw.out_partial, op0) and torch.equal(dw.lse_partial, lp0)
    assert int(dw.err.item()) == 0
