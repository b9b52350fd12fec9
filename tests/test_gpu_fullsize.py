"""GPU parity at the benchmark's full workload sizes, on sampled sequences.

Each workload is filled and stepped on the GPU exactly as the benchmark runs
it (same split count from the library's heuristic, same launches). The
oracle then recomputes, from the same seeded inputs, the sampled sequences
(the longest, the shortest and two drawn at random): their cache bytes and
rotated q bit for bit, their partial records, merged outputs and LSEs within
tolerance. Every output of every sequence must also be finite and the error
word zero."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_04_gb300 import harness, synth
from tests._compare import assert_close_lse, assert_close_out, bf16_u16_to_f64
from tests._pipeline import oracle_step

pytestmark = pytest.mark.gpu


def _sample(w, n_random=2):
    L = w.seq_lens
    picks = [int(np.argmax(L)), int(np.argmin(L))]
    u = synth.uniform(synth.stream_key(w.seed, "sample"), n_random)
    picks += [int(x * w.B) for x in u]
    out = []
    for p in picks:
        if p not in out:
            out.append(p)
    return out


def _check(w, dw, seqs):
    st = oracle_step(w, seqs=seqs, num_splits=dw.num_splits)
    q = dw.bf16_u16(dw.decode_inputs["q"])
    out = bf16_u16_to_f64(dw.bf16_u16(dw.out))
    lse = dw.lse.cpu().numpy()
    op = dw.out_partial.cpu().numpy()
    lp = dw.lse_partial.cpu().numpy()
    for i, b in enumerate(seqs):
        assert np.array_equal(q[b], st["q_rot"][i]), f"q bytes of sequence {b}"
        n = int(w.pages_per_seq[b])
        pairs = [(dw.k_cache, st["k_cache"]), (dw.v_cache, st["v_cache"])]
        if dw.nvfp4:
            pairs += [(dw.k_block_scale, st["k_block_scale"]), (dw.v_block_scale, st["v_block_scale"])]
        for gc, oc in pairs:
            got = dw.cache_pages_u(gc, w.block_tables[b, :n])
            assert np.array_equal(got, oc[st["block_tables"][i, :n]]), f"cache bytes of sequence {b}"
        assert_close_out(op[b], st["out_partial"][i], f"out_partial[{b}]")
        assert_close_lse(lp[b], st["lse_partial"][i], f"lse_partial[{b}]")
        assert_close_out(out[b], st["out"][i], f"out[{b}]")
        assert_close_lse(lse[b], st["lse"][i], f"lse[{b}]")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert int(dw.err.item()) == 0


@pytest.fixture(scope="module")
def filled():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            w = synth.make_workload(name)
            dw = harness.DeviceWorkload(w)
            dw.fill()
            dw.upload_decode()
            cache[name] = (w, dw)
        return cache[name]
    yield get
    cache.clear()


@pytest.mark.parametrize("name", ["qwen", "longctx", "ragged", "fp8", "million", "fp4"])
def test_full_size_sampled(filled, name):
    w, dw = filled(name)
    dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    _check(w, dw, _sample(w))


@pytest.mark.parametrize("S", [16, 32, 48, 64])
def test_long_context_split_sweep(filled, S):
    w, dw = filled("longctx")
    dw.set_splits(S)
    dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    _check(w, dw, [0, 1])
