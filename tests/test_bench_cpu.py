"""CPU tests of the benchmark's host logic: the CPU-baseline samples keep
the batch's mix of lengths and stay within their work bound, both arms
describe the same configuration, and the statistics are what they say."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from paged_kv_gqa_04_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("name", ["ragged", "qwen", "fp8", "longctx", "million"])
def test_quantile_sample_spans_the_length_distribution(name):
    w = synth.make_workload(name)
    for n in (1, 3, 16, w.B, w.B + 5):
        seqs = bench.quantile_sample(w, n)
        k = min(n, w.B)
        assert len(seqs) == len(set(seqs)) == k and seqs == sorted(seqs)
        assert all(0 <= b < w.B for b in seqs)
        L = np.sort(w.seq_lens)
        got = np.sort(w.seq_lens[seqs])
        # the i-th smallest sampled length is the batch's length at quantile (i + 1/2) / k
        for i, x in enumerate(got):
            assert x == L[min(w.B - 1, int((i + 0.5) * w.B / k))]


def test_cpu_sample_respects_its_work_bound():
    for name in ["ragged", "qwen", "fp8", "longctx", "million"]:
        w = synth.make_workload(name)
        for budget in (1e8, 2e9):
            seqs = bench.cpu_sample(w, 16, budget)
            assert 1 <= len(seqs) <= 16
            if len(seqs) > 1:
                assert sum(bench.seq_flops(w, b) for b in seqs) <= budget


def test_both_arms_describe_the_same_configuration():
    w = synth.make_workload("ragged")
    a = bench.workload_config(w, "ragged")
    b = bench.workload_config(w, "ragged")
    assert a == b and a["batch"] == 256 and a["context_tokens"] == int(w.seq_lens.sum())
    assert bench.WORKLOAD_TEXT["ragged"].startswith("ragged large-batch decode: B256")


def test_stats_of_a_known_series():
    s = bench.stats([1.0, 2.0, 3.0, 4.0])  # milliseconds
    assert s["mean"] == pytest.approx(2500.0) and s["median"] == pytest.approx(2500.0)
    assert s["min"] == pytest.approx(1000.0) and s["max"] == pytest.approx(4000.0) and s["n"] == 4
    assert s["p10"] == pytest.approx(1300.0) and s["p90"] == pytest.approx(3700.0)


def test_byte_counts_of_the_roofline():
    """Decode bytes: Q + K/V + block-table entries + output; the cache fill
    counts each distinct position's cos/sin row once when asked."""
    w = synth.make_workload("ragged")
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    kv = int(w.seq_lens.astype(np.int64).sum()) * Hkv * D * 2 * 2
    expect = B * Hq * D * 2 + kv + int(w.pages_per_seq.sum()) * 4 + B * Hq * D * 2
    assert bench.decode_alg_bytes(w) == expect
    T, rows = 1000, 10
    per = 2 * Hkv * D * 2 + 2 * Hkv * D * 2 + 8
    assert bench.write_alg_bytes(w, T, False) == T * per + T * D * 4
    assert bench.write_alg_bytes(w, T, False, rows) == T * per + rows * D * 4


def test_launch_mean_leaves_out_host_stalls_only():
    m, out = bench.launch_mean([0.25, 0.26, 0.255, 61.3, 0.25])
    assert out == 1 and abs(m - 0.25375) < 1e-12
    m, out = bench.launch_mean([1.0, 1.9, 1.5])       # within twice the median: all kept
    assert out == 0 and abs(m - 1.4666666666666666) < 1e-12
