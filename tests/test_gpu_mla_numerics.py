"""GPU parity of the MLA decode on inputs aimed at its FP8 operand forms and
its online softmax, against the float64 oracle through the C ABI.

* Rising scores: the latent rows of head 0 follow its query's sign pattern
  with a weight that ramps up along the sequence (and those of head 1 the
  opposite pattern), so head 0's running maximum grows by far more than 8
  (log2 units) from one 128-token chunk to the next: the kernel must
  rescale its tensor-memory accumulator every chunk; head 1's maximum is at
  the start and never moves.
* Query dynamic range: heads whose 512 latent query values span 2^-30 .. 2
  (most far below the largest, where the two-term E4M3 form of the query
  loses its exactness), a head of values near 2^-40 (a large power-of-two
  scale), an all-zero head, one of larger values, the rest normal.
The inputs are drawn by the workload's own seeded generators (subclassed
here), so the oracle and the GPU see the same bytes."""
import dataclasses

import numpy as np
import pytest
import torch

from paged_kv_gqa_04_gb300 import harness, synth
from tests._pipeline import mla_oracle_step
from tests.test_gpu_mla import _compare

pytestmark = pytest.mark.gpu


def _bf16(x: np.ndarray) -> np.ndarray:
    return synth.f32_to_bf16_trunc(np.asarray(x, np.float32))


class _RampWorkload(synth.MlaWorkload):
    """Latent rows = r_t (sign(q_lat[0]) - sign(q_lat[1])) + noise, r_t
    rising from 0 to 2 along each sequence."""

    def seq_latent(self, b):
        L = int(self.seq_lens[b])
        ql, _ = super().seq_q(b)
        qv = (ql.astype(np.uint32) << 16).view(np.float32).reshape(self.H, self.Dc)
        u = np.sign(qv[0]) - np.sign(qv[1])
        r = 2.0 * np.arange(L, dtype=np.float64) / max(L, 1)
        noise = synth.normal_f32(synth.stream_key(self.seed, "ramp", b), L * self.Dc).reshape(L, self.Dc)
        ckv = r[:, None] * u[None, :] + 0.3 * noise
        kpe = synth.normal_f32(synth.stream_key(self.seed, "kpe", b), L * self.Dr).reshape(L, self.Dr)
        return _bf16(ckv), _bf16(kpe)


class _RangeWorkload(synth.MlaWorkload):
    """Per-head query scales and spreads chosen to stress the query's FP8
    form (see the module docstring)."""

    def seq_q(self, b):
        ql, qp = super().seq_q(b)
        qv = (ql.astype(np.uint32) << 16).view(np.float32).reshape(self.H, self.Dc).astype(np.float64)
        spread = synth.uniform(synth.stream_key(self.seed, "spread", b), self.H * self.Dc).reshape(self.H, self.Dc)
        for h in range(self.H):
            if h % 5 == 0:      # values spanning 2^-30 .. 2
                qv[h] = qv[h] * np.exp2(-30.0 * spread[h])
                qv[h, h % self.Dc] = 2.0
            elif h % 5 == 1:    # a tiny head
                qv[h] = qv[h] * 2.0 ** -40
            elif h % 5 == 2:    # all zero
                qv[h] = 0.0
            elif h % 5 == 3:    # larger values
                qv[h] = qv[h] * 4.0
        return _bf16(qv), qp


def _run(w, S_list):
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


def _as(cls, w):
    return cls(**{f.name: getattr(w, f.name) for f in dataclasses.fields(w)})


def _chunk_maxima_log2(w, b, h):
    """Head h's score maximum (log2 units, the positional part left out)
    over each 128-token chunk of sequence b, from the inputs."""
    ckv, _ = w.seq_latent(b)
    ql, _ = w.seq_q(b)
    c = (ckv.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qh = (ql[h].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    s = c @ qh * w.softmax_scale / np.log(2.0)
    return [s[i:i + 128].max() for i in range(0, len(s), 128)]


@pytest.mark.parametrize("H", [8, 16])
def test_mla_rescale_every_chunk(H):
    w = _as(_RampWorkload, synth.custom_mla_workload("ramp", 411, [700, 300], H, ckv_scale=0.02))
    m = _chunk_maxima_log2(w, 0, 0)
    full = m[:700 // 128]  # the full chunks of the 700-token sequence
    assert all(y - x > 10.0 for x, y in zip(full, full[1:])), m  # each moves head 0's reference maximum
    _run(w, (1, 3))


def test_mla_query_dynamic_range():
    w = _as(_RangeWorkload, synth.custom_mla_workload("qrange", 412, [450, 129, 64], 16))
    _run(w, (1, 2))
