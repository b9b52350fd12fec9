"""The bounded in-kernel waits behind PKV_FLAG_WAIT_TIMEOUT, made to run out
on purpose by pkv_selftest_bounded_wait (mbarriers that nothing completes):
the kernel gives up after its limit, reports the flag, stops a second
waiter through the CTA's abort signal, and the GPU context stays usable
(a decode step afterwards is still correct)."""
import pytest
import torch

from paged_kv_gqa_04_gb300 import _abi, harness, synth
from tests._pipeline import oracle_step
from tests._compare import assert_close_out, bf16_u16_to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [1, 5])
def test_wait_gives_up_and_reports(limit_ms):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    _abi.selftest_bounded_wait(limit_ms * 1_000_000, err, elapsed)
    torch.cuda.synchronize()
    assert int(err.item()) == _abi.FLAG_WAIT_TIMEOUT
    t0, t1 = (int(x) / 1e6 for x in elapsed.cpu())
    assert limit_ms <= t0 < limit_ms + 2.0                  # gave up at its limit (retries suspend <= 100 us)
    assert t1 < t0 + 1.0                                     # the second waiter (limit 100x) stopped on the abort signal


def test_context_usable_after_timeouts():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    for _ in range(3):
        _abi.selftest_bounded_wait(1_000_000, err, elapsed)
    torch.cuda.synchronize()
    w = synth.make_workload("tiny")
    dw = harness.DeviceWorkload(w, num_splits=2)
    dw.fill()
    dw.upload_decode()
    dw.step()
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0
    st = oracle_step(w, num_splits=2)
    assert_close_out(bf16_u16_to_f64(dw.bf16_u16(dw.out)), st["out"], "out")
