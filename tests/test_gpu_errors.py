"""GPU tests of the error contract: bad index values are skipped and
reported through the device error word (never a fault), bad arguments are
rejected at the boundary before anything is launched, and the index
validation call finds out-of-range and duplicate entries.

Every bad value used here is one the kernels' own bounds checks turn into a
flag: slots past the pool, positions past the table, block-table entries
outside the pool, sequence lengths past the block table."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_04_gb300 import _abi, harness, synth
from tests._compare import assert_close_lse, assert_close_out, bf16_u16_to_f64
from tests._pipeline import oracle_step

pytestmark = pytest.mark.gpu


def _dw(seq_lens=(40, 70), S=2, **kw):
    w = synth.custom_workload("err", 50, list(seq_lens), 4, 2, 128, **kw)
    dw = harness.DeviceWorkload(w, num_splits=S)
    dw.fill()
    dw.upload_decode()
    return w, dw


def test_bad_slot_and_position_are_flagged_and_skipped():
    w, dw = _dw()
    d = dw.decode_inputs
    before_k = dw.k_cache.clone()
    slots = d["slot_mapping"].clone()
    pos = d["positions"].clone()
    slots[0] = w.num_pages * 16 + 5            # past the pool
    pos[1] = dw.cos_sin.shape[0] + 3           # past the table
    q = d["q0"].clone()
    dw.err.zero_()
    dw.write(q, d["k"], d["v"], pos, slots)
    torch.cuda.synchronize()
    e = int(dw.err.item())
    assert e & _abi.FLAG_SLOT_RANGE and e & _abi.FLAG_POSITION_RANGE
    assert torch.equal(dw.k_cache, before_k)   # neither token was written
    assert torch.equal(q, d["q0"])             # and neither q was rotated


def test_negative_slot_is_skipped_silently():
    w, dw = _dw()
    d = dw.decode_inputs
    before = dw.v_cache.clone()
    slots = torch.full_like(d["slot_mapping"], -1)
    dw.err.zero_()
    dw.write(d["q"], d["k"], d["v"], d["positions"], slots)
    torch.cuda.synchronize()
    assert int(dw.err.item()) == 0 and torch.equal(dw.v_cache, before)


def test_bad_page_id_is_flagged_and_left_out():
    w, dw = _dw(seq_lens=(48, 70))
    dw.step()
    torch.cuda.synchronize()
    bt_bad = w.block_tables.copy()
    bt_bad[0, 1] = w.num_pages + 1000          # tokens 16..31 of sequence 0
    st = oracle_step(w, num_splits=2)
    # the oracle leaves the same page out
    import oracle
    bt_orc = st["block_tables"].copy()
    bt_orc[0, 1] = st["k_cache"].shape[0] + 1000
    op, lp = oracle.paged_decode(st["q_rot"], st["k_cache"], st["v_cache"], bt_orc, st["seq_lens"],
                                 w.softmax_scale, 2, w.layout)
    out_ref, lse_ref = oracle.lse_merge(op, lp)
    dw.block_tables = torch.from_numpy(bt_bad).cuda()
    dw.err.zero_()
    dw.decode(dw.decode_inputs["q"])
    dw.merge()
    torch.cuda.synchronize()
    assert int(dw.err.item()) & _abi.FLAG_PAGE_RANGE
    assert_close_out(bf16_u16_to_f64(dw.bf16_u16(dw.out)), out_ref)
    assert_close_lse(dw.lse.cpu().numpy(), lse_ref)


def test_seq_len_past_block_table_is_flagged():
    w, dw = _dw(seq_lens=(40, 70))
    dw.step()
    sl = dw.seq_lens.clone()
    sl[0] = 10 ** 6
    dw.seq_lens = sl
    dw.err.zero_()
    dw.decode(dw.decode_inputs["q"])
    torch.cuda.synchronize()
    assert int(dw.err.item()) & _abi.FLAG_SEQ_LEN_RANGE
    assert torch.isfinite(dw.out_partial[1]).all()


def test_validate_indices_finds_each_problem():
    w = synth.custom_workload("val", 51, [40, 70, 5], 4, 2, 128, num_pages=20)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bitmap = torch.empty(((w.num_pages * 16 + 31) // 32,), dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 5, 17, 319], dtype=torch.int32, device="cuda")
    _abi.validate_indices(bt, sl, slots, w.num_pages, err, bitmap)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    checks = []
    bt2 = bt.clone(); bt2[1, 2] = 20; checks.append((bt2, sl, slots, _abi.FLAG_PAGE_RANGE))
    bt3 = bt.clone(); bt3[2, 0] = -1; checks.append((bt3, sl, slots, _abi.FLAG_PAGE_RANGE))
    sl2 = sl.clone(); sl2[0] = -3; checks.append((bt, sl2, slots, _abi.FLAG_SEQ_LEN_RANGE))
    # clamped to the block-table width, the sequence then also reaches its -1 padding entries
    sl3 = sl.clone(); sl3[2] = 16 * bt.shape[1] + 1
    checks.append((bt, sl3, slots, _abi.FLAG_SEQ_LEN_RANGE | _abi.FLAG_PAGE_RANGE))
    s2 = slots.clone(); s2[3] = 320; checks.append((bt, sl, s2, _abi.FLAG_SLOT_RANGE))
    s3 = slots.clone(); s3[3] = 5; checks.append((bt, sl, s3, _abi.FLAG_DUPLICATE_SLOT))
    for b_, l_, s_, flag in checks:
        err.zero_()
        bitmap.fill_(-1)  # stale contents: the call clears the bitmap itself
        _abi.validate_indices(b_, l_, s_, w.num_pages, err, bitmap)
        torch.cuda.synchronize()
        assert int(err.item()) == flag
    # padding past a sequence's pages is never read
    bt4 = bt.clone(); bt4[2, 1:] = 10 ** 6
    err.zero_()
    _abi.validate_indices(bt4, sl, slots, w.num_pages, err, bitmap)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def _expect(status, fn, *a, **k):
    with pytest.raises(_abi.PkvError) as e:
        fn(*a, **k)
    assert e.value.status == status


def test_bad_arguments_are_rejected_before_launch():
    w, dw = _dw()
    d = dw.decode_inputs
    # wrong dtype of k (float32 instead of bf16)
    _expect(_abi.PKV_ERR_INVALID_ARG, dw.write, d["q"], d["k"].float(), d["v"], d["positions"], d["slot_mapping"])
    # q heads not a multiple of kv heads
    _expect(_abi.PKV_ERR_INVALID_ARG, dw.write, d["q"][:, :3], d["k"], d["v"], d["positions"], d["slot_mapping"])
    # split count disagreeing with out_partial
    _expect(_abi.PKV_ERR_INVALID_ARG, _abi.paged_gqa_decode, d["q"], dw.k_cache, dw.v_cache, dw.block_tables,
            dw.seq_lens, w.softmax_scale, dw.num_splits + 1, dw.out_partial, dw.lse_partial)
    # head dim 96 is outside the supported set
    q96 = torch.zeros((2, 4, 96), dtype=torch.bfloat16, device="cuda")
    kc96 = torch.zeros((4, 2, 16, 96), dtype=torch.bfloat16, device="cuda")
    op = torch.zeros((2, 1, 4, 96), device="cuda"); lp = torch.zeros((2, 1, 4), device="cuda")
    _expect(_abi.PKV_ERR_UNSUPPORTED, _abi.paged_gqa_decode, q96, kc96, kc96, dw.block_tables, dw.seq_lens,
            0.1, 1, op, lp)
    # group of 32 query heads per kv head is outside the supported set
    q32 = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    op = torch.zeros((2, 1, 64, 128), device="cuda"); lp = torch.zeros((2, 1, 64), device="cuda")
    _expect(_abi.PKV_ERR_UNSUPPORTED, _abi.paged_gqa_decode, q32, dw.k_cache, dw.v_cache, dw.block_tables,
            dw.seq_lens, 0.1, 1, op, lp)
    # fp8 cache without scales
    kc8 = dw.k_cache.view(torch.uint8)[..., :128].contiguous()
    _expect(_abi.PKV_ERR_INVALID_ARG, _abi.rope_kv_write, None, d["k"], d["v"], d["positions"], dw.cos_sin, kc8,
            kc8.clone(), d["slot_mapping"])
    # page size 8 is outside the decode kernel's set
    kc_p8 = torch.zeros((8, 2, 8, 128), dtype=torch.bfloat16, device="cuda")
    _expect(_abi.PKV_ERR_UNSUPPORTED, _abi.paged_gqa_decode, d["q"], kc_p8, kc_p8, dw.block_tables, dw.seq_lens,
            0.1, dw.num_splits, dw.out_partial, dw.lse_partial)
    torch.cuda.synchronize()
