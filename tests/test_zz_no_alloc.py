"""GPU test of pkv_validate_indices_static, the validation entry point for
callers that cannot allocate device memory (an engine whose allocator has
already taken all free memory for its KV pool, or a path that must not call
cudaMalloc/cudaFree because they can synchronise the device).

Its result must equal that of pkv_validate_indices given a caller-allocated
bitmap, on two calls in a row: the second call must not see the bits the
first call left in the shared static bitmap. This file is collected last on
purpose; it also passes when run alone in a fresh process."""
import pytest
import torch

from paged_kv_gqa_04_gb300 import _abi, synth

pytestmark = pytest.mark.gpu


def _inputs():
    w = synth.custom_workload("noalloc", 71, [40, 70, 5, 300], 4, 2, 128, num_pages=64)
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    return w, bt, sl


def _both(bt, sl, slots, num_pages):
    """Flags from the allocating entry point and from the static one."""
    err_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    err_b = torch.zeros(1, dtype=torch.int32, device="cuda")
    bitmap = torch.empty(((num_pages * 16 + 31) // 32,), dtype=torch.int32, device="cuda")
    _abi.validate_indices(bt, sl, slots, num_pages, err_a, bitmap)
    _abi.validate_indices_static(bt, sl, slots, num_pages, err_b)
    torch.cuda.synchronize()
    return int(err_a.item()), int(err_b.item())


def test_static_validation_matches_allocating_validation_on_two_calls():
    w, bt, sl = _inputs()
    n = w.num_pages
    dup = torch.tensor([3, 17, 3, 900], dtype=torch.int32, device="cuda")       # slot 3 twice
    clean = torch.tensor([3, 17, 18, 900], dtype=torch.int32, device="cuda")    # same slots, no repeat
    a1, b1 = _both(bt, sl, dup, n)
    assert a1 == b1 == _abi.FLAG_DUPLICATE_SLOT
    # the second call follows the first on the same stream: the bits the
    # first call left for slots 3, 17 and 900 must have been cleared
    a2, b2 = _both(bt, sl, clean, n)
    assert a2 == b2 == 0
    # and again with range errors, to compare every flag the check can raise
    bad = torch.tensor([3, n * 16 + 2, 17], dtype=torch.int32, device="cuda")
    bt_bad = bt.clone()
    bt_bad[1, 2] = n + 5
    a3, b3 = _both(bt_bad, sl, bad, n)
    assert a3 == b3 == (_abi.FLAG_SLOT_RANGE | _abi.FLAG_PAGE_RANGE)


def test_static_validation_rejects_pools_beyond_its_bitmap():
    _, bt, sl = _inputs()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    too_many = (1 << 23) // 16 + 1
    with pytest.raises(_abi.PkvError) as e:
        _abi.validate_indices_static(bt, sl, None, too_many, err)
    assert e.value.status == _abi.PKV_ERR_UNSUPPORTED
    # at the limit it runs
    _abi.validate_indices_static(bt, sl, None, (1 << 23) // 16, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_bits_left_by_a_larger_pool_do_not_reach_a_smaller_one():
    """Each call clears only the bits of its own pool. A call on a large pool
    that leaves bits set (a duplicate), then a clean call on a small pool,
    then a clean call on the large pool: the last two must report nothing,
    and the allocating entry point must agree on each."""
    big = synth.custom_workload("noalloc_big", 72, [3000, 1200, 40], 4, 2, 128, num_pages=4096)
    small = synth.custom_workload("noalloc_small", 73, [20, 7], 4, 2, 128, num_pages=4)
    bt_b, sl_b = torch.from_numpy(big.block_tables).cuda(), torch.from_numpy(big.seq_lens).cuda()
    bt_s, sl_s = torch.from_numpy(small.block_tables).cuda(), torch.from_numpy(small.seq_lens).cuda()
    hi = big.num_pages * 16 - 1  # slots far above the small pool's bits
    dup = torch.tensor([hi, 5, hi - 40, hi, 60000], dtype=torch.int32, device="cuda")
    a1, b1 = _both(bt_b, sl_b, dup, big.num_pages)
    assert a1 == b1 == _abi.FLAG_DUPLICATE_SLOT
    clean_small = torch.tensor([5, 6, 63, 0], dtype=torch.int32, device="cuda")
    a2, b2 = _both(bt_s, sl_s, clean_small, small.num_pages)
    assert a2 == b2 == 0
    clean_big = torch.tensor([hi, 5, hi - 40, 60000], dtype=torch.int32, device="cuda")
    a3, b3 = _both(bt_b, sl_b, clean_big, big.num_pages)
    assert a3 == b3 == 0
