"""pkv_copy (the SMs moving bytes between device memory and pinned host
memory): every byte equal for each direction, sizes with ragged tails and
both the 16-byte and the byte path; host memory CUDA did not page-lock is
refused before anything is launched."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_04_gb300 import _abi

pytestmark = pytest.mark.gpu


def _buf(n, where, fill=None):
    t = torch.zeros(n + 64, dtype=torch.uint8)
    if where == "host":
        t = t.pin_memory()
    else:
        t = t.cuda()
    if fill is not None:
        t[:fill.numel()].copy_(fill.to(t.device))
    return t


@pytest.mark.parametrize("direction", ["d2d", "h2d", "d2h", "h2h"])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 4099, 163840, 1 << 20])
@pytest.mark.parametrize("offset", [0, 1, 16])
def test_copy_bytes(direction, n, offset):
    src_where = "host" if direction[0] == "h" else "dev"
    dst_where = "host" if direction[2] == "h" else "dev"
    data = torch.from_numpy(np.random.default_rng(n + offset).integers(0, 256, n + 64, dtype=np.uint8))
    src = _buf(n, src_where, data)
    dst = _buf(n, dst_where)
    _abi.copy(dst[offset:offset + n], src[64 - offset:64 - offset + n] if offset else src[:n])
    torch.cuda.synchronize()
    want = data[64 - offset:64 - offset + n] if offset else data[:n]
    assert torch.equal(dst[offset:offset + n].cpu(), want)
    assert int(dst[:offset].cpu().sum()) == 0 and int(dst[offset + n:].cpu().sum()) == 0  # nothing outside


def test_copy_refuses_unregistered_host_memory():
    host = np.zeros(4096, np.uint8)  # ordinary (pageable) memory
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    lib = _abi.lib()
    assert lib.pkv_copy(dev.data_ptr(), host.ctypes.data, 4096, None) == _abi.PKV_ERR_UNSUPPORTED
    assert lib.pkv_copy(host.ctypes.data, dev.data_ptr(), 4096, None) == _abi.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
