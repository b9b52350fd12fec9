"""GPU tests of the NVFP4 cache write beyond the decode-step parity cases.

The quantiser is checked byte for byte against the oracle on every finite
bf16 value: rows are made of 16-value blocks, each an "anchor" value that
fixes the block's largest magnitude (at a rotating position, so either lane
of the pair may hold it) and 15 values no larger, swept over all bf16
patterns up to the anchor. Anchors and static scales are chosen so that the
block scale is 1 (every E2M1 tie exact), a few-bit value (ties exact in the
quotient but not in its reciprocal product), an arbitrary value, zero
(blocks below E4M3's range) and saturated (448). The NHD layout is checked
for the write (the decode takes HND only)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import _abi, synth
from tests._compare import bf16_u16_to_f64

pytestmark = pytest.mark.gpu


def _bf16_u16(x: float) -> int:
    return int((np.array([x], np.float32).view(np.uint32)[0] >> 16))   # truncation: exact for the anchors used


def _blocks(anchor: int, seed: int) -> np.ndarray:
    """uint16 [n, 16]: every finite bf16 pattern of magnitude <= the anchor's,
    15 to a block, the anchor at position (block index % 16)."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # the NaN patterns (signalling ones raise "invalid"), filtered below
        vals = bf16_u16_to_f64(pats)
    a = bf16_u16_to_f64(np.array([anchor], np.uint16))[0]
    sel = pats[np.isfinite(vals) & (np.abs(vals) <= a)]
    perm = np.argsort(synth.uniform(synth.stream_key(seed, "blk"), len(sel)))
    sel = sel[perm]
    n = -(-len(sel) // 15)
    sel = np.concatenate([sel, np.zeros(n * 15 - len(sel), np.uint16)]).reshape(n, 15)
    out = np.empty((n, 16), np.uint16)
    for i in range(n):
        p = i % 16
        out[i, :p] = sel[i, :p]
        out[i, p] = anchor
        out[i, p + 1:] = sel[i, p:]
    return out


def _write_both(vals, g, layout="HND", style="neox", positions=None, cs=None):
    """Write vals [T, Hkv, D] (uint16 bf16 bits) as k and v through the GPU
    and the oracle; return (gpu, oracle) tuples of (kc, vc, kbs, vbs)."""
    T, Hkv, D = vals.shape
    pages = -(-T // 16)
    if layout == "HND":
        vshape, sshape = (pages, Hkv, 16, D // 2), (pages, Hkv, 16, D // 16)
    else:
        vshape, sshape = (pages, 16, Hkv, D // 2), (pages, 16, Hkv, D // 16)
    if cs is None:  # position 0 of an identity table: k is written unrotated
        cs = np.zeros((1, D), np.float32)
        cs[0, :D // 2] = 1.0
    pos = np.zeros(T, np.int32) if positions is None else positions
    slots = np.arange(T, dtype=np.int32)
    ref = [np.zeros(vshape, np.uint8), np.zeros(vshape, np.uint8), np.zeros(sshape, np.uint8),
           np.zeros(sshape, np.uint8)]
    bad = oracle.rope_kv_write_nvfp4(None, vals, vals, pos, cs, ref[0], ref[1], ref[2], ref[3], slots, layout, style,
                                     g, g)
    assert bad == 0
    dev = "cuda"
    x = torch.from_numpy(np.ascontiguousarray(vals).view(np.int16)).to(dev).view(torch.bfloat16)
    got = [torch.zeros(vshape, dtype=torch.uint8, device=dev), torch.zeros(vshape, dtype=torch.uint8, device=dev),
           torch.zeros(sshape, dtype=torch.uint8, device=dev), torch.zeros(sshape, dtype=torch.uint8, device=dev)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gt = torch.from_numpy(g).to(dev)
    _abi.rope_kv_write_nvfp4(None, x, x, torch.from_numpy(pos).to(dev), torch.from_numpy(cs).to(dev), got[0], got[1],
                             got[2], got[3], torch.from_numpy(slots).to(dev), gt, gt, layout, style, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return [t.cpu().numpy() for t in got], ref


@pytest.mark.parametrize("g", [1.0, 0.375, 0.7, 1.3])
def test_nvfp4_write_every_bf16_under_anchors(g):
    D = 128
    anchors = [_bf16_u16(6.0 * g) if g in (1.0, 0.375) else _bf16_u16(5.5), _bf16_u16(0.05), _bf16_u16(100.0),
               _bf16_u16(1e-5), _bf16_u16(6144.0)]
    rows = np.concatenate([_blocks(a, i) for i, a in enumerate(anchors)])
    n = -(-rows.size // D)
    flat = np.concatenate([rows.reshape(-1), np.zeros(n * D - rows.size, np.uint16)])
    vals = flat.reshape(n, 1, D)
    got, ref = _write_both(vals, np.array([g], np.float32))
    for name, a, b in zip(("k values", "v values", "k scales", "v scales"), got, ref):
        if not np.array_equal(a, b):
            i = np.argwhere(a != b)[0]
            raise AssertionError(f"{name} differ at {tuple(i)}: gpu {a[tuple(i)]:#04x} oracle {b[tuple(i)]:#04x}")
    # the sweep reaches the degenerate scales: 0 (anchor 1e-5) and 448 (anchor 6144 for g <= 1.3)
    assert (ref[3] == 0).any() and (ref[3] == 0x7E).any()


@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_nvfp4_write_nhd_layout(style):
    w = synth.custom_workload("fp4nhd", 61, [40], 4, 3, 128, layout="NHD", style=style, cache_dtype="nvfp4",
                              rope_base=5e5)
    k, v = w.seq_kv(0)
    pos = np.arange(40, dtype=np.int32)[::-1].copy()           # positions out of order
    cs = w.cos_sin()
    T, Hkv, D = k.shape
    # k and v separately through both paths (the helper writes one array as both)
    for arr in (k, v):
        got, ref = _write_both(arr, w.k_scale, layout="NHD", style=style, positions=pos, cs=cs)
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)


def test_nvfp4_decode_rejects_nhd():
    P, Hkv, D = 4, 1, 128
    z = lambda *s: torch.zeros(s, dtype=torch.uint8, device="cuda")  # noqa: E731
    q = torch.zeros((1, 2, D), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    op = torch.empty((1, 1, 2, D), device="cuda")
    lp = torch.empty((1, 1, 2), device="cuda")
    g = torch.ones(1, device="cuda")
    with pytest.raises(_abi.PkvError) as e:
        _abi.paged_gqa_decode_nvfp4(q, z(P, 16, Hkv, D // 2), z(P, 16, Hkv, D // 2), z(P, 16, Hkv, D // 16),
                                    z(P, 16, Hkv, D // 16), bt, sl, 0.1, 1, op, lp, g, g, layout="NHD")
    assert e.value.status == _abi.PKV_ERR_UNSUPPORTED
