"""CPU tests of the C ABI: the library loads, exports every function that
include/pkv.h declares, rejects inconsistent arguments before touching the
GPU, and its split heuristic behaves as specified. No GPU work is launched."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import paged_kv_gqa_04_gb300 as pkv
from paged_kv_gqa_04_gb300 import _abi, _build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(names) == set(_abi.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    assert set(names) <= exported


def test_abi_version_and_status_strings(lib):
    assert lib.pkv_abi_version() == 7
    for s in range(4):
        assert pkv.status_string(s)
    assert "invalid" in pkv.status_string(1)


def _t(shape, dtype, ptr=0x1000, strides=None):
    d = _abi.PkvTensor()
    d.ptr = ptr
    d.dtype = {"bf16": 0, "fp8": 1, "f32": 2, "i32": 3, "fp4": 4}[dtype]
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for n in reversed(shape):
            strides.insert(0, acc)
            acc *= n
    for i, (n, s) in enumerate(zip(shape, strides)):
        d.shape[i] = n
        d.stride[i] = s
    return ctypes.pointer(d)


NULL = None


def test_write_rejects_inconsistent_arguments(lib):
    """Host validation only: fake (never dereferenced) pointers; every call
    must return before any CUDA work."""
    T, Hq, Hkv, D = 4, 8, 2, 128
    kc = _t((10, Hkv, 16, D), "bf16")
    args = dict(q=_t((T, Hq, D), "bf16"), k=_t((T, Hkv, D), "bf16"), v=_t((T, Hkv, D), "bf16"),
                pos=_t((T,), "i32"), cs=_t((100, D), "f32"), kc=kc, vc=_t((10, Hkv, 16, D), "bf16"),
                slot=_t((T,), "i32"), ks=NULL, vs=NULL)

    def call(layout=1, style=0, **over):
        a = dict(args, **over)
        return lib.pkv_rope_kv_write(a["q"], a["k"], a["v"], a["pos"], a["cs"], a["kc"], a["vc"], a["slot"],
                                     a["ks"], a["vs"], layout, style, None, None)

    assert call(layout=2) == _abi.PKV_ERR_INVALID_ARG
    assert call(style=5) == _abi.PKV_ERR_INVALID_ARG
    assert call(k=_t((T, Hkv, D), "f32")) == _abi.PKV_ERR_INVALID_ARG
    assert call(v=_t((T + 1, Hkv, D), "bf16")) == _abi.PKV_ERR_INVALID_ARG
    assert call(q=_t((T, 7, D), "bf16")) == _abi.PKV_ERR_INVALID_ARG           # 7 % 2 != 0
    assert call(pos=_t((T - 1,), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert call(cs=_t((100, D // 2), "f32")) == _abi.PKV_ERR_INVALID_ARG
    assert call(vc=_t((10, Hkv, 16, D), "fp8")) == _abi.PKV_ERR_INVALID_ARG   # cache dtypes differ
    fp8c = _t((10, Hkv, 16, D), "fp8")
    assert call(kc=fp8c, vc=fp8c) == _abi.PKV_ERR_INVALID_ARG                # fp8 without scales
    assert call(kc=fp8c, vc=fp8c, ks=_t((3,), "f32"), vs=_t((3,), "f32")) == _abi.PKV_ERR_INVALID_ARG
    d96 = dict(q=_t((T, Hq, 96), "bf16"), k=_t((T, Hkv, 96), "bf16"), v=_t((T, Hkv, 96), "bf16"),
               cs=_t((100, 96), "f32"), kc=_t((10, Hkv, 16, 96), "bf16"), vc=_t((10, Hkv, 16, 96), "bf16"))
    assert call(**d96) == _abi.PKV_ERR_UNSUPPORTED
    assert call(k=_t((T, Hkv, D), "bf16", ptr=0x1002)) == _abi.PKV_ERR_UNSUPPORTED  # not 16-byte aligned
    # an empty call is valid and launches nothing
    e = dict(q=_t((0, Hq, D), "bf16"), k=_t((0, Hkv, D), "bf16"), v=_t((0, Hkv, D), "bf16"),
             pos=_t((0,), "i32"), slot=_t((0,), "i32"))
    assert call(**e) == _abi.PKV_OK


def test_decode_and_merge_reject_inconsistent_arguments(lib):
    B, Hq, Hkv, D, S = 3, 12, 2, 128, 4
    q = _t((B, Hq, D), "bf16")
    kc = _t((50, Hkv, 16, D), "bf16")
    bt = _t((B, 10), "i32")
    sl = _t((B,), "i32")
    op = _t((B, S, Hq, D), "f32")
    lp = _t((B, S, Hq), "f32")

    def dec(**o):
        a = dict(q=q, kc=kc, vc=kc, bt=bt, sl=sl, scale=0.1, S=S, op=op, lp=lp, ks=NULL, vs=NULL, layout=1)
        a.update(o)
        return lib.pkv_paged_gqa_decode(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["scale"], a["S"], a["op"],
                                        a["lp"], a["ks"], a["vs"], a["layout"], None, None)

    assert dec(S=0) == _abi.PKV_ERR_INVALID_ARG
    assert dec(S=5) == _abi.PKV_ERR_INVALID_ARG
    assert dec(bt=_t((B + 1, 10), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(lp=_t((B, S, Hq + 1), "f32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(scale=float("nan")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(kc=_t((50, Hkv, 8, D), "bf16"), vc=_t((50, Hkv, 8, D), "bf16")) == _abi.PKV_ERR_UNSUPPORTED
    q64 = _t((B, 64, D), "bf16")
    assert dec(q=q64, op=_t((B, S, 64, D), "f32"), lp=_t((B, S, 64), "f32"),
               kc=_t((50, 2, 16, D), "bf16"), vc=_t((50, 2, 16, D), "bf16")) == _abi.PKV_ERR_UNSUPPORTED
    assert dec(q=_t((0, Hq, D), "bf16"), bt=_t((0, 10), "i32"), sl=_t((0,), "i32"), op=_t((0, S, Hq, D), "f32"),
               lp=_t((0, S, Hq), "f32")) == _abi.PKV_OK

    out = _t((B, Hq, D), "bf16")
    m = lib.pkv_lse_merge
    assert m(op, lp, _t((B, Hq + 1, D), "bf16"), NULL, None) == _abi.PKV_ERR_INVALID_ARG
    assert m(op, _t((B, S + 1, Hq), "f32"), out, NULL, None) == _abi.PKV_ERR_INVALID_ARG
    assert m(_t((B, S, Hq, 96), "f32"), lp, _t((B, Hq, 96), "bf16"), NULL, None) == _abi.PKV_ERR_UNSUPPORTED
    assert m(op, lp, out, _t((B, Hq + 2), "f32"), None) == _abi.PKV_ERR_INVALID_ARG
    assert lib.pkv_validate_indices(bt, sl, NULL, 50, NULL, None, None) == _abi.PKV_ERR_INVALID_ARG


def test_validation_entry_points_reject_bad_arguments_before_any_cuda_call(lib):
    """Host checks of both index-validation entry points; every call returns
    before the static one looks up its device array or anything launches."""
    B = 3
    bt = _t((B, 10), "i32")
    sl = _t((B,), "i32")
    slots = _t((7,), "i32")
    err = ctypes.c_void_p(0x2000)
    st = lib.pkv_validate_indices_static
    assert st(bt, sl, slots, 50, None, None) == _abi.PKV_ERR_INVALID_ARG              # no error word
    assert st(bt, _t((B + 1,), "i32"), slots, 50, err, None) == _abi.PKV_ERR_INVALID_ARG
    assert st(_t((B, 10), "f32"), sl, slots, 50, err, None) == _abi.PKV_ERR_INVALID_ARG
    assert st(bt, sl, _t((7, 2), "i32"), 50, err, None) == _abi.PKV_ERR_INVALID_ARG
    assert st(bt, sl, slots, -1, err, None) == _abi.PKV_ERR_INVALID_ARG
    limit = (1 << 23) // 16
    assert st(bt, sl, slots, limit + 1, err, None) == _abi.PKV_ERR_UNSUPPORTED
    # pools whose slot count would overflow a 64-bit product are refused, not wrapped
    for huge in ((1 << 59) + 1, (1 << 62), (1 << 63) - 1):
        assert st(bt, sl, slots, huge, err, None) == _abi.PKV_ERR_UNSUPPORTED
        assert lib.pkv_validate_indices(bt, sl, slots, huge, NULL, err, None) == _abi.PKV_ERR_UNSUPPORTED
    al = lib.pkv_validate_indices
    assert al(bt, sl, slots, -1, NULL, err, None) == _abi.PKV_ERR_INVALID_ARG
    assert al(bt, sl, slots, 50, _t((10,), "i32"), err, None) == _abi.PKV_ERR_INVALID_ARG  # bitmap too small


def test_nvfp4_entry_points_reject_inconsistent_arguments(lib):
    """Host validation of the NVFP4 write and decode: fake pointers, every
    call returns before any CUDA work."""
    T, B, Hq, Hkv, D, S, P = 4, 3, 12, 2, 128, 4, 50
    kc = _t((P, Hkv, 16, D // 2), "fp4")
    bs = _t((P, Hkv, 16, D // 16), "fp8")
    g = _t((Hkv,), "f32")
    w = dict(q=_t((T, Hq, D), "bf16"), k=_t((T, Hkv, D), "bf16"), v=_t((T, Hkv, D), "bf16"),
             pos=_t((T,), "i32"), cs=_t((100, D), "f32"), kc=kc, vc=kc, kbs=bs, vbs=bs, slot=_t((T,), "i32"),
             ks=g, vs=g)

    def write(layout=1, **over):
        a = dict(w, **over)
        return lib.pkv_rope_kv_write_nvfp4(a["q"], a["k"], a["v"], a["pos"], a["cs"], a["kc"], a["vc"], a["kbs"],
                                           a["vbs"], a["slot"], a["ks"], a["vs"], layout, 0, None, None)

    assert write(kc=_t((P, Hkv, 16, D // 2), "fp8"), vc=_t((P, Hkv, 16, D // 2), "fp8")) == _abi.PKV_ERR_INVALID_ARG
    # value caches of D/4 bytes describe D = 64: inconsistent with k, v and the scale caches
    assert write(kc=_t((P, Hkv, 16, D // 4), "fp4"), vc=_t((P, Hkv, 16, D // 4), "fp4")) == _abi.PKV_ERR_INVALID_ARG
    assert write(kc=_t((P, Hkv, 16, D), "fp4"), vc=_t((P, Hkv, 16, D), "fp4")) == _abi.PKV_ERR_UNSUPPORTED  # D = 256
    assert write(kbs=_t((P, Hkv, 16, D // 8), "fp8")) == _abi.PKV_ERR_INVALID_ARG
    assert write(vbs=_t((P, Hkv, 16, D // 16), "bf16")) == _abi.PKV_ERR_INVALID_ARG
    assert write(kbs=NULL) == _abi.PKV_ERR_INVALID_ARG
    assert write(ks=NULL, vs=NULL) == _abi.PKV_ERR_INVALID_ARG            # static scales are required
    # the bf16/fp8 entry point does not take NVFP4 caches
    assert lib.pkv_rope_kv_write(w["q"], w["k"], w["v"], w["pos"], w["cs"], kc, kc, w["slot"], g, g, 1, 0,
                                 None, None) == _abi.PKV_ERR_INVALID_ARG
    e = dict(q=_t((0, Hq, D), "bf16"), k=_t((0, Hkv, D), "bf16"), v=_t((0, Hkv, D), "bf16"),
             pos=_t((0,), "i32"), slot=_t((0,), "i32"))
    assert write(**e) == _abi.PKV_OK
    assert write(layout=0, kc=_t((P, 16, Hkv, D // 2), "fp4"), vc=_t((P, 16, Hkv, D // 2), "fp4"),
                 kbs=_t((P, 16, Hkv, D // 16), "fp8"), vbs=_t((P, 16, Hkv, D // 16), "fp8"), **e) == _abi.PKV_OK

    d = dict(q=_t((B, Hq, D), "bf16"), kc=kc, vc=kc, kbs=bs, vbs=bs, bt=_t((B, 10), "i32"), sl=_t((B,), "i32"),
             op=_t((B, S, Hq, D), "f32"), lp=_t((B, S, Hq), "f32"), ks=g, vs=g)

    def dec(layout=1, **over):
        a = dict(d, **over)
        return lib.pkv_paged_gqa_decode_nvfp4(a["q"], a["kc"], a["vc"], a["kbs"], a["vbs"], a["bt"], a["sl"], 0.1, S,
                                              a["op"], a["lp"], a["ks"], a["vs"], layout, None, None)

    nhd = dict(kc=_t((P, 16, Hkv, D // 2), "fp4"), vc=_t((P, 16, Hkv, D // 2), "fp4"),
               kbs=_t((P, 16, Hkv, D // 16), "fp8"), vbs=_t((P, 16, Hkv, D // 16), "fp8"))
    assert dec(layout=0, **nhd) == _abi.PKV_ERR_UNSUPPORTED                 # HND only
    # the scale bytes of one (page, head) must be contiguous and 16-byte aligned
    strided = _t((P, Hkv, 16, D // 16), "fp8", strides=[Hkv * 16 * 16, 16 * 16, 16, 1])
    assert dec(kbs=strided) == _abi.PKV_ERR_UNSUPPORTED
    assert dec(vbs=_t((P, Hkv, 16, D // 16), "fp8", ptr=0x1008)) == _abi.PKV_ERR_UNSUPPORTED
    assert dec(ks=NULL) == _abi.PKV_ERR_INVALID_ARG
    assert dec(q=_t((B, Hq, 64), "bf16")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(q=_t((0, Hq, D), "bf16"), bt=_t((0, 10), "i32"), sl=_t((0,), "i32"), op=_t((0, S, Hq, D), "f32"),
               lp=_t((0, S, Hq), "f32")) == _abi.PKV_OK


def test_split_heuristic(lib):
    sms = 152

    def choose(name):
        w = synth.make_workload(name)
        return pkv.choose_num_splits(w.B, w.Hkv, w.Hq, w.D, int(w.pages_per_seq.sum()), int(w.pages_per_seq.max()),
                                     w.cache_dtype, sms)

    # long context, 8 (sequence, kv head) units: enough splits to cover every SM
    s3 = choose("longctx")
    assert 16 <= s3 <= 64 and 2 * 4 * s3 >= sms
    # large ragged batch already has 2048 units: few splits
    assert choose("ragged") <= 4
    for name in synth.WORKLOADS:
        assert 1 <= choose(name) <= 1024
    # one 1M-token sequence with one kv head: one to three splits per SM (on
    # GB300 the chained step measured 93.0 / 92.3 / 94.3 us at S = 228 / 304 /
    # 456: past ~2 CTAs per SM the HBM is saturated and more splits only add
    # start-up and merge work)
    s_m = choose("million")
    assert sms <= s_m <= 3 * sms
    # the bench workload: one wave of CTAs (measured best, S = 6-7)
    assert 6 <= choose("qwen") <= 7
    # degenerate inputs
    assert pkv.choose_num_splits(0, 1, 1, 128, 0, 0, "bf16", sms) == 1
    assert pkv.choose_num_splits(1, 1, 1, 128, 1, 1, "bf16", sms) == 1
    # never more splits than pages
    assert pkv.choose_num_splits(1, 1, 8, 128, 3, 3, "bf16", sms) <= 3


def test_mla_split_heuristic(lib):
    sms = 152

    def choose(name):
        w = synth.make_mla_workload(name)
        return pkv.choose_num_splits_mla(w.B, w.H, int(w.pages_per_seq.sum()), int(w.pages_per_seq.max()), sms)

    # one 800-page sequence: 4-page splits (two whole 128-token chunks each),
    # one item per CTA, as many (empty) extra splits as keep those items
    # (measured on GB300: 24.9 us per step at 266, 25.6 at 200, 29.8 at
    # 5-page splits)
    s1 = choose("mla")
    assert s1 == 266
    # 32 sequences of 64-256 pages over 304 CTAs: about one long item per
    # CTA (measured: 71.6 us per step at S = 12, 74.2 at 19, 80.9 at 8)
    assert 10 <= choose("mla_batch") <= 16
    assert pkv.choose_num_splits_mla(0, 8, 0, 0, sms) == 1
    assert pkv.choose_num_splits_mla(1, 8, 3, 3, sms) <= 3


def test_split_heuristics_stay_in_range_on_random_and_extreme_inputs():
    rng = np.random.default_rng(7)
    for _ in range(400):
        B = int(rng.integers(1, 4096))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.integers(1, 17))
        D = int(rng.choice([64, 128]))
        max_pages = int(rng.integers(1, 70000))
        total = int(rng.integers(max_pages, max_pages * B + 1))
        sms = int(rng.choice([1, 76, 132, 152, 160]))
        for dt in ("bf16", "fp8", "nvfp4"):
            S = pkv.choose_num_splits(B, Hkv, Hkv * G, D, total, max_pages, dt, sms)
            assert 1 <= S <= min(1024, max_pages)
            assert S == pkv.choose_num_splits(B, Hkv, Hkv * G, D, total, max_pages, dt, sms)  # deterministic
        Sm = pkv.choose_num_splits_mla(B, int(rng.integers(1, 17)), total, max_pages, sms)
        assert 1 <= Sm <= min(1024, max_pages)
    # extreme but valid sizes
    assert 1 <= pkv.choose_num_splits(65535, 64, 1024, 128, (1 << 40), 1 << 24, "bf16", 152) <= 1024
    assert 1 <= pkv.choose_num_splits_mla(65535, 16, (1 << 40), 1 << 24, 152) <= 1024


def test_package_exports_resolve():
    for name in pkv.__all__:
        assert getattr(pkv, name) is not None, name


def test_binding_copy_checks_its_tensors():
    import torch
    from paged_kv_gqa_04_gb300 import _abi
    a = torch.zeros(8, 8, dtype=torch.uint8)
    with pytest.raises(ValueError):
        _abi.copy(a.t(), a)                               # not contiguous
    with pytest.raises(ValueError):
        _abi.copy(torch.zeros(63, dtype=torch.uint8), a)  # sizes differ


def test_copy_rejects_bad_arguments_before_any_cuda_call():
    from paged_kv_gqa_04_gb300 import _abi
    lib = _abi.lib()
    assert lib.pkv_copy(0x2000, 0x1000, -1, None) == _abi.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy(None, 0x1000, 16, None) == _abi.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy(0x2000, None, 16, None) == _abi.PKV_ERR_INVALID_ARG
    assert lib.pkv_copy(0x1008, 0x1000, 16, None) == _abi.PKV_ERR_INVALID_ARG  # overlapping ranges
    assert lib.pkv_copy(None, None, 0, None) == _abi.PKV_OK                   # nothing to copy


def test_selftest_bounded_wait_rejects_bad_limits():
    from paged_kv_gqa_04_gb300 import _abi
    lib = _abi.lib()
    for limit in (0, 99_999, 10_000_001):
        assert lib.pkv_selftest_bounded_wait(limit, None, None, None) == _abi.PKV_ERR_INVALID_ARG


def _plan_pages(np_b, S):
    """Pages of each split of a sequence of np_b pages dealt into S splits
    (the decode's rule, written out for the test)."""
    pps = -(-np_b // S) if np_b else 0
    return [max(0, min(pps, np_b - s * pps)) for s in range(S)]


@pytest.mark.parametrize("name", ["qwen", "ragged", "fp8", "fp4", "longctx", "million", "tiny"])
def test_split_plan_covers_every_split_once_longest_first(lib, name):
    w = synth.make_workload(name)
    sp, nrec, work = _abi.plan_splits(w.seq_lens, w.Hkv, w.Hq, w.D, w.max_pages, w.cache_dtype, 152)
    npg = w.pages_per_seq.astype(int)
    assert sp.shape == (w.B,) and (sp >= 1).all() and nrec == int(sp.max())
    items = [(int(e) >> 12, int(e) & 0xFFF, int(p0)) for e, p0 in work]
    assert sorted((b, s) for b, s, _ in items) == [(b, s) for b in range(w.B) for s in range(int(sp[b]))]
    pages = []
    for b, s, p0 in items:
        pp = _plan_pages(npg[b], int(sp[b]))
        pps = pp[0]
        assert p0 == min(s * pps, npg[b])                      # the hint is the split's first page
        pages.append(pp[s])
    assert all(x >= y for x, y in zip(pages, pages[1:]))      # longest first
    for b in range(w.B):                                       # no empty split where pages exist
        if npg[b]:
            assert all(p > 0 for p in _plan_pages(npg[b], int(sp[b])))
    # deterministic
    sp2, nrec2, work2 = _abi.plan_splits(w.seq_lens, w.Hkv, w.Hq, w.D, w.max_pages, w.cache_dtype, 152)
    assert np.array_equal(sp, sp2) and nrec == nrec2 and np.array_equal(work, work2)


def test_split_plan_with_a_page_target(lib):
    lens = np.array([0, 1, 16, 17, 160, 161, 1000, 4000, 33], np.int32)
    npg = (lens.astype(int) + 15) // 16
    for T in (1, 2, 3, 7, 16, 1000):
        sp, nrec, work = _abi.plan_splits(lens, 2, 12, 128, 300, "bf16", 152, 4095, T)
        for b in range(len(lens)):
            pp = _plan_pages(npg[b], int(sp[b]))
            assert max(pp) <= T                                 # no split above the target
            if npg[b] > T:                                      # and no more splits than needed
                assert int(sp[b]) == -(-npg[b] // T) or max(_plan_pages(npg[b], int(sp[b]) - 1)) > T
        assert len(work) == int(sp.sum())
    # a record cap binds: S_b <= max_splits, pages spread over the cap
    sp, nrec, work = _abi.plan_splits(lens, 2, 12, 128, 300, "bf16", 152, 5, 1)
    assert nrec == 5 and (sp <= 5).all() and int(sp[7]) == 5


def test_split_plan_rejects_bad_arguments(lib):
    f = lib.pkv_plan_splits
    sl = np.array([10, 20], np.int32)
    sp = np.zeros(2, np.int32)
    nrec, nwork = ctypes.c_int32(0), ctypes.c_int64(0)

    def call(B=2, Hkv=2, Hq=4, D=128, mp=4, dt=0, sms=152, ms=4095, T=0, work=None, cap=0, sl_p=True, sp_p=True):
        return f(sl.ctypes.data if sl_p else None, B, Hkv, Hq, D, mp, dt, sms, ms, T, sp.ctypes.data if sp_p else None,
                 ctypes.byref(nrec), work, cap, ctypes.byref(nwork))
    assert call() == _abi.PKV_OK and nwork.value == int(sp.sum())
    assert call(Hq=3) == _abi.PKV_ERR_INVALID_ARG
    assert call(ms=0) == _abi.PKV_ERR_INVALID_ARG and call(ms=4096) == _abi.PKV_ERR_INVALID_ARG
    assert call(T=-1) == _abi.PKV_ERR_INVALID_ARG
    assert call(sl_p=False) == _abi.PKV_ERR_INVALID_ARG and call(sp_p=False) == _abi.PKV_ERR_INVALID_ARG
    assert call(B=-1) == _abi.PKV_ERR_INVALID_ARG
    small = np.zeros((1, 2), np.int32)
    assert call(work=small.ctypes.data, cap=1) == _abi.PKV_ERR_INVALID_ARG   # capacity below the item count
    assert nwork.value == int(sp.sum()) > 1                                  # the counts are still written
    assert call(B=0, sl_p=False, sp_p=False) == _abi.PKV_OK and nwork.value == 0


def test_planned_decode_and_merge_reject_inconsistent_arguments(lib):
    B, Hq, Hkv, D, S = 3, 12, 2, 128, 4
    q = _t((B, Hq, D), "bf16")
    kc = _t((50, Hkv, 16, D), "bf16")
    bt = _t((B, 10), "i32")
    sl = _t((B,), "i32")
    op = _t((B, S, Hq, D), "f32")
    lp = _t((B, S, Hq), "f32")
    sp = _t((B,), "i32")
    wk = _t((7, 2), "i32")

    def dec(**o):
        a = dict(q=q, kc=kc, vc=kc, kbs=NULL, vbs=NULL, bt=bt, sl=sl, scale=0.1, sp=sp, wk=wk, op=op, lp=lp)
        a.update(o)
        return lib.pkv_paged_gqa_decode_planned(a["q"], a["kc"], a["vc"], a["kbs"], a["vbs"], a["bt"], a["sl"],
                                                a["scale"], a["sp"], a["wk"], a["op"], a["lp"], NULL, NULL, 1, None,
                                                None)
    assert dec(sp=_t((B + 1,), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(wk=_t((7, 3), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(wk=_t((7,), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(sp=None) == _abi.PKV_ERR_INVALID_ARG and dec(wk=None) == _abi.PKV_ERR_INVALID_ARG
    assert dec(op=_t((B, 4096, Hq, D), "f32"), lp=_t((B, 4096, Hq), "f32")) == _abi.PKV_ERR_UNSUPPORTED
    assert dec(lp=_t((B, S + 1, Hq), "f32")) == _abi.PKV_ERR_INVALID_ARG
    out = _t((B, Hq, D), "bf16")
    m = lib.pkv_lse_merge_planned
    assert m(op, lp, None, out, NULL, None) == _abi.PKV_ERR_INVALID_ARG
    assert m(op, lp, _t((B + 1,), "i32"), out, NULL, None) == _abi.PKV_ERR_INVALID_ARG
    assert m(op, lp, _t((B,), "f32"), out, NULL, None) == _abi.PKV_ERR_INVALID_ARG


def _mla_plan_pages(np_b, S):
    pps = -(-np_b // S) if np_b else 0
    return [max(0, min(pps, np_b - s * pps)) for s in range(S)]


@pytest.mark.parametrize("name", ["mla_tiny", "mla", "mla_batch"])
def test_mla_split_plan_covers_every_split_once_longest_first(lib, name):
    w = synth.make_mla_workload(name)
    mp = int(w.block_tables.shape[1])
    sp, nrec, work = _abi.plan_splits_mla(w.seq_lens, w.H, mp, 152)
    npg = w.pages_per_seq.astype(int)
    assert sp.shape == (w.B,) and (sp >= 1).all() and nrec == int(sp.max())
    items = [(int(e) >> 12, int(e) & 0xFFF, int(p0)) for e, p0 in work]
    assert sorted((b, s) for b, s, _ in items) == [(b, s) for b in range(w.B) for s in range(int(sp[b]))]
    pages = [_mla_plan_pages(npg[b], int(sp[b]))[s] for b, s, _ in items]
    assert all(x >= y for x, y in zip(pages, pages[1:]))
    for b in range(w.B):
        if npg[b]:
            assert all(p > 0 for p in _mla_plan_pages(npg[b], int(sp[b])))
    if len(work) <= 2 * 152:
        # one item per CTA at most: the longest item is as short as an even page
        # target allows (one target lower would need more items than CTAs)
        T = max(pages)
        T = T + (T & 1)
        if T > 2:
            n_lower = sum(-(-int(n) // (T - 2)) if n else 1 for n in npg)
            assert n_lower > 2 * 152


def test_mla_split_plan_with_a_page_target_and_bad_arguments(lib):
    lens = np.array([0, 1, 64, 65, 640, 641, 9000, 33], np.int32)
    npg = (lens.astype(int) + 63) // 64
    for T in (1, 2, 4, 100):
        sp, nrec, work = _abi.plan_splits_mla(lens, 16, 200, 152, 4095, T)
        assert len(work) == int(sp.sum())
        for b in range(len(lens)):
            assert max(_mla_plan_pages(npg[b], int(sp[b]))) <= T
    f = lib.pkv_plan_splits_mla
    sp = np.zeros(len(lens), np.int32)
    nrec, nwork = ctypes.c_int32(0), ctypes.c_int64(0)

    def call(B=len(lens), H=16, mp=200, sms=152, ms=4095, T=0, work=None, cap=0):
        return f(lens.ctypes.data, B, H, mp, sms, ms, T, sp.ctypes.data, ctypes.byref(nrec), work, cap,
                 ctypes.byref(nwork))
    assert call() == _abi.PKV_OK and nwork.value == int(sp.sum())
    assert call(ms=0) == _abi.PKV_ERR_INVALID_ARG and call(ms=4096) == _abi.PKV_ERR_INVALID_ARG
    assert call(T=-1) == _abi.PKV_ERR_INVALID_ARG and call(B=-1) == _abi.PKV_ERR_INVALID_ARG
    small = np.zeros((1, 2), np.int32)
    assert call(work=small.ctypes.data, cap=1) == _abi.PKV_ERR_INVALID_ARG


def test_planned_mla_decode_rejects_inconsistent_arguments(lib):
    B, H, S = 3, 16, 4
    ql = _t((B, H, 512), "bf16")
    qp = _t((B, H, 64), "bf16")
    ckv = _t((50, 64, 512), "fp8")
    kpe = _t((50, 64, 64), "bf16")
    bt = _t((B, 10), "i32")
    sl = _t((B,), "i32")
    op = _t((B, S, H, 512), "f32")
    lp = _t((B, S, H), "f32")
    sc = _t((1,), "f32")

    def dec(sp=_t((B,), "i32"), wk=_t((7, 2), "i32"), op=op, lp=lp):
        return lib.pkv_paged_mla_decode_planned(ql, qp, ckv, kpe, bt, sl, 0.05, sp, wk, op, lp, sc, None, None)
    assert dec(sp=_t((B + 1,), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(sp=_t((B,), "f32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(wk=_t((7, 3), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(wk=_t((7,), "i32")) == _abi.PKV_ERR_INVALID_ARG
    assert dec(sp=None) == _abi.PKV_ERR_INVALID_ARG and dec(wk=None) == _abi.PKV_ERR_INVALID_ARG
    assert dec(op=_t((B, 4096, H, 512), "f32"), lp=_t((B, 4096, H), "f32")) == _abi.PKV_ERR_UNSUPPORTED
    assert dec(lp=_t((B, S + 1, H), "f32")) == _abi.PKV_ERR_INVALID_ARG
