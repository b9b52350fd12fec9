"""GPU parity of the decode step against the float64 oracle (small sizes).

Every case runs the CUDA path through the C ABI (cache fill, new-token RoPE
+ cache write, paged GQA decode, LSE merge) and the oracle on the same seeded
inputs, and compares: rotated q and every cache byte bit for bit; partial
outputs, merged output and LSE within the tolerance of tests/_compare.py.
Sizes span several pages per warp, ragged last pages, empty splits, block
tables longer than one 32-entry batch per warp, both layouts, both RoPE
styles, bf16, FP8 and NVFP4 caches (NVFP4 block scales bit for bit too),
head dims 64 and 128 and groups of 1 to 16."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_04_gb300 import _abi, harness, synth
from tests._compare import assert_close_lse, assert_close_out, bf16_u16_to_f64
from tests._pipeline import oracle_step

pytestmark = pytest.mark.gpu


def _case(name, S_list, **kw):
    return pytest.param(name, S_list, kw, id=name)


CASES = [
    _case("tiny", (1, 2)),
    _case("hnd_d128_g6_tails", (1, 3, 8), seq_lens=[1, 16, 17, 31, 32, 33, 100, 257], Hq=12, Hkv=2, D=128,
          rope_base=1e6, k_mult=0.5),
    _case("nhd_d128_g4_interleaved", (1, 2), seq_lens=[5, 48, 130], Hq=16, Hkv=4, D=128, layout="NHD",
          style="interleaved", rope_base=5e5, outlier_p=0.05),
    _case("fp8_hnd_d128_g6_head_scales", (1, 4), seq_lens=[15, 16, 17, 200], Hq=12, Hkv=2, D=128,
          cache_dtype="fp8", rope_base=1e6),
    _case("fp8_nhd_d64_g2_tensor_scale", (1, 2), seq_lens=[3, 70], Hq=4, Hkv=2, D=64, layout="NHD",
          cache_dtype="fp8", per_head_scale=False),
    _case("bf16_hnd_d64_g16", (1, 3), seq_lens=[40, 9], Hq=16, Hkv=1, D=64),
    _case("fp8_hnd_d128_g12", (2,), seq_lens=[33, 64], Hq=24, Hkv=2, D=128, cache_dtype="fp8"),
    _case("mha_nhd_d128", (1,), seq_lens=[50], Hq=3, Hkv=3, D=128, layout="NHD"),
    _case("empty_and_short", (5,), seq_lens=[0, 1, 20], Hq=8, Hkv=2, D=128),
    _case("long_blocktable_batches", (1, 2), seq_lens=[4800, 4799], Hq=7, Hkv=1, D=128, rope_base=1e6),
    _case("nvfp4_hnd_d128_g6_tails", (1, 3, 8), seq_lens=[1, 15, 16, 17, 31, 33, 100, 257], Hq=12, Hkv=2,
          D=128, cache_dtype="nvfp4", rope_base=1e6),
    _case("nvfp4_hnd_d64_g2_tensor_scale", (1, 2), seq_lens=[3, 70], Hq=4, Hkv=2, D=64, cache_dtype="nvfp4",
          per_head_scale=False),
    _case("nvfp4_hnd_d128_g12_interleaved", (2,), seq_lens=[33, 64], Hq=24, Hkv=2, D=128, cache_dtype="nvfp4",
          style="interleaved", rope_base=5e5, outlier_p=0.05),
    _case("nvfp4_hnd_d64_g16", (1, 3), seq_lens=[40, 9], Hq=16, Hkv=1, D=64, cache_dtype="nvfp4"),
    _case("nvfp4_empty_and_short", (5,), seq_lens=[0, 1, 20], Hq=8, Hkv=2, D=128, cache_dtype="nvfp4"),
    _case("nvfp4_long_blocktable_batches", (1, 2), seq_lens=[4800, 4799], Hq=8, Hkv=1, D=128,
          cache_dtype="nvfp4", rope_base=1e6),
]


def _workload(name, kw):
    return synth.make_workload("tiny") if name == "tiny" else synth.custom_workload(name, 101, **kw)


def run_and_compare(w, S, dw=None):
    if dw is None:
        dw = harness.DeviceWorkload(w, num_splits=S)
        dw.fill()
        dw.upload_decode()
    else:
        dw.set_splits(S)
    dw.err.zero_()
    dw.step()
    torch.cuda.synchronize()
    st = oracle_step(w, num_splits=S)
    d = dw.decode_inputs
    assert np.array_equal(dw.bf16_u16(d["q"]), st["q_rot"]), "rotated q bytes"
    for b in range(w.B):
        n = int(w.pages_per_seq[b])
        if n == 0:
            continue
        pairs = [(dw.k_cache, st["k_cache"]), (dw.v_cache, st["v_cache"])]
        if dw.nvfp4:
            pairs += [(dw.k_block_scale, st["k_block_scale"]), (dw.v_block_scale, st["v_block_scale"])]
        for gc, oc in pairs:
            got = dw.cache_pages_u(gc, w.block_tables[b, :n])
            assert np.array_equal(got, oc[st["block_tables"][b, :n]]), f"cache bytes of sequence {b}"
    assert_close_out(dw.out_partial.cpu().numpy(), st["out_partial"], "out_partial")
    assert_close_lse(dw.lse_partial.cpu().numpy(), st["lse_partial"], "lse_partial")
    assert_close_out(bf16_u16_to_f64(dw.bf16_u16(dw.out)), st["out"], "out")
    assert_close_lse(dw.lse.cpu().numpy(), st["lse"], "lse")
    assert int(dw.err.item()) == 0
    return dw


@pytest.mark.parametrize("name,S_list,kw", CASES)
def test_decode_step_parity(name, S_list, kw):
    w = _workload(name, kw)
    dw = None
    for S in S_list:
        if dw is not None:  # re-run the step on unrotated q with another split count
            dw.decode_inputs["q"].copy_(dw.decode_inputs["q0"])
        dw = run_and_compare(w, S, dw)


@pytest.mark.parametrize("scale", [1.0, 0.0137, 3.5])
def test_e4m3_write_exhaustive_over_bf16(scale):
    """Every finite bf16 pattern, written as v (no rotation) and as k at
    position 0 (identity rotation), to an FP8 cache with the given scale:
    the bytes equal the oracle's encoder of f32(x / scale). Also the bf16
    cache path for the same values."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # the NaN patterns (signalling ones raise "invalid"), replaced below
        fin = np.isfinite(bf16_u16_to_f64(pats))
    pats = np.where(fin, pats, 0).astype(np.uint16)
    D, T = 128, 512
    vals = pats.reshape(T, 1, D)
    for cache_dtype in ("fp8", "bf16"):
        w = synth.custom_workload("exh", 5, [T], 1, 1, D, cache_dtype=cache_dtype)
        kc_ref = oracle.empty_cache(w.cache_shape(), cache_dtype)
        vc_ref = np.zeros_like(kc_ref)
        sc = np.array([scale], np.float32)
        cs = np.zeros((1, D), np.float32)
        cs[0, :D // 2] = 1.0
        pos = np.zeros(T, np.int32)
        slots = np.arange(T, dtype=np.int32)
        oracle.rope_kv_write(None, vals, vals, pos, cs, kc_ref, vc_ref, slots, "HND", "neox",
                             sc if cache_dtype == "fp8" else None, sc if cache_dtype == "fp8" else None)
        dw = harness.DeviceWorkload(w, num_splits=1)
        dw.cos_sin = torch.from_numpy(cs).cuda()
        if cache_dtype == "fp8":
            dw.k_scale = torch.from_numpy(sc).cuda()
            dw.v_scale = torch.from_numpy(sc).cuda()
        kv = harness._u16_to_bf16(vals, "cuda")
        dw.write(None, kv, kv, torch.from_numpy(pos).cuda(), torch.from_numpy(slots).cuda())
        torch.cuda.synchronize()
        pages = np.arange(T // 16)
        assert np.array_equal(dw.cache_pages_u(dw.k_cache, pages), kc_ref)
        assert np.array_equal(dw.cache_pages_u(dw.v_cache, pages), vc_ref)


@pytest.mark.parametrize("style", synth.STYLES)
@pytest.mark.parametrize("layout", synth.LAYOUTS)
@pytest.mark.parametrize("cache_dtype", synth.CACHE_DTYPES)
def test_rope_write_random_positions(style, layout, cache_dtype):
    """4096 tokens at random positions of a 8192-row table, written to a
    shuffled set of slots: q, k and v bytes bit-exact."""
    T, Hq, Hkv, D = 4096, 8, 2, 128
    key = synth.stream_key(17, style + layout + cache_dtype)
    q = synth.f32_to_bf16_trunc(synth.normal_f32(key, T * Hq * D) * 3).reshape(T, Hq, D)
    k = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(18, "k"), T * Hkv * D) * 3).reshape(T, Hkv, D)
    v = synth.f32_to_bf16_trunc(synth.normal_f32(synth.stream_key(18, "v"), T * Hkv * D) * 3).reshape(T, Hkv, D)
    cs = synth.cos_sin_table(8192, D, 1e6)
    pos = (synth.uniform(synth.stream_key(19, "p"), T) * 8192).astype(np.int32)
    pool = 512
    slots = np.argsort(synth.uniform(synth.stream_key(19, "s"), pool * 16))[:T].astype(np.int32)
    w = synth.custom_workload("rw", 20, [16], Hq, Hkv, D, layout=layout, style=style, cache_dtype=cache_dtype,
                              num_pages=pool)
    kc = oracle.empty_cache(w.cache_shape(), cache_dtype); vc = np.zeros_like(kc)
    q_ref = q.copy()
    oracle.rope_kv_write(q_ref, k, v, pos, cs, kc, vc, slots, layout, style, w.k_scale, w.v_scale)
    dw = harness.DeviceWorkload(w, num_splits=1)
    dw.cos_sin = torch.from_numpy(cs).cuda()
    qg = harness._u16_to_bf16(q, "cuda")
    dw.write(qg, harness._u16_to_bf16(k, "cuda"), harness._u16_to_bf16(v, "cuda"), torch.from_numpy(pos).cuda(),
             torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(dw.bf16_u16(qg), q_ref)
    assert np.array_equal(dw.cache_pages_u(dw.k_cache, np.arange(pool)), kc)
    assert np.array_equal(dw.cache_pages_u(dw.v_cache, np.arange(pool)), vc)
    assert int(dw.err.item()) == 0


def test_page_permutation_gives_identical_output():
    """The same logical cache in a differently shuffled pool gives a
    bit-identical GPU output (pages are read in logical order)."""
    kw = dict(seq_lens=[37, 300, 16], Hq=12, Hkv=2, D=128)
    w1 = synth.custom_workload("perm", 30, num_pages=64, **kw)
    outs = []
    for seed_off in (0, 1):
        w = synth.custom_workload("perm", 30, num_pages=64, **kw)
        if seed_off:
            perm = np.argsort(synth.uniform(synth.stream_key(31, "perm"), 64)).astype(np.int32)
            w.block_tables = np.where(w1.block_tables >= 0, perm[np.maximum(w1.block_tables, 0)], -1).astype(np.int32)
        dw = harness.DeviceWorkload(w, num_splits=3)
        dw.fill()
        dw.upload_decode()
        dw.step()
        torch.cuda.synchronize()
        outs.append((dw.bf16_u16(dw.out), dw.lse.cpu().numpy(), dw.out_partial.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][2], outs[1][2])


@pytest.mark.parametrize("D,S", [(64, 37), (128, 37), (128, 1), (128, 32), (128, 33), (64, 100), (128, 1000),
                                 (128, 4096)])
def test_lse_merge_random_partials(D, S):
    """Both merge forms: one warp per row (S <= 32) and the two-level tree
    (S > 32: 32 warps per 64-column slice; past 256 splits more than one
    batch of loads per warp)."""
    B, Hq = (5, 6) if S <= 1000 else (2, 3)
    op = synth.normal_f32(synth.stream_key(40, "o"), B * S * Hq * D).reshape(B, S, Hq, D)
    lp = (synth.normal_f32(synth.stream_key(40, "l"), B * S * Hq) * 4).reshape(B, S, Hq)
    lp[0, :, 0] = -np.inf                       # an all-empty row
    lp[1, 3:, :] = -np.inf                      # empty tail splits
    op[1, 3:, :, :] = 0.0
    if S > 40:
        lp[0, : S // 2, 1] = -np.inf            # a row whose first half is empty (whole warps' chunks)
        op[0, : S // 2, 1, :] = 0.0
    out_ref, lse_ref = oracle.lse_merge(op.astype(np.float64), lp.astype(np.float64))
    opg = torch.from_numpy(op).cuda(); lpg = torch.from_numpy(lp).cuda()
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    _abi.lse_merge(opg, lpg, out, lse)
    torch.cuda.synchronize()
    assert_close_out(bf16_u16_to_f64(harness.DeviceWorkload.bf16_u16(out)), out_ref)
    assert_close_lse(lse.cpu().numpy(), lse_ref)


def test_back_to_back_steps_and_step_graphs_match_a_single_step():
    """Steps issued back to back (decode and merge start early behind their
    predecessors) and the CUDA-graph forms of the step give bit-identical
    results to one synchronised step."""
    w = synth.custom_workload("b2b", 60, [700, 33, 1500, 250], 12, 2, 128, rope_base=1e6)
    dw = harness.DeviceWorkload(w, num_splits=3)
    dw.fill()
    d = dw.upload_decode()
    dw.step()
    torch.cuda.synchronize()
    ref = (dw.bf16_u16(dw.out), dw.lse.cpu().numpy(), dw.out_partial.cpu().numpy(), dw.bf16_u16(d["q"]))
    ref_k = dw.cache_pages_u(dw.k_cache, np.arange(w.num_pages))

    def same():
        assert np.array_equal(dw.bf16_u16(dw.out), ref[0])
        assert np.array_equal(dw.lse.cpu().numpy(), ref[1])
        assert np.array_equal(dw.out_partial.cpu().numpy(), ref[2])
        assert np.array_equal(dw.bf16_u16(d["q"]), ref[3])

    for _ in range(6):
        d["q"].copy_(d["q0"])
        dw.step()
    torch.cuda.synchronize()
    same()
    g = harness.StepGraph(dw)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    same()
    dw.out.zero_()
    g2 = harness.StepGraph(dw, host_io=True)
    g2.replay()
    torch.cuda.synchronize()
    same()
    assert np.array_equal(g2.out_h.view(torch.int16).numpy().view(np.uint16), ref[0])
    assert np.array_equal(dw.cache_pages_u(dw.k_cache, np.arange(w.num_pages)), ref_k)
    assert int(dw.err.item()) == 0


@pytest.mark.parametrize("cache_dtype", synth.CACHE_DTYPES)
def test_packed_qkv_views(cache_dtype):
    """q, k and v given as strided views of one packed [T, Hq + 2 Hkv, D]
    projection output (no copies): same bytes as contiguous inputs; the
    decode then reads q from the same packed buffer."""
    w = synth.custom_workload("packed", 80, [23, 64, 130], 12, 2, 128, cache_dtype=cache_dtype, rope_base=1e6)
    ref = harness.DeviceWorkload(w, num_splits=2)
    ref.fill()
    d = ref.upload_decode()
    ref.step()
    torch.cuda.synchronize()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    packed = torch.empty((B, Hq + 2 * Hkv, D), dtype=torch.bfloat16, device="cuda")
    packed[:, :Hq] = d["q0"]
    packed[:, Hq:Hq + Hkv] = d["k"]
    packed[:, Hq + Hkv:] = d["v"]
    q, k, v = packed[:, :Hq], packed[:, Hq:Hq + Hkv], packed[:, Hq + Hkv:]
    assert not q.is_contiguous()
    dw = harness.DeviceWorkload(w, num_splits=2)
    dw.fill()
    dw.write(q, k, v, d["positions"], d["slot_mapping"])
    dw.decode(q)
    dw.merge()
    torch.cuda.synchronize()
    assert np.array_equal(dw.bf16_u16(q), ref.bf16_u16(d["q"]))
    for cache in ("k_cache", "v_cache"):
        assert torch.equal(getattr(dw, cache), getattr(ref, cache))
    assert np.array_equal(dw.bf16_u16(dw.out), ref.bf16_u16(ref.out))
    assert torch.equal(dw.lse, ref.lse)


def test_validate_without_slots_and_strided_tables():
    """Block tables given as a column slice of a wider buffer, and no slot
    mapping: only the sequence checks run."""
    w = synth.custom_workload("val2", 81, [40, 3, 100], 4, 2, 128, num_pages=30)
    wide = np.full((w.B, w.max_pages + 5), 7, np.int32)
    wide[:, 2:2 + w.max_pages] = w.block_tables
    bt = torch.from_numpy(wide).cuda()[:, 2:2 + w.max_pages]
    assert not bt.is_contiguous()
    sl = torch.from_numpy(w.seq_lens).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _abi.validate_indices(bt, sl, None, w.num_pages, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bt[1, 0] = -5
    _abi.validate_indices(bt, sl, None, w.num_pages, err)
    torch.cuda.synchronize()
    assert int(err.item()) == _abi.FLAG_PAGE_RANGE


def _e4m3_midpoints():
    """Positive midpoints between consecutive E4M3 magnitudes, normal range
    and below (from the oracle's decode table), plus the saturation edge."""
    mags = np.array(sorted(v for v in oracle.e4m3_table()[:127]), np.float64)
    mids = (mags[1:] + mags[:-1]) / 2
    return np.concatenate([mids, [448.0, 464.0, 2.0 ** -6, 2.0 ** -9]])


@pytest.mark.parametrize("scale", [0.0137, 0.05, 1.0 / 3.0, 0.1, 3.5])
def test_fp8_write_near_every_rounding_boundary(scale):
    """Arbitrary float32 values reach the quantiser through the table:
    with k = [1 .. 1 | 0 .. 0] (NeoX halves), the rotated row is exactly
    (cos_i, sin_i). Values are placed at scale * (each E4M3 midpoint) and up
    to 8 float steps either side, both signs: the E4M3 bytes must equal the
    oracle's f32(y / scale) encoding."""
    D = 128
    sc = np.float32(scale)
    base = (_e4m3_midpoints() * np.float64(sc)).astype(np.float32)
    vals = []
    for k in range(-8, 9):
        vals.append((base.view(np.int32) + k).view(np.float32))
    vals = np.concatenate(vals)
    vals = np.concatenate([vals, -vals])
    T = (len(vals) + D - 1) // D
    vals = np.resize(vals, T * D).astype(np.float32)
    cs = vals.reshape(T, D).copy()                    # row t: cos half, sin half
    k = np.zeros((T, 1, D), np.uint16)
    k[:, 0, :D // 2] = 0x3F80                         # 1.0 in bf16; second half 0
    v = np.zeros_like(k)
    pos = np.arange(T, dtype=np.int32)
    slots = np.arange(T, dtype=np.int32)
    w = synth.custom_workload("mid", 6, [max(T, 1)], 1, 1, D, cache_dtype="fp8", num_pages=(T + 15) // 16)
    sca = np.array([sc], np.float32)
    kc = oracle.empty_cache(w.cache_shape(), "fp8"); vc = np.zeros_like(kc)
    oracle.rope_kv_write(None, k, v, pos, cs, kc, vc, slots, "HND", "neox", sca, sca)
    dw = harness.DeviceWorkload(w, num_splits=1)
    dw.cos_sin = torch.from_numpy(cs).cuda()
    dw.k_scale = torch.from_numpy(sca).cuda()
    dw.v_scale = torch.from_numpy(sca).cuda()
    dw.write(None, harness._u16_to_bf16(k, "cuda"), harness._u16_to_bf16(v, "cuda"), torch.from_numpy(pos).cuda(),
             torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    got = dw.cache_pages_u(dw.k_cache, np.arange(w.num_pages))
    assert np.array_equal(got, kc)
    assert int(dw.err.item()) == 0
