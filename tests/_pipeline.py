"""Oracle-side assembly of a decode step for a synthetic workload.

Test infrastructure: drives the float64 oracle over a workload from the
seeded generators. For a subset of sequences it builds a compact page pool
(the sequences' pages renumbered 0..n-1), which holds the same logical
contents as the full pool, so a sample of a large workload can be checked
without materialising all of it on the host."""
import numpy as np

import oracle
from paged_kv_gqa_04_gb300 import synth


def oracle_step(w: synth.Workload, seqs=None, num_splits: int = 1):
    """Run the oracle's cache write (context tokens, then the new token with
    q) and decode + merge for the given sequences.

    Returns dict(q_rot [n,Hq,D] uint16, k_cache, v_cache (compact pool),
    block_tables [n, maxp], seq_lens [n], out_partial, lse_partial, out, lse)."""
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    n = len(seqs)
    P = w.page_size
    npg = [int((int(w.seq_lens[b]) + P - 1) // P) for b in seqs]
    width = max(1, max(npg) if npg else 1)
    bt = np.full((n, width), -1, np.int32)
    base = 0
    for i, c in enumerate(npg):
        bt[i, :c] = np.arange(base, base + c, dtype=np.int32)
        base += c
    pool = max(base, 1)
    nv = w.cache_dtype == "nvfp4"
    last = w.D // 2 if nv else w.D
    shape = (pool, w.Hkv, P, last) if w.layout == "HND" else (pool, P, w.Hkv, last)
    kc = oracle.empty_cache(shape, w.cache_dtype)
    vc = np.zeros_like(kc)
    if nv:
        sshape = shape[:3] + (w.D // 16,)
        ksc = np.zeros(sshape, np.uint8)
        vsc = np.zeros(sshape, np.uint8)

    def write(q, k, v, pos, slots):
        if nv:
            oracle.rope_kv_write_nvfp4(q, k, v, pos, cs, kc, vc, ksc, vsc, slots, w.layout, w.style,
                                       w.k_scale, w.v_scale)
        else:
            oracle.rope_kv_write(q, k, v, pos, cs, kc, vc, slots, w.layout, w.style, w.k_scale, w.v_scale)
    cs = w.cos_sin()
    q_rot = np.zeros((n, w.Hq, w.D), np.uint16)
    sl = np.array([int(w.seq_lens[b]) for b in seqs], np.int32)
    for i, b in enumerate(seqs):
        L = int(w.seq_lens[b])
        if L == 0:
            # no token to write (its slot is -1): q stays as it came
            q_rot[i] = w.seq_q(b)
            continue
        k, v = w.seq_kv(b)
        pos = np.arange(L, dtype=np.int32)
        slots = (bt[i, pos // P].astype(np.int64) * P + pos % P).astype(np.int32)
        # context tokens (no q) ...
        if L > 1:
            write(None, k[:L - 1], v[:L - 1], pos[:L - 1], slots[:L - 1])
        # ... then the new token with its q
        q = w.seq_q(b).reshape(1, w.Hq, w.D).copy()
        write(q, k[L - 1:], v[L - 1:], pos[L - 1:], slots[L - 1:])
        q_rot[i] = q[0]
    if nv:
        op, lp = oracle.paged_decode_nvfp4(q_rot, kc, vc, ksc, vsc, bt, sl, w.softmax_scale, num_splits, w.layout,
                                           w.k_scale, w.v_scale)
    else:
        op, lp = oracle.paged_decode(q_rot, kc, vc, bt, sl, w.softmax_scale, num_splits, w.layout,
                                     w.k_scale, w.v_scale)
    out, lse = oracle.lse_merge(op, lp)
    r = dict(q_rot=q_rot, k_cache=kc, v_cache=vc, block_tables=bt, seq_lens=sl,
             out_partial=op, lse_partial=lp, out=out, lse=lse)
    if nv:
        r.update(k_block_scale=ksc, v_block_scale=vsc)
    return r


def cache_values_f64(cache: np.ndarray, cache_dtype: str) -> np.ndarray:
    """Cache bytes as float64 through torch's own dtype views (independent of
    the oracle's decoders)."""
    import torch
    if cache_dtype == "fp8":
        t = torch.from_numpy(cache.view(np.uint8)).view(torch.float8_e4m3fn)
    else:
        t = torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


# The 16 E2M1 code values, written out from the OCP Microscaling Formats
# definition of the FP4 (e2m1) element: codes 0-7 positive, 8-15 negative.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], np.float64)


def nvfp4_values_f64(cache: np.ndarray, block_scale: np.ndarray) -> np.ndarray:
    """NVFP4 cache [.., D/2] packed bytes + [.., D/16] E4M3 scale bytes ->
    float64 values [.., D] (without the static per-head scale), decoded with
    the literal E2M1 table and torch's float8_e4m3fn view for the scales
    (independent of the oracle's decoders)."""
    import torch
    lo = E2M1_VALUES[cache & 0xF]
    hi = E2M1_VALUES[cache >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(cache.shape[:-1] + (2 * cache.shape[-1],))
    s = torch.from_numpy(np.ascontiguousarray(block_scale)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(s, 16, axis=-1)


def mla_oracle_step(w: synth.MlaWorkload, seqs=None, num_splits: int = 1):
    """The oracle's MLA cache write (context, then the new token with q_pe)
    and decode + merge for the given sequences, on a compact pool.

    Returns dict(q_lat, q_pe_rot [n,H,*] uint16, ckv_cache [pool,P,Dc] uint8,
    kpe_cache [pool,P,Dr] uint16, block_tables, seq_lens, out_partial,
    lse_partial, out, lse)."""
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    n = len(seqs)
    P = w.page_size
    npg = [int((int(w.seq_lens[b]) + P - 1) // P) for b in seqs]
    width = max(1, max(npg) if npg else 1)
    bt = np.full((n, width), -1, np.int32)
    base = 0
    for i, c in enumerate(npg):
        bt[i, :c] = np.arange(base, base + c, dtype=np.int32)
        base += c
    pool = max(base, 1)
    ckv_cache = np.zeros((pool, P, w.Dc), np.uint8)
    kpe_cache = np.zeros((pool, P, w.Dr), np.uint16)
    cs = w.cos_sin()
    q_lat = np.zeros((n, w.H, w.Dc), np.uint16)
    q_pe = np.zeros((n, w.H, w.Dr), np.uint16)
    sl = np.array([int(w.seq_lens[b]) for b in seqs], np.int32)
    for i, b in enumerate(seqs):
        L = int(w.seq_lens[b])
        ql, qp = w.seq_q(b)
        q_lat[i] = ql
        if L == 0:
            q_pe[i] = qp
            continue
        ckv, kpe = w.seq_latent(b)
        pos = np.arange(L, dtype=np.int32)
        slots = (bt[i, pos // P].astype(np.int64) * P + pos % P).astype(np.int32)
        if L > 1:
            oracle.mla_cache_write(None, ckv[:L - 1], kpe[:L - 1], pos[:L - 1], cs, ckv_cache, kpe_cache,
                                   slots[:L - 1], w.ckv_scale, w.style)
        qpr = qp.reshape(1, w.H, w.Dr).copy()
        oracle.mla_cache_write(qpr, ckv[L - 1:], kpe[L - 1:], pos[L - 1:], cs, ckv_cache, kpe_cache, slots[L - 1:],
                               w.ckv_scale, w.style)
        q_pe[i] = qpr[0]
    op, lp = oracle.mla_decode(q_lat, q_pe, ckv_cache, kpe_cache, bt, sl, w.softmax_scale, num_splits, w.ckv_scale)
    out, lse = oracle.lse_merge(op, lp)
    return dict(q_lat=q_lat, q_pe_rot=q_pe, ckv_cache=ckv_cache, kpe_cache=kpe_cache, block_tables=bt,
                seq_lens=sl, out_partial=op, lse_partial=lp, out=out, lse=lse)
