"""Benchmark of the paged-KV GQA decode step on GB300.

One step = the whole hot path over one batch: fused RoPE + paged-KV write of
the new token (q rotated in place), paged GQA split-K decode, LSE merge --
three launches of the library's kernels through the C ABI.

Default workload: the Qwen2.5-1.5B-shaped decode (batch 32, seq_lens uniform
in [512, 4096], 12 query / 2 kv heads, head dim 128, page size 16, HND, bf16
cache, NeoX RoPE base 1e6, 12000-page shuffled pool). The cache holds every
context token (written by the library's cache-write call before timing).

Timing: W warm-up steps, then exactly K steps between a barrier and a device
synchronise on each side. Before every timed step the L2 is flushed (a 512 MiB
device write, then a 512 MiB read so that the write-back of dirty lines also
happens before the step) and q is restored from its unrotated copy, both
outside the step's CUDA events. Events on the launching stream bracket each
step (the launches chained as a program issues them); a second pass puts an
event between the launches for each kernel's own time. Reported:
  value       tokens/s = B*K / sum of step times (inputs resident in HBM)
  e2e         the same through the Python binding with host buffers: every
              step copies its inputs from pinned host memory to the device and
              its output (out, lse) back (pkv_copy), inside the step's events
  roofline    of the decode kernel: algorithmic bytes (Q + K/V pages + block-
              table entries + output) / its mean event time, against the
              measured HBM copy bandwidth
  cache_write GB/s of one cache-fill call over all context tokens
  cpu_baseline the float64 oracle on the host, single thread
`--impl reference` times that oracle alone as the reference arm.
Under torchrun with N > 1 every rank runs an independent replica (weak
scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode-attn KV-read GB/s & % of HBM peak; tokens/s/step; RoPE+KV-write GB/s"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20

WORKLOAD_TEXT = {
    "qwen": "Qwen2.5-1.5B-shaped paged GQA decode: B32, seq_lens ~U[512,4096], 12 q / 2 kv heads (GQA 6), "
            "D128, page 16, HND, bf16 cache, NeoX RoPE base 1e6, 12000-page shuffled pool",
    "longctx": "long-context decode: B2, seq_len 32768, 28 q / 4 kv heads (GQA 7), D128, page 16, HND, bf16, "
               "8192-page fragmented pool",
    "ragged": "ragged large-batch decode: B256, lognormal seq_lens (median 1024, sigma 1, [1,8192]), 32 q / 8 kv "
              "heads (GQA 4), D128, NHD, interleaved RoPE 5e5, 1% outlier K rows x8",
    "fp8": "FP8 E4M3 paged cache decode: B64, seq_lens ~U[2048,16384], 12 q / 2 kv heads, D128, HND, per-head "
           "static K/V scales ~U[0.01,0.1]",
    "tiny": "tiny paged GQA decode: B2, seq_lens {37,100}, 4 q / 2 kv heads, D64, HND",
    "million": "1M-token decode: B1, seq_len 1048576, 8 q / 1 kv heads (GQA 8), D128, page 16, HND, bf16, "
               "65536-page shuffled pool",
    "fp4": "NVFP4 paged cache decode (E2M1 values + E4M3 scale per 16 + per-head static scale ~U[0.5,1.5]): "
           "B64, seq_lens ~U[2048,16384], 12 q / 2 kv heads, D128, HND",
    "mla": "paged MLA decode (absorbed form; latent 512 E4M3 + positional 64 bf16 per token, 64-token pages): "
           "B1, seq_len 51200 (800 pages), 8 heads -- mainarch's MLA run",
    "mla_batch": "paged MLA decode (absorbed form, 64-token pages): B32, seq_lens ~U[4096,16384], 16 heads",
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default="qwen", choices=sorted(WORKLOAD_TEXT))
    p.add_argument("--splits", type=int, default=0, help="num_splits (0 = the library's heuristic)")
    p.add_argument("--also", default="longctx,ragged,fp8,million,fp4,mla,mla_batch",
                   help="extra workloads whose decode roofline is reported under 'other_workloads' ('' = none)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--clock-window", type=float, default=1.0,
                   help="seconds of untimed steps run under the clock sampler before the timed steps")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


# ---- distributed plumbing (replicas only) -----------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- clocks --------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def is_mla(name: str) -> bool:
    return name.startswith("mla")


def kernel_names(name: str) -> tuple:
    """(cache write, decode, merge) entry points of a workload's step."""
    if is_mla(name):
        return "mla_cache_write", "paged_mla_decode", "lse_merge"
    return "rope_kv_write", "paged_gqa_decode", "lse_merge"


def decode_kernel_source_hash(name: str = "qwen") -> str:
    f = "mla_decode.cu" if is_mla(name) else "paged_decode.cu"
    src = open(os.path.join(ROOT, "paged_kv_gqa_04_gb300", "csrc", f), "rb").read()
    return hashlib.sha256(src).hexdigest()[:16]


def ncu_traffic(workload: str, num_splits: int):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if it was taken on the current kernel source and with the
    same split count (else None)."""
    p = os.path.join(ROOT, "profiles", f"{kernel_names(workload)[1]}_{workload}.md")
    try:
        txt = open(p).read()
    except OSError:
        return None
    h = t = s = None
    for line in txt.splitlines():
        key, _, val = line.partition(":")
        try:
            if key == "kernel_source_sha256_16":
                h = val.strip()
            elif key == "dram_bytes_per_launch":
                t = float(val.strip())
            elif key == "num_splits":
                s = int(val.strip())
        except ValueError:
            return None
    return t if (h == decode_kernel_source_hash(workload) and s == num_splits and t) else None


# ---- byte counts ---------------------------------------------------------------------
def decode_alg_bytes(w) -> float:
    """Q + K/V pages of every sequence (values and any block scales) +
    block-table entries read + bf16 out. MLA: q_lat + q_pe, the latent rows
    (512 E4M3 + 64 bf16 per token), block-table entries, the 512-wide out."""
    if hasattr(w, "Dc"):
        q = w.B * w.H * (w.Dc + w.Dr) * 2
        kv = float(w.seq_lens.astype(np.int64).sum()) * (w.Dc + 2 * w.Dr)
        bt = float(w.pages_per_seq.sum()) * 4
        return q + kv + bt + w.B * w.H * w.Dc * 2
    e = w.cache_bytes_per_value
    q = w.B * w.Hq * w.D * 2
    kv = float(w.seq_lens.astype(np.int64).sum()) * w.Hkv * w.D * 2 * e
    bt = float(w.pages_per_seq.sum()) * 4
    out = w.B * w.Hq * w.D * 2
    return q + kv + bt + out


def partial_bytes(w, S) -> float:
    if hasattr(w, "Dc"):
        return 2.0 * w.B * S * w.H * (w.Dc + 1) * 4
    return 2.0 * w.B * S * w.Hq * (w.D + 1) * 4


def write_alg_bytes(w, T: int, with_q: bool, table_rows=None) -> float:
    """q read+write (if given) + k, v read + cache write + position and slot
    + one cos_sin row per token; with table_rows, the cos_sin rows are
    counted once per distinct position instead (rows shared by tokens at the
    same position are read from L2, not HBM). MLA (no q): ckv and kpe read
    (bf16), E4M3 ckv and bf16 kpe written, position and slot, one 64-value
    cos_sin row."""
    if hasattr(w, "Dc"):
        assert not with_q
        per = w.Dc * 2 + w.Dr * 2 + w.Dc + w.Dr * 2 + 8
        rows = T if table_rows is None else table_rows
        return float(T) * per + float(rows) * w.Dr * 4
    e = w.cache_bytes_per_value
    per = 2 * w.Hkv * w.D * 2 + 2 * w.Hkv * w.D * e + 8
    if with_q:
        per += 2 * w.Hq * w.D * 2
    rows = T if table_rows is None else table_rows
    return float(T) * per + float(rows) * w.D * 4


# ---- GPU measurements ----------------------------------------------------------------
class L2Flush:
    """Before each timed step: write a 512 MiB buffer (every cached line of
    the step's data is evicted), then read another 512 MiB buffer with the
    library's streaming read, so that the L2 is left holding clean lines:
    the write's own dirty lines are written back here, outside the events,
    not during the timed kernels."""

    def __init__(self):
        from paged_kv_gqa_04_gb300 import _abi
        self._abi = _abi
        self.wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.rbuf = torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        self.sink = torch.empty(4 * sms, dtype=torch.int32, device="cuda")

    def zero_(self) -> None:
        self.wbuf.zero_()
        self._abi.stream_read(self.rbuf, self.sink)


def flush_buffer():
    return L2Flush()


def time_steps(dw, steps: int, warmup: int, world: int, flush, per_kernel: bool) -> dict:
    """Device-resident steps: per step flush L2 and restore q (both outside
    the events), then the step's three launches. With per_kernel, events also
    separate the launches (which stops the decode and merge kernels from
    starting early behind their predecessors); without, events bracket the
    step only."""
    d = dw.decode_inputs
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        d["q"].copy_(d["q0"])
        dw.step()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        d["q"].copy_(d["q0"])
        e = ev[i]
        e[0].record(stream)
        dw.write_step()
        if per_kernel:
            e[1].record(stream)
        dw.decode(d["q"])
        if per_kernel:
            e[2].record(stream)
        dw.merge()
        e[3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    r = dict(step_ms=[e[0].elapsed_time(e[3]) for e in ev], wall_s=wall)
    if per_kernel:
        r.update(write_ms=[e[0].elapsed_time(e[1]) for e in ev], decode_ms=[e[1].elapsed_time(e[2]) for e in ev],
                 merge_ms=[e[2].elapsed_time(e[3]) for e in ev])
    return r


def time_e2e(dw, steps: int, warmup: int, world: int, flush) -> dict:
    """Through the binding with host buffers, one CUDA-graph submission per
    step (harness.StepGraph): one pinned-host -> device copy of the step's
    packed inputs, the three C-ABI launches reading them in place, one
    device -> pinned-host copy of the packed out and lse (both copies by
    pkv_copy, the SMs reading / writing the pinned buffers); CUDA events
    around each replay."""
    from paged_kv_gqa_04_gb300 import harness
    g = harness.StepGraph(dw, host_io=True)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        g.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return dict(step_ms=[a.elapsed_time(b) for a, b in ev], h2d=g.h2d_bytes, d2h=g.d2h_bytes, B=dw.w.B)


def time_fill(dw, reps: int, flush) -> dict:
    """One cache-fill call (all context tokens, no q), timed alone."""
    fi = dw.fill_inputs()
    T = int(fi["positions"].numel())
    rows = int(torch.unique(fi["positions"]).numel())
    stream = torch.cuda.current_stream()
    for _ in range(2):
        flush.zero_()
        dw.write_fill(fi)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        dw.write_fill(fi)
        b.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    del fi
    return dict(T=T, rows=rows, ms=statistics.median(ms), ms_all=ms)


def stream_ceiling(nbytes: int, flush, reps: int = 20) -> float:
    """GB/s of one streaming-read launch (the library's pkv_stream_read) over
    the given number of bytes, L2 flushed before each launch."""
    from paged_kv_gqa_04_gb300 import _abi
    n = max(16, int(nbytes) // 16 * 16)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.empty(4 * sms, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    _abi.stream_read(buf, sink)
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        _abi.stream_read(buf, sink)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    del buf
    return n / (ms * 1e-3) / 1e9


def measure_layered(dw, layers: int, reps: int, flush, peak: float) -> dict:
    """Decode as a model's layers run it: `layers` decode launches back to
    back, each over its own cache (distinct memory, so nothing one layer
    reads is in L2 for the next), each launch free to start behind the
    previous one; L2 flushed before each group. Bytes / time of the group."""
    w = dw.w
    caches = [dw.caches()]
    for _ in range(layers - 1):
        caches.append(tuple(c.clone() for c in dw.caches()))
    d = dw.decode_inputs
    outs = [(torch.empty_like(dw.out_partial), torch.empty_like(dw.lse_partial)) for _ in range(layers)]

    def group():
        for cs, (op, lp) in zip(caches, outs):
            dw.decode_into(d["q"], cs, op, lp)
    stream = torch.cuda.current_stream()
    group()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        group()
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    gbs = layers * decode_alg_bytes(w) / (ms * 1e-3) / 1e9
    ok = all(torch.equal(op, outs[0][0]) for op, _ in outs[1:])
    del caches, outs
    return dict(layers=layers, us_per_layer=1e3 * ms / layers, gbs=gbs, frac=gbs / peak, layers_agree=ok)


def measure_decode_only(name: str, splits: int, reps: int, flush, peak: float) -> dict:
    """Decode-kernel roofline of another workload (filled, then `reps`
    flushed launches)."""
    from paged_kv_gqa_04_gb300 import harness
    dw = harness.make_device_workload(name, num_splits=splits or None)
    w = dw.w
    dw.fill()
    d = dw.upload_decode()
    dw.step()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        dw.decode(d["q"])
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    rs = time_steps(dw, 20, 3, 1, flush, True)
    rc = time_steps(dw, 20, 3, 1, flush, False)
    step = dict(chained_us=1e3 * statistics.mean(rc["step_ms"]),
                tokens_per_s=w.B / (statistics.mean(rc["step_ms"]) * 1e-3),
                separated_us=dict(zip(kernel_names(name), (1e3 * statistics.mean(rs["write_ms"]),
                                                           1e3 * statistics.mean(rs["decode_ms"]),
                                                           1e3 * statistics.mean(rs["merge_ms"])))))
    layered = measure_layered(dw, 4 if decode_alg_bytes(w) < 1e9 else 2, 5, flush, peak)
    fill = time_fill(dw, 5, flush)
    wb = write_alg_bytes(w, fill["T"], False)
    wbu = write_alg_bytes(w, fill["T"], False, fill["rows"])
    alg = decode_alg_bytes(w)
    r = dict(workload=WORKLOAD_TEXT[name], num_splits=dw.num_splits, decode_us=ms * 1e3,
             decode_gbs=alg / (ms * 1e-3) / 1e9, decode_frac=alg / (ms * 1e-3) / 1e9 / peak,
             cache_write_gbs=wb / (fill["ms"] * 1e-3) / 1e9,
             cache_write_frac=wb / (fill["ms"] * 1e-3) / 1e9 / peak,
             cache_write_frac_table_rows_once=wbu / (fill["ms"] * 1e-3) / 1e9 / peak, err_flag=int(dw.err.item()),
             stream_read_frac_same_bytes=stream_ceiling(alg, flush) / peak, layered=layered, step=step)
    del dw
    torch.cuda.empty_cache()
    return r


# ---- CPU oracle -------------------------------------------------------------------------
def oracle_step_timer(w, seqs, num_splits):
    """Prepare the oracle's cache for `seqs` (untimed) and return a function
    that runs one oracle decode step over them (new-token write with q,
    decode, merge) and returns its seconds."""
    import oracle
    from tests._pipeline import mla_oracle_step, oracle_step
    if hasattr(w, "Dc"):  # MLA
        st = mla_oracle_step(w, seqs=seqs, num_splits=num_splits)
        db = w.decode_batch()
        qp0 = db["q_pe"][seqs].copy()
        ckv, kpe, pos = db["ckv"][seqs], db["kpe"][seqs], db["positions"][seqs]
        P = w.page_size
        bt = st["block_tables"]
        slots = np.array([bt[i, p // P] * P + p % P if w.seq_lens[b] > 0 else -1
                          for i, (b, p) in enumerate(zip(seqs, pos))], np.int32)
        cs = w.cos_sin()

        def run_mla() -> float:
            qp = qp0.copy()
            t0 = time.perf_counter()
            oracle.mla_cache_write(qp, ckv, kpe, pos, cs, st["ckv_cache"], st["kpe_cache"], slots, w.ckv_scale,
                                   w.style)
            op, lp = oracle.mla_decode(st["q_lat"], qp, st["ckv_cache"], st["kpe_cache"], bt, st["seq_lens"],
                                       w.softmax_scale, num_splits, w.ckv_scale)
            oracle.lse_merge(op, lp)
            return time.perf_counter() - t0
        return run_mla
    st = oracle_step(w, seqs=seqs, num_splits=num_splits)
    db = w.decode_batch()
    q0 = db["q"][seqs].copy()
    k = db["k"][seqs]
    v = db["v"][seqs]
    pos = db["positions"][seqs]
    P = w.page_size
    bt = st["block_tables"]
    slots = np.array([bt[i, p // P] * P + p % P if w.seq_lens[b] > 0 else -1
                      for i, (b, p) in enumerate(zip(seqs, pos))], np.int32)
    cs = w.cos_sin()

    def run() -> float:
        q = q0.copy()
        t0 = time.perf_counter()
        if w.cache_dtype == "nvfp4":
            oracle.rope_kv_write_nvfp4(q, k, v, pos, cs, st["k_cache"], st["v_cache"], st["k_block_scale"],
                                       st["v_block_scale"], slots, w.layout, w.style, w.k_scale, w.v_scale)
            op, lp = oracle.paged_decode_nvfp4(q, st["k_cache"], st["v_cache"], st["k_block_scale"],
                                               st["v_block_scale"], bt, st["seq_lens"], w.softmax_scale,
                                               num_splits, w.layout, w.k_scale, w.v_scale)
        else:
            oracle.rope_kv_write(q, k, v, pos, cs, st["k_cache"], st["v_cache"], slots, w.layout, w.style,
                                 w.k_scale, w.v_scale)
            op, lp = oracle.paged_decode(q, st["k_cache"], st["v_cache"], bt, st["seq_lens"], w.softmax_scale,
                                         num_splits, w.layout, w.k_scale, w.v_scale)
        oracle.lse_merge(op, lp)
        return time.perf_counter() - t0
    return run


def cpu_baseline(w, num_splits, seconds: float) -> dict:
    run = oracle_step_timer(w, list(range(w.B)), num_splits)
    total, n = 0.0, 0
    while total < seconds or n == 0:
        total += run()
        n += 1
    return {"value": w.B * n / total, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} oracle decode steps over the whole batch ({w.B} sequences, {num_splits} splits): "
                      f"new-token cache write, decode, merge; float64, single thread; cache prepared untimed"}


_ALLCORE_BARRIER = None


def _allcore_init(barrier):
    global _ALLCORE_BARRIER
    _ALLCORE_BARRIER = barrier


def _allcore_worker(job):
    """One host process of the all-core oracle baseline: prepare its slice of
    the batch (untimed), wait for the others, then time whole steps."""
    name, seqs, num_splits, seconds = job
    from paged_kv_gqa_04_gb300 import synth
    w = synth.make_mla_workload(name) if is_mla(name) else synth.make_workload(name)
    run = oracle_step_timer(w, seqs, num_splits)
    _ALLCORE_BARRIER.wait()
    total, n = 0.0, 0
    while total < seconds or n == 0:
        total += run()
        n += 1
    return len(seqs) * n / total


def cpu_baseline_allcore(name, B, num_splits, seconds: float) -> dict:
    """The oracle on every host core: one process per core (spawned: this
    process has initialised CUDA), the batch's sequences dealt round-robin,
    all timed over the same window; throughput = the sum of the processes'."""
    import multiprocessing as mp
    procs = max(1, min(os.cpu_count() or 1, B))
    groups = [list(range(i, B, procs)) for i in range(procs)]
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    with ctx.Pool(procs, initializer=_allcore_init, initargs=(barrier,)) as pool:
        rates = pool.map(_allcore_worker, [(name, g, num_splits, seconds) for g in groups])
    return {"value": sum(rates), "unit": UNIT, "cores": procs, "kind": "oracle",
            "sample": f"{procs} processes, each its round-robin share of the {B} sequences, {num_splits} splits, "
                      f"whole oracle decode steps (new-token write, decode, merge) for about {seconds:g} s; "
                      f"float64, one thread each"}


def run_reference(args, world, rank):
    """Reference arm: the float64 oracle timed on the host cores."""
    if rank != 0:
        return
    from paged_kv_gqa_04_gb300 import synth
    w = synth.make_mla_workload(args.workload) if is_mla(args.workload) else synth.make_workload(args.workload)
    S = args.splits or 1
    import oracle
    oracle.build()
    # size the per-step sample so that warm-up + timed steps take about a minute
    probe = oracle_step_timer(w, [0], S)
    t1 = probe()
    n = int(max(1, min(w.B, round(60.0 / max(1, args.steps + args.warmup) / max(t1, 1e-6)))))
    seqs = list(range(n))
    run = oracle_step_timer(w, seqs, S)
    for _ in range(args.warmup):
        run()
    ts = [run() for _ in range(args.steps)]
    total = sum(ts)
    value = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "batch_sample": n, "num_splits": S},
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": 1,
                         "sample": f"each step: the first {n} of {w.B} sequences (new-token write, decode, merge)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- main -------------------------------------------------------------------------------
def main():
    args = parse_args()
    world, rank = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_gqa_04_gb300 import harness, synth

    peak, peak_kind = hbm_peak()
    dw = harness.make_device_workload(args.workload, num_splits=args.splits or None)
    w = dw.w
    dw.fill()
    dw.upload_decode()
    flush = flush_buffer()
    gpu_index = torch.cuda.current_device()
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(gpu_index)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else gpu_index)
    clocks.start()
    time.sleep(0.4)
    # keep the GPU under this load for about a second before the timed steps so
    # the clock samples describe it
    t_end = time.perf_counter() + args.clock_window
    while time.perf_counter() < t_end:
        time_steps(dw, 20, 0, 1, flush, False)
    r = time_steps(dw, args.steps, args.warmup, world, flush, False)
    clk = clocks.stop()
    rk = time_steps(dw, args.steps, args.warmup, world, flush, True)
    err = int(dw.err.item())

    step_s = sum(r["step_ms"]) * 1e-3
    step_s = max_over_ranks(step_s, world)
    value = world * w.B * args.steps / step_s
    dec_ms = statistics.mean(rk["decode_ms"])
    alg = decode_alg_bytes(w)
    achieved = alg / (dec_ms * 1e-3) / 1e9

    e2e = None if args.no_e2e else time_e2e(dw, args.steps, max(3, args.warmup // 2), world, flush)
    e2e_s = max_over_ranks(sum(e2e["step_ms"]) * 1e-3, world) if e2e else None
    fill = time_fill(dw, 10, flush)
    wb = write_alg_bytes(w, fill["T"], False)
    wbu = write_alg_bytes(w, fill["T"], False, fill["rows"])
    write_gbs = wb / (fill["ms"] * 1e-3) / 1e9

    ceiling = stream_ceiling(alg, flush)
    layered = measure_layered(dw, 4, 10, flush, peak)
    others = {}
    if args.also:
        for name in [x for x in args.also.split(",") if x]:
            others[name] = measure_decode_only(name, 0, 20, flush, peak)

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, dw.num_splits, args.cpu_seconds)
        cpu_all = cpu_baseline_allcore(args.workload, w.B, dw.num_splits, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "batch": w.B, "num_splits": dw.num_splits,
                   "context_tokens": int(w.seq_lens.sum()),
                   "l2": "flushed before every timed step (512 MiB device write, then a 512 MiB read so the "
                         "write's dirty lines are written back before the step; both outside the step's events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "step_us": {"step": 1e3 * statistics.mean(r["step_ms"]),
                    "separated": {kernel_names(args.workload)[0]: 1e3 * statistics.mean(rk["write_ms"]),
                                  kernel_names(args.workload)[1]: 1e3 * dec_ms,
                                  "lse_merge": 1e3 * statistics.mean(rk["merge_ms"]),
                                  "step": 1e3 * statistics.mean(rk["step_ms"]),
                                  "note": "second K-step pass with an event between launches (no early "
                                          "start of decode/merge); the roofline uses its decode time"}},
        "decode_kv_read_gbs": achieved,
        "decode_hbm_frac": achieved / peak,
        "rope_kv_write_gbs": write_gbs,
        "rope_kv_write_hbm_frac": write_gbs / peak,
        "cache_fill": {"tokens": fill["T"], "us": fill["ms"] * 1e3, "bytes": wb,
                       "hbm_frac_table_rows_once": wbu / (fill["ms"] * 1e-3) / 1e9 / peak,
                       "note": "rope_kv_write_gbs counts one cos_sin row per token; hbm_frac_table_rows_once counts "
                               "each distinct position's row once"},
        "roofline": {"kernel": kernel_names(args.workload)[1], "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": ncu_traffic(args.workload, dw.num_splits),
                     "alg_bytes_per_launch": alg, "partial_record_bytes": partial_bytes(w, dw.num_splits),
                     "stream_read_same_bytes_gbs": ceiling,
                     "stream_read_same_bytes_frac": ceiling / peak,
                     "layered": layered},
        "e2e": None if e2e is None else {"value": world * w.B * args.steps / e2e_s, "unit": UNIT,
                                         "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "err_flag": err,
    }
    if others:
        line["other_workloads"] = others
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if cpu_all is not None:
        line["cpu_baseline_all_cores"] = cpu_all
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
