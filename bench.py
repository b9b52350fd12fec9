"""Benchmark of the paged-KV GQA decode step on GB300.

One step = the whole hot path over one batch: fused RoPE + paged-KV write of
the new token (q rotated in place), paged GQA split-K decode, LSE merge --
three launches of the library's kernels through the C ABI.

Default workload: the ragged large-batch decode, the largest single-GPU
configuration (batch 256, lognormal seq_lens with median 1024, sigma 1,
clipped to [1, 8192]; 32 query / 8 kv heads, head dim 128, page size 16, NHD,
bf16 cache, interleaved RoPE base 5e5, 1% of K rows scaled x8). The cache
holds every context token (written by the library's cache-write call before
timing). Every other configuration is measured the same way under
'other_workloads'.

Timing: W warm-up steps, then exactly K steps between a barrier and a device
synchronise on each side. Before every timed step the L2 is flushed (a 512 MiB
device write, then a 512 MiB read so that the write-back of dirty lines also
happens before the step) and q is restored from its unrotated copy, both
outside the step's CUDA events. Events on the launching stream bracket each
step (the launches chained as a program issues them); a second pass puts an
event between the launches for each kernel's own time. Reported:
  value       tokens/s = B*K / sum of step times (inputs resident in HBM)
  e2e         the same through the binding with host buffers: every step
              copies its inputs from pinned host memory to the device and its
              output (out, lse) back (pkv_copy), inside the step's events
  roofline    of the decode kernel: algorithmic bytes (Q + K/V pages + block-
              table entries + output) / its mean event time, against the
              measured HBM copy bandwidth
  cache_fill  GB/s of one cache-fill call over all context tokens, counting
              each distinct position's cos/sin row once
  cpu_baseline the float64 oracle on the host, single thread and on every
              core, over a sample of sequences at evenly spaced length
              quantiles of the batch
`--impl reference` times that oracle alone as the reference arm.
Under torchrun with N > 1 every rank runs an independent replica (weak
scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import gc
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
    p.add_argument("--workload", default="ragged", choices=sorted(WORKLOAD_TEXT))
    p.add_argument("--splits", type=int, default=0,
                   help="one split count for every sequence (0 = the library's split plan, or its heuristic "
                        "count with --split-mode uniform)")
    p.add_argument("--split-mode", default="plan", choices=["plan", "uniform"],
                   help="plan: a split count per sequence from pkv_plan_splits (pkv_plan_splits_mla for MLA); "
                        "uniform: one count for the batch from pkv_choose_num_splits (_mla)")
    p.add_argument("--also", default="qwen,longctx,fp8,fp4,million,mla,mla_batch",
                   help="other workloads measured the same way, reported under 'other_workloads' ('' = none)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=8.0,
                   help="seconds of oracle work per CPU-baseline leg of the headline workload")
    p.add_argument("--cpu-seconds-other", type=float, default=3.0,
                   help="seconds of oracle work per CPU-baseline leg of each other workload")
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


def kernel_source_hash(kind: str, name: str = "ragged") -> str:
    """First 16 hex digits of the SHA-256 of the source file that holds the
    workload's decode ("decode") or cache-write ("write") kernel."""
    if kind == "decode":
        f = "mla_decode.cu" if is_mla(name) else "paged_decode.cu"
    else:
        f = "rope_kv_write.cu"
    src = open(os.path.join(ROOT, "paged_kv_gqa_04_gb300", "csrc", f), "rb").read()
    return hashlib.sha256(src).hexdigest()[:16]


def decode_kernel_source_hash(name: str = "ragged") -> str:
    return kernel_source_hash("decode", name)


def _profile_fields(path: str) -> dict:
    out = {}
    try:
        txt = open(path).read()
    except OSError:
        return out
    for line in txt.splitlines():
        key, sep, val = line.partition(":")
        if sep and key and " " not in key.strip():
            out[key.strip()] = val.strip()
    return out


def ncu_traffic(workload: str, splits: dict):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if it was taken on the current kernel source with the same
    split configuration (mode and record count; for a plan, also its item
    count), else None."""
    f = _profile_fields(os.path.join(ROOT, "profiles", f"{kernel_names(workload)[1]}_{workload}.md"))
    try:
        h, t, s = f["kernel_source_sha256_16"], float(f["dram_bytes_per_launch"]), int(f["num_splits"])
        mode = f.get("split_mode", "uniform")
        items = int(f.get("plan_items", "0"))
    except (KeyError, ValueError):
        return None
    same = mode == splits["mode"] and s == splits["records"] and (mode != "plan" or items == splits["items"])
    return t if (h == decode_kernel_source_hash(workload) and same and t) else None


def ncu_fill_traffic(workload: str, tokens: int):
    """DRAM bytes of the cache-fill launch over `tokens` tokens from the
    committed ncu summary of this workload's fill, if it was taken on the
    current kernel source and the same token count (else None)."""
    f = _profile_fields(os.path.join(ROOT, "profiles", f"{kernel_names(workload)[0]}_fill_{workload}.md"))
    try:
        h, t, n = f["kernel_source_sha256_16"], float(f["dram_bytes_per_launch"]), int(f["tokens"])
    except (KeyError, ValueError):
        return None
    return t if (h == kernel_source_hash("write", workload) and n == tokens and t) else None


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            if k.strip() == "model name" and v.strip():
                return v.strip()
    except OSError:
        pass
    import platform
    return platform.machine() or "unknown"


def launch_mean(ms) -> tuple:
    """(mean, number left out) of event-timed launch durations, leaving out
    launches above twice the median: an event interval that long took in a
    stall of the host that enqueues the launches (the GPU waited for the
    next launch inside the interval), not kernel time."""
    med = statistics.median(ms)
    kept = [x for x in ms if x <= 2.0 * med]
    return statistics.mean(kept), len(ms) - len(kept)


def stats(ms) -> dict:
    """Mean, median, 10th / 90th percentile, min and max (microseconds) of a
    list of millisecond timings."""
    a = np.asarray(list(ms), dtype=np.float64) * 1e3
    return {"mean": float(a.mean()), "median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "min": float(a.min()), "max": float(a.max()), "n": int(a.size)}


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


def time_fill(dw, reps: int, flush, fi=None) -> dict:
    """One cache-fill call (all context tokens, no q), timed alone. `fi` is
    the fill call's device inputs (dw.fill_inputs()), made here if absent."""
    fi = dw.fill_inputs() if fi is None else fi
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
    return dict(T=T, rows=rows, ms=statistics.median(ms), ms_all=ms)


def fill_cache(dw) -> dict:
    """Write every context token into the cache with one cache-fill call and
    return that call's device inputs (kept for timing the fill)."""
    fi = dw.fill_inputs()
    if int(fi["positions"].numel()):
        dw.write_fill(fi)
    return fi


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
    # zeroed, so that records a split plan leaves unwritten compare equal
    outs = [(torch.zeros_like(dw.out_partial), torch.zeros_like(dw.lse_partial)) for _ in range(layers)]

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
    ok = all(torch.equal(op, outs[0][0]) and torch.equal(lp, outs[0][1]) for op, lp in outs[1:])
    del caches, outs
    return dict(layers=layers, us_per_layer=1e3 * ms / layers, gbs=gbs, frac=gbs / peak, layers_agree=ok)


def make_workload(name: str, splits: int, split_mode: str):
    """The device workload with its split configuration: an explicit count,
    else the library's split plan (pkv_plan_splits, or pkv_plan_splits_mla
    for an MLA workload) or, with split_mode "uniform", its heuristic count."""
    from paged_kv_gqa_04_gb300 import harness
    dw = harness.make_device_workload(name, num_splits=splits or None)
    if not splits and split_mode == "plan":
        dw.set_plan(uniform_if_equal=True)  # a plan with one count for every sequence runs as the uniform launch
    return dw


def split_desc(dw) -> dict:
    """The split configuration of a workload, for the JSON line."""
    if getattr(dw, "planned", False):
        sp, work = dw.plan_host
        pages = dw.w.pages_per_seq
        pps = -(-pages // np.maximum(sp, 1))
        # GQA: one CTA per (item, kv head); MLA: the items go to a persistent grid
        ctas = int(len(work)) * dw.w.Hkv if hasattr(dw.w, "Hkv") else None
        return {"mode": "plan", "records": dw.num_splits, "items": int(len(work)),
                "ctas": ctas, "splits_per_seq_min": int(sp.min()),
                "splits_per_seq_max": int(sp.max()), "max_pages_per_split": int(pps.max())}
    if getattr(dw, "uniform_from_plan", False):
        return {"mode": "uniform", "records": dw.num_splits, "from_plan": True}
    return {"mode": "uniform", "records": dw.num_splits}


def measure_workload(name: str, splits: int, reps: int, flush, peak: float, cpu_seconds: float,
                     with_e2e: bool = True, with_cpu: bool = True, split_mode: str = "plan") -> dict:
    """Every figure of one workload: the decode kernel alone (`reps` flushed
    launches), the chained and separated step, the step end to end with
    host buffers, the cache-fill call, decode layered over distinct caches,
    and the oracle on the host (single thread and all cores)."""
    dw = make_workload(name, splits, split_mode)
    w = dw.w
    fi = fill_cache(dw)
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
    dec = [a.elapsed_time(b) for a, b in ev]
    ms, dec_out = launch_mean(dec)
    rs = time_steps(dw, reps, 3, 1, flush, True)
    rc = time_steps(dw, reps, 3, 1, flush, False)
    names = kernel_names(name)
    step = dict(tokens_per_s=w.B * len(rc["step_ms"]) / (sum(rc["step_ms"]) * 1e-3),
                tokens_per_s_median_step=w.B / (statistics.median(rc["step_ms"]) * 1e-3),
                chained_us=stats(rc["step_ms"]),
                separated_us={names[0]: stats(rs["write_ms"]), names[1]: stats(rs["decode_ms"]),
                              names[2]: stats(rs["merge_ms"])})
    layered = measure_layered(dw, 4 if decode_alg_bytes(w) < 1e9 else 2, 5, flush, peak)
    fill = time_fill(dw, 5, flush, fi)
    del fi
    alg = decode_alg_bytes(w)
    r = dict(workload=WORKLOAD_TEXT[name], batch=w.B, context_tokens=int(w.seq_lens.sum()),
             num_splits=dw.num_splits, splits=split_desc(dw), decode_us=ms * 1e3, decode_us_stats=stats(dec),
             decode_launches_left_out=dec_out,
             decode_gbs=alg / (ms * 1e-3) / 1e9, decode_frac=alg / (ms * 1e-3) / 1e9 / peak,
             decode_traffic=ncu_traffic(name, split_desc(dw)), decode_alg_bytes=alg,
             stream_read_frac_same_bytes=stream_ceiling(alg, flush) / peak, layered=layered, step=step,
             cache_fill=fill_figures(w, fill, peak, name), err_flag=int(dw.err.item()))
    if with_e2e:
        e = time_e2e(dw, reps, 3, 1, flush)
        r["e2e"] = {"value": w.B * len(e["step_ms"]) / (sum(e["step_ms"]) * 1e-3), "unit": UNIT,
                    "step_us": stats(e["step_ms"]), "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
    del dw
    torch.cuda.empty_cache()
    if with_cpu:
        r["cpu_baseline"] = cpu_baseline(w, r["num_splits"], cpu_seconds, max_seqs=8)
        r["cpu_baseline_all_cores"] = cpu_baseline_allcore(name, w, r["num_splits"], cpu_seconds, max_seqs=8)
    return r


def fill_figures(w, fill: dict, peak: float, name: str) -> dict:
    """Figures of one cache-fill call. The headline fraction counts the
    cos/sin row of each distinct position once (tokens at the same position
    share the row, which is read from L2 after its first use); the
    one-row-per-token figure is kept beside it. `dram_bytes` is the fill
    launch's DRAM traffic from the committed ncu summary (null when that
    summary is of another kernel source or token count)."""
    wb = write_alg_bytes(w, fill["T"], False)
    wbu = write_alg_bytes(w, fill["T"], False, fill["rows"])
    s = fill["ms"] * 1e-3
    return {"tokens": fill["T"], "distinct_positions": fill["rows"], "us": fill["ms"] * 1e3,
            "us_stats": stats(fill["ms_all"]), "bytes": wbu, "gbs": wbu / s / 1e9, "hbm_frac": wbu / s / 1e9 / peak,
            "bytes_one_row_per_token": wb, "hbm_frac_one_row_per_token": wb / s / 1e9 / peak,
            "dram_bytes": ncu_fill_traffic(name, fill["T"])}


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


def quantile_sample(w, n: int) -> list:
    """n sequences of the batch at evenly spaced quantiles of its seq_len
    distribution (sorted by length, the middle of each of n equal groups),
    so the sample's mix of lengths is the batch's."""
    n = max(1, min(int(n), w.B))
    order = np.argsort(w.seq_lens, kind="stable")
    return sorted(int(order[min(w.B - 1, int((i + 0.5) * w.B / n))]) for i in range(n))


def seq_flops(w, b: int) -> float:
    """Oracle arithmetic of one sequence's decode: scores and weighted sum,
    two flops per product."""
    if hasattr(w, "Dc"):
        return 2.0 * float(w.seq_lens[b]) * w.H * (w.Dc + w.Dr + w.Dc)
    return 2.0 * float(w.seq_lens[b]) * w.Hq * 2 * w.D


def cpu_sample(w, max_seqs: int = 16, flop_budget: float = 2e9) -> list:
    """The largest quantile sample of at most max_seqs sequences whose
    oracle step stays within flop_budget (at least one sequence)."""
    best = quantile_sample(w, 1)
    for n in range(2, min(max_seqs, w.B) + 1):
        cand = quantile_sample(w, n)
        if sum(seq_flops(w, b) for b in cand) > flop_budget:
            break
        best = cand
    return best


def _sample_text(w, seqs) -> str:
    L = w.seq_lens.astype(np.float64)
    return (f"{len(seqs)} of {w.B} sequences at evenly spaced length quantiles (mean length "
            f"{L[seqs].mean():.0f} vs the batch's {L.mean():.0f})")


def cpu_baseline(w, num_splits, seconds: float, max_seqs: int = 16) -> dict:
    """The oracle on one host thread: whole steps (new-token write with q,
    decode, merge) over a quantile sample of the batch, repeated for about
    `seconds`; tokens/s = sequences decoded per second."""
    seqs = cpu_sample(w, max_seqs)
    run = oracle_step_timer(w, seqs, num_splits)
    total, n = 0.0, 0
    while total < seconds or n == 0:
        total += run()
        n += 1
    return {"value": len(seqs) * n / total, "unit": UNIT, "cores": 1, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{n} oracle decode steps over {_sample_text(w, seqs)}, {num_splits} splits: new-token "
                      f"cache write, decode, merge; float64, single thread; cache prepared untimed"}


_ALLCORE_BARRIER = None


def _allcore_init(barrier):
    global _ALLCORE_BARRIER
    _ALLCORE_BARRIER = barrier


def _allcore_worker(job):
    """One host process of the all-core oracle baseline: prepare the sample
    (untimed), wait for the others, then time whole steps over it."""
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


def cpu_baseline_allcore(name, w, num_splits, seconds: float, max_seqs: int = 16):
    """The oracle on every host core: one process per core (spawned: this
    process has initialised CUDA), each running whole steps over the same
    quantile sample as the single-thread baseline, all timed over the same
    window; throughput = the sum of the processes' (each keeps the batch's
    mix of lengths). Null for a single-sequence batch, which the oracle
    cannot spread over processes."""
    import multiprocessing as mp
    if w.B < 2:
        return None
    seqs = cpu_sample(w, max_seqs)
    procs = max(1, os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    with ctx.Pool(procs, initializer=_allcore_init, initargs=(barrier,)) as pool:
        rates = pool.map(_allcore_worker, [(name, seqs, num_splits, seconds)] * procs)
    return {"value": sum(rates), "unit": UNIT, "cores": procs, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{procs} processes, each running whole oracle decode steps (new-token write, decode, "
                      f"merge) over {_sample_text(w, seqs)}, {num_splits} splits, for about {seconds:g} s; "
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
    # size the per-step sample so that warm-up + timed steps take about a
    # minute, from the time per sequence of a probe at four length quantiles
    probe_seqs = quantile_sample(w, min(4, w.B))
    t1 = oracle_step_timer(w, probe_seqs, S)() / max(1, len(probe_seqs))
    n = int(max(1, min(w.B, round(60.0 / max(1, args.steps + args.warmup) / max(t1, 1e-6)))))
    seqs = quantile_sample(w, n)
    run = oracle_step_timer(w, seqs, S)
    for _ in range(args.warmup):
        run()
    ts = [run() for _ in range(args.steps)]
    total = sum(ts)
    value = len(seqs) * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.workload),
        "batch_sample": len(seqs), "num_splits": S,
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": 1, "cpu_model": cpu_model(),
                         "sample": f"each step: {_sample_text(w, seqs)} (new-token write, decode, merge)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, name: str) -> dict:
    """The line's `config`: the workload's description and sizes (the same
    in both arms)."""
    return {"workload": WORKLOAD_TEXT[name], "batch": w.B, "context_tokens": int(w.seq_lens.sum()),
            "l2": "GPU arm: flushed before every timed step (512 MiB device write, then a 512 MiB read so "
                  "the write's dirty lines are written back before the step; both outside the step's events)"}


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
    # no cyclic garbage collection pauses while launches are being enqueued
    gc.collect()
    gc.disable()
    peak, peak_kind = hbm_peak()
    dw = make_workload(args.workload, args.splits, args.split_mode)
    w = dw.w
    fi = fill_cache(dw)
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
    dec_ms, dec_out = launch_mean(rk["decode_ms"])
    alg = decode_alg_bytes(w)
    achieved = alg / (dec_ms * 1e-3) / 1e9

    e2e = None if args.no_e2e else time_e2e(dw, args.steps, max(3, args.warmup // 2), world, flush)
    e2e_s = max_over_ranks(sum(e2e["step_ms"]) * 1e-3, world) if e2e else None
    fill = fill_figures(w, time_fill(dw, 10, flush, fi), peak, args.workload)
    del fi

    ceiling = stream_ceiling(alg, flush)
    layered = measure_layered(dw, 4 if alg < 1e9 else 2, 10, flush, peak)
    num_splits = dw.num_splits
    splits = split_desc(dw)
    del dw
    torch.cuda.empty_cache()
    others = {}
    if args.also:
        for name in [x for x in args.also.split(",") if x and x != args.workload]:
            others[name] = measure_workload(name, 0, 20, flush, peak, args.cpu_seconds_other,
                                            with_e2e=not args.no_e2e,
                                            with_cpu=rank == 0 and not args.no_cpu_baseline,
                                            split_mode=args.split_mode)

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, num_splits, args.cpu_seconds)
        cpu_all = cpu_baseline_allcore(args.workload, w, num_splits, args.cpu_seconds)

    names = kernel_names(args.workload)
    cfg = workload_config(w, args.workload)
    cfg["parallelism"] = f"replicas x{world}" if world > 1 else "single GPU"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if getattr(w, "cache_dtype", "bf16") == "bf16"
        else w.cache_dtype, "data": "synthetic",
        "config": cfg,
        "num_splits": num_splits,
        "splits": splits,
        "step_us": {"chained": stats(r["step_ms"]),
                    "separated": {names[0]: stats(rk["write_ms"]), names[1]: stats(rk["decode_ms"]),
                                  names[2]: stats(rk["merge_ms"]), "step": stats(rk["step_ms"]),
                                  "note": "second K-step pass with an event between launches (no early "
                                          "start of decode/merge); the roofline uses its decode time"}},
        "decode_kv_read_gbs": achieved,
        "decode_hbm_frac": achieved / peak,
        "rope_kv_write_gbs": fill["gbs"],
        "rope_kv_write_hbm_frac": fill["hbm_frac"],
        "cache_fill": fill,
        "roofline": {"kernel": names[1], "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": ncu_traffic(args.workload, splits),
                     "alg_bytes_per_launch": alg, "partial_record_bytes": partial_bytes(w, num_splits),
                     "launch_us": dec_ms * 1e3, "launches_timed": len(rk["decode_ms"]),
                     "launches_left_out": dec_out,
                     "launch_us_basis": "mean of the separated pass's event-timed decode launches, leaving out "
                                        "launches above twice the median (host stalls inside the interval)",
                     "stream_read_same_bytes_gbs": ceiling,
                     "stream_read_same_bytes_frac": ceiling / peak,
                     "layered": layered},
        "e2e": None if e2e is None else {"value": world * w.B * args.steps / e2e_s, "unit": UNIT,
                                         "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                                         "step_us": stats(e2e["step_ms"])},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "err_flag": err,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if cpu_all is not None:
        line["cpu_baseline_all_cores"] = cpu_all
    if others:
        line["other_workloads"] = others
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
