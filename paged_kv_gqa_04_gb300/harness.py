"""Device-side setup and execution of a synthetic decode workload.

Allocates the paged caches and the step's buffers on the GPU, uploads the
seeded inputs from ``synth``, fills the cache with the context tokens through
the library's own cache-write call, and runs one decode step (cache write of
the new token, paged GQA decode, LSE merge) through the C ABI. Used by the
GPU tests, the smoke check and the benchmark; it computes nothing itself.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import _abi, synth


def make_device_workload(name: str, device: str = "cuda", num_splits: Optional[int] = None):
    """The device workload of a named GQA (synth.WORKLOADS) or MLA
    (synth.MLA_WORKLOADS) workload."""
    if name in synth.MLA_WORKLOADS:
        return MlaDeviceWorkload(synth.make_mla_workload(name), device, num_splits)
    return DeviceWorkload(synth.make_workload(name), device, num_splits)


def _u16_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceWorkload:
    """Caches, metadata and step buffers of one workload on one GPU."""

    # the step's per-token inputs a host-to-device step copies ("q" = q0)
    H2D_KEYS = ("q", "k", "v", "positions", "slot_mapping")

    def __init__(self, w: synth.Workload, device: str = "cuda", num_splits: Optional[int] = None):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.nvfp4 = w.cache_dtype == "nvfp4"
        cache_dtype = torch.bfloat16 if w.cache_dtype == "bf16" else torch.uint8
        self.k_cache = torch.zeros(w.cache_shape(), dtype=cache_dtype, device=dev)
        self.v_cache = torch.zeros(w.cache_shape(), dtype=cache_dtype, device=dev)
        # NVFP4 block scales (E4M3 bytes, one per 16 values)
        self.k_block_scale = torch.zeros(w.scale_shape(), dtype=torch.uint8, device=dev) if self.nvfp4 else None
        self.v_block_scale = torch.zeros(w.scale_shape(), dtype=torch.uint8, device=dev) if self.nvfp4 else None
        self.cos_sin = torch.from_numpy(w.cos_sin()).to(dev)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.k_scale = None if w.k_scale is None else torch.from_numpy(w.k_scale).to(dev)
        self.v_scale = None if w.v_scale is None else torch.from_numpy(w.v_scale).to(dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        if num_splits is None:
            props = torch.cuda.get_device_properties(dev)
            num_splits = _abi.choose_num_splits(w.B, w.Hkv, w.Hq, w.D, int(w.pages_per_seq.sum()),
                                                max(1, int(w.pages_per_seq.max()) if w.B else 1), w.cache_dtype,
                                                props.multi_processor_count)
        self.splits_per_seq = None  # a split plan (set_plan), else one split count for the batch
        self.work = None
        self.set_splits(num_splits)
        self.out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        self.decode_inputs = None

    def set_splits(self, num_splits: int) -> None:
        """One split count for every sequence (drops any split plan)."""
        w = self.w
        self.splits_per_seq = self.work = None
        self.uniform_from_plan = False
        self.num_splits = int(num_splits)
        self.out_partial = torch.empty((w.B, self.num_splits, w.Hq, w.D), dtype=torch.float32, device=self.device)
        self.lse_partial = torch.empty((w.B, self.num_splits, w.Hq), dtype=torch.float32, device=self.device)

    def set_plan(self, target_pages: int = 0, max_splits: int = 4095, uniform_if_equal: bool = False) -> None:
        """A split count per sequence from the library's planner (host
        seq_lens), uploaded with its work list; the partials get the plan's
        record count. With uniform_if_equal, a plan that gives every
        sequence the same count runs as the uniform launch with that count
        (the same records, without the work list's extra read)."""
        w = self.w
        props = torch.cuda.get_device_properties(self.device)
        sp, nrec, work = _abi.plan_splits(w.seq_lens, w.Hkv, w.Hq, w.D, max(1, w.max_pages), w.cache_dtype,
                                          props.multi_processor_count, max_splits, target_pages)
        self.set_splits(nrec)
        if uniform_if_equal and w.B and bool((sp == nrec).all()):
            self.uniform_from_plan = True
            return
        self.plan_host = (sp, work)
        self.splits_per_seq = torch.from_numpy(sp).to(self.device)
        self.work = torch.from_numpy(np.ascontiguousarray(work)).to(self.device)

    @property
    def planned(self) -> bool:
        return self.work is not None

    # ---- cache fill ----------------------------------------------------------
    def fill(self, max_tokens: int = 1 << 18) -> int:
        """Write context tokens 0..L-2 of every sequence with the library's
        cache-write call (no q), in chunks of whole sequences. Returns the
        number of tokens written."""
        w = self.w
        written = 0
        b = 0
        while b < w.B:
            seqs = []
            n = 0
            while b < w.B and (not seqs or n + max(0, int(w.seq_lens[b]) - 1) <= max_tokens):
                seqs.append(b)
                n += max(0, int(w.seq_lens[b]) - 1)
                b += 1
            fb = w.fill_batch(seqs)
            if len(fb["positions"]) == 0:
                continue
            k = _u16_to_bf16(fb["k"], self.device)
            v = _u16_to_bf16(fb["v"], self.device)
            pos = torch.from_numpy(fb["positions"]).to(self.device)
            slot = torch.from_numpy(fb["slot_mapping"]).to(self.device)
            self.write(None, k, v, pos, slot)
            written += len(fb["positions"])
        return written

    def fill_inputs(self, seqs=None):
        """Device tensors of one fill call (for timing the cache write)."""
        fb = self.w.fill_batch(seqs)
        return dict(k=_u16_to_bf16(fb["k"], self.device), v=_u16_to_bf16(fb["v"], self.device),
                    positions=torch.from_numpy(fb["positions"]).to(self.device),
                    slot_mapping=torch.from_numpy(fb["slot_mapping"]).to(self.device))

    # ---- the three calls -------------------------------------------------------
    def write(self, q, k, v, positions, slot_mapping, stream=None) -> None:
        w = self.w
        if self.nvfp4:
            _abi.rope_kv_write_nvfp4(q, k, v, positions, self.cos_sin, self.k_cache, self.v_cache,
                                     self.k_block_scale, self.v_block_scale, slot_mapping, self.k_scale,
                                     self.v_scale, w.layout, w.style, self.err, stream)
            return
        _abi.rope_kv_write(q, k, v, positions, self.cos_sin, self.k_cache, self.v_cache, slot_mapping,
                           self.k_scale, self.v_scale, w.layout, w.style, self.err, stream)

    def caches(self) -> tuple:
        """The cache tensors: (k, v), plus the block scales for NVFP4."""
        if self.nvfp4:
            return self.k_cache, self.v_cache, self.k_block_scale, self.v_block_scale
        return self.k_cache, self.v_cache

    def decode(self, q, stream=None) -> None:
        self.decode_into(q, self.caches(), self.out_partial, self.lse_partial, stream)

    def decode_into(self, q, caches: tuple, out_partial, lse_partial, stream=None) -> None:
        """The decode over the given caches (as returned by caches(), or
        copies of them) into the given partial buffers."""
        w = self.w
        if self.planned:
            kbs, vbs = (caches[2], caches[3]) if self.nvfp4 else (None, None)
            _abi.paged_gqa_decode_planned(q, caches[0], caches[1], self.block_tables, self.seq_lens,
                                          w.softmax_scale, self.splits_per_seq, self.work, out_partial, lse_partial,
                                          self.k_scale, self.v_scale, w.layout, self.err, stream,
                                          k_block_scale=kbs, v_block_scale=vbs)
            return
        if self.nvfp4:
            kc, vc, kbs, vbs = caches
            _abi.paged_gqa_decode_nvfp4(q, kc, vc, kbs, vbs, self.block_tables, self.seq_lens, w.softmax_scale,
                                        self.num_splits, out_partial, lse_partial, self.k_scale, self.v_scale,
                                        w.layout, self.err, stream)
            return
        kc, vc = caches
        _abi.paged_gqa_decode(q, kc, vc, self.block_tables, self.seq_lens, w.softmax_scale, self.num_splits,
                              out_partial, lse_partial, self.k_scale, self.v_scale, w.layout, self.err, stream)

    def merge(self, stream=None) -> None:
        if self.planned:
            _abi.lse_merge_planned(self.out_partial, self.lse_partial, self.splits_per_seq, self.out, self.lse,
                                   stream)
            return
        _abi.lse_merge(self.out_partial, self.lse_partial, self.out, self.lse, stream)

    def upload_decode(self) -> dict:
        """Device copies of the new token's q, k, v, position and slot. q0 is
        kept unrotated; `q` is the working copy the step rotates in place."""
        db = self.w.decode_batch()
        d = dict(q0=_u16_to_bf16(db["q"], self.device), k=_u16_to_bf16(db["k"], self.device),
                 v=_u16_to_bf16(db["v"], self.device), positions=torch.from_numpy(db["positions"]).to(self.device),
                 slot_mapping=torch.from_numpy(db["slot_mapping"]).to(self.device))
        d["q"] = d["q0"].clone()
        self.decode_inputs = d
        return d

    def write_step(self, stream=None) -> None:
        """The step's cache write: the new token of every sequence, with q."""
        d = self.decode_inputs
        self.write(d["q"], d["k"], d["v"], d["positions"], d["slot_mapping"], stream)

    def write_fill(self, fi: dict, stream=None) -> None:
        """A cache-fill call (no q) on inputs from fill_inputs()."""
        self.write(None, fi["k"], fi["v"], fi["positions"], fi["slot_mapping"], stream)

    def step(self, stream=None) -> None:
        """One decode step on the current inputs: cache write of the new
        token (q rotated in place), decode, merge."""
        self.write_step(stream)
        self.decode(self.decode_inputs["q"], stream)
        self.merge(stream)

    # ---- host views -------------------------------------------------------------
    def cache_pages_u(self, cache: torch.Tensor, pages) -> np.ndarray:
        """Raw bytes (uint16 for bf16, uint8 for fp8 / nvfp4) of the given pages."""
        idx = torch.as_tensor(np.asarray(pages, np.int64), device=self.device)
        sel = cache.index_select(0, idx).cpu()
        if sel.dtype == torch.bfloat16:
            return sel.view(torch.int16).numpy().view(np.uint16)
        return sel.numpy()

    @staticmethod
    def bf16_u16(t: torch.Tensor) -> np.ndarray:
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class StepGraph:
    """One decode step captured as a CUDA graph: one submission per step.

    The graph holds the three C-ABI launches (the cache write; the decode and
    the merge as programmatic dependents, so each starts its prologue while
    its predecessor finishes). With ``host_io`` the step's inputs -- the
    workload's H2D_KEYS (q, k, v, positions, slot_mapping, or the MLA step's
    q_pe, q_lat, ckv, kpe, positions, slot_mapping), then block_tables and
    seq_lens -- live in one packed device buffer (each tensor a 256-byte
    aligned view the kernels read directly) filled by ONE copy from a pinned
    host buffer of the same layout, and out and lse live in one packed device
    buffer read back by ONE copy to pinned host memory. Both copies are
    pkv_copy launches (the SMs move the bytes over the host link; the
    result's copy starts behind the merge as its programmatic dependent).
    Without host_io the
    graph starts by restoring the unrotated q (MLA: q_pe) on the device.
    """

    def __init__(self, dw, host_io: bool = False):
        self.dw = dw
        self.host_io = host_io
        if host_io:
            self._pack()
        self._body()  # run once outside the capture (first-call set-up)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()
        torch.cuda.synchronize()

    @staticmethod
    def _layout(tensors: dict) -> tuple:
        offs, off = {}, 0
        for k, t in tensors.items():
            offs[k] = off
            off = (off + t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    @staticmethod
    def _views(buf: torch.Tensor, tensors: dict, offs: dict) -> dict:
        return {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for k, t in tensors.items()}

    def _pack(self) -> None:
        dw, d = self.dw, self.dw.decode_inputs
        ins = {k: (d["q0"] if k == "q" else d[k]) for k in dw.H2D_KEYS}
        ins["block_tables"] = dw.block_tables
        ins["seq_lens"] = dw.seq_lens
        if getattr(dw, "planned", False):  # a split plan is made per step on the host and travels with the inputs
            ins["splits_per_seq"] = dw.splits_per_seq
            ins["work"] = dw.work
        offs, size = self._layout(ins)
        self.dev_in = torch.zeros(size, dtype=torch.uint8, device=dw.device)
        self.host_in = torch.zeros(size, dtype=torch.uint8).pin_memory()
        hv = self._views(self.host_in, ins, offs)
        for k, t in ins.items():
            hv[k].copy_(t.cpu())
        dv = self._views(self.dev_in, ins, offs)
        for k in dw.H2D_KEYS:  # the step now reads its inputs from the packed buffer
            d[k] = dv[k]
        dw.block_tables = dv["block_tables"]
        dw.seq_lens = dv["seq_lens"]
        if getattr(dw, "planned", False):
            dw.splits_per_seq = dv["splits_per_seq"]
            dw.work = dv["work"]
        outs = {"out": dw.out, "lse": dw.lse}
        offs, size = self._layout(outs)
        self.dev_out = torch.zeros(size, dtype=torch.uint8, device=dw.device)
        self.host_out = torch.zeros(size, dtype=torch.uint8).pin_memory()
        ov = self._views(self.dev_out, outs, offs)
        dw.out, dw.lse = ov["out"], ov["lse"]
        hv = self._views(self.host_out, outs, offs)
        self.out_h, self.lse_h = hv["out"], hv["lse"]

    def _body(self) -> None:
        dw, d = self.dw, self.dw.decode_inputs
        if not self.host_io:
            d["q"].copy_(d["q0"])
        else:
            _abi.copy(self.dev_in, self.host_in)  # pinned host -> device, by the SMs
        dw.step()
        if self.host_io:
            _abi.copy(self.host_out, self.dev_out)  # device -> pinned host, behind the merge

    @property
    def h2d_bytes(self) -> int:
        return self.host_in.numel() if self.host_io else 0

    @property
    def d2h_bytes(self) -> int:
        return self.host_out.numel() if self.host_io else 0

    def replay(self) -> None:
        self.graph.replay()


class MlaDeviceWorkload:
    """Latent caches, metadata and step buffers of one MLA workload on one
    GPU: the MLA cache write, the paged MLA decode and the D = 512 merge,
    through the C ABI. decode_inputs["q"] is the working copy of q_pe (rotated
    in place by the write), "q0" the unrotated one."""

    H2D_KEYS = ("q", "q_lat", "ckv", "kpe", "positions", "slot_mapping")
    nvfp4 = False

    def __init__(self, w: synth.MlaWorkload, device: str = "cuda", num_splits: Optional[int] = None):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.ckv_cache = torch.zeros((w.num_pages, w.page_size, w.Dc), dtype=torch.uint8, device=dev)
        self.kpe_cache = torch.zeros((w.num_pages, w.page_size, w.Dr), dtype=torch.bfloat16, device=dev)
        self.cos_sin = torch.from_numpy(w.cos_sin()).to(dev)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.ckv_scale = torch.tensor([w.ckv_scale], dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.splits_per_seq = self.work = None
        if num_splits is None:
            props = torch.cuda.get_device_properties(dev)
            num_splits = _abi.choose_num_splits_mla(w.B, w.H, int(w.pages_per_seq.sum()),
                                                    max(1, int(w.pages_per_seq.max()) if w.B else 1),
                                                    props.multi_processor_count)
        self.set_splits(num_splits)
        self.out = torch.empty((w.B, w.H, w.Dc), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
        self.decode_inputs = None

    def set_splits(self, num_splits: int) -> None:
        """One split count for every sequence (drops any split plan)."""
        w = self.w
        self.splits_per_seq = self.work = None
        self.uniform_from_plan = False
        self.num_splits = int(num_splits)
        self.out_partial = torch.empty((w.B, self.num_splits, w.H, w.Dc), dtype=torch.float32, device=self.device)
        self.lse_partial = torch.empty((w.B, self.num_splits, w.H), dtype=torch.float32, device=self.device)

    def set_plan(self, target_pages: int = 0, max_splits: int = 4095, uniform_if_equal: bool = False) -> None:
        """A split count per sequence from the library's MLA planner (host
        seq_lens), uploaded with its work list (uniform_if_equal: as
        DeviceWorkload.set_plan)."""
        w = self.w
        props = torch.cuda.get_device_properties(self.device)
        sp, nrec, work = _abi.plan_splits_mla(w.seq_lens, w.H, max(1, int(w.block_tables.shape[1])),
                                              props.multi_processor_count, max_splits, target_pages)
        self.set_splits(nrec)
        if uniform_if_equal and w.B and bool((sp == nrec).all()):
            self.uniform_from_plan = True
            return
        self.plan_host = (sp, work)
        self.splits_per_seq = torch.from_numpy(sp).to(self.device)
        self.work = torch.from_numpy(np.ascontiguousarray(work)).to(self.device)

    @property
    def planned(self) -> bool:
        return self.work is not None

    def fill(self, max_tokens: int = 1 << 18) -> int:
        """Context tokens 0..L-2 of every sequence through the library's MLA
        cache write (no q_pe), in chunks of whole sequences."""
        w = self.w
        written = 0
        b = 0
        while b < w.B:
            seqs = []
            n = 0
            while b < w.B and (not seqs or n + max(0, int(w.seq_lens[b]) - 1) <= max_tokens):
                seqs.append(b)
                n += max(0, int(w.seq_lens[b]) - 1)
                b += 1
            fb = w.fill_batch(seqs)
            if len(fb["positions"]) == 0:
                continue
            self.write(None, _u16_to_bf16(fb["ckv"], self.device), _u16_to_bf16(fb["kpe"], self.device),
                       torch.from_numpy(fb["positions"]).to(self.device),
                       torch.from_numpy(fb["slot_mapping"]).to(self.device))
            written += len(fb["positions"])
        return written

    def fill_inputs(self, seqs=None):
        fb = self.w.fill_batch(seqs)
        return dict(ckv=_u16_to_bf16(fb["ckv"], self.device), kpe=_u16_to_bf16(fb["kpe"], self.device),
                    positions=torch.from_numpy(fb["positions"]).to(self.device),
                    slot_mapping=torch.from_numpy(fb["slot_mapping"]).to(self.device))

    def caches(self) -> tuple:
        return self.ckv_cache, self.kpe_cache

    def write(self, q_pe, ckv, kpe, positions, slot_mapping, stream=None) -> None:
        _abi.mla_cache_write(q_pe, ckv, kpe, positions, self.cos_sin, self.ckv_cache, self.kpe_cache, slot_mapping,
                             self.ckv_scale, self.w.style, self.err, stream)

    def decode(self, q_pe, stream=None) -> None:
        self.decode_into(q_pe, self.caches(), self.out_partial, self.lse_partial, stream)

    def decode_into(self, q_pe, caches: tuple, out_partial, lse_partial, stream=None) -> None:
        w = self.w
        if self.planned:
            _abi.paged_mla_decode_planned(self.decode_inputs["q_lat"], q_pe, caches[0], caches[1], self.block_tables,
                                          self.seq_lens, w.softmax_scale, self.splits_per_seq, self.work,
                                          out_partial, lse_partial, self.ckv_scale, self.err, stream)
            return
        _abi.paged_mla_decode(self.decode_inputs["q_lat"], q_pe, caches[0], caches[1], self.block_tables,
                              self.seq_lens, w.softmax_scale, self.num_splits, out_partial, lse_partial,
                              self.ckv_scale, self.err, stream)

    def merge(self, stream=None) -> None:
        if self.planned:
            _abi.lse_merge_planned(self.out_partial, self.lse_partial, self.splits_per_seq, self.out, self.lse,
                                   stream)
            return
        _abi.lse_merge(self.out_partial, self.lse_partial, self.out, self.lse, stream)

    def upload_decode(self) -> dict:
        db = self.w.decode_batch()
        dev = self.device
        d = dict(q0=_u16_to_bf16(db["q_pe"], dev), q_lat=_u16_to_bf16(db["q_lat"], dev),
                 ckv=_u16_to_bf16(db["ckv"], dev), kpe=_u16_to_bf16(db["kpe"], dev),
                 positions=torch.from_numpy(db["positions"]).to(dev),
                 slot_mapping=torch.from_numpy(db["slot_mapping"]).to(dev))
        d["q"] = d["q0"].clone()
        self.decode_inputs = d
        return d

    def write_step(self, stream=None) -> None:
        d = self.decode_inputs
        self.write(d["q"], d["ckv"], d["kpe"], d["positions"], d["slot_mapping"], stream)

    def write_fill(self, fi: dict, stream=None) -> None:
        self.write(None, fi["ckv"], fi["kpe"], fi["positions"], fi["slot_mapping"], stream)

    def step(self, stream=None) -> None:
        """One MLA decode step: cache write of the new token (q_pe rotated in
        place), decode, merge."""
        self.write_step(stream)
        self.decode(self.decode_inputs["q"], stream)
        self.merge(stream)

    cache_pages_u = DeviceWorkload.cache_pages_u
    bf16_u16 = staticmethod(DeviceWorkload.bf16_u16)
