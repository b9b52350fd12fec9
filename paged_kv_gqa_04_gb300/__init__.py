"""Paged-KV GQA decode step for NVIDIA GB300 (sm_103a).

The three calls of one decode step -- fused RoPE + paged-KV write, paged
GQA split-K decode attention, LSE merge -- run in hand-written CUDA kernels
behind the C ABI of include/pkv.h (libpkv.so). This package is the thin
Python binding of that ABI (``_abi``), its build (``_build``) and the seeded
synthetic workload generator (``synth``). The library is loaded on first
use; without it every call raises.
"""
from ._abi import (EXPORTED, FLAG_DUPLICATE_SLOT, FLAG_PAGE_RANGE, FLAG_POSITION_RANGE, FLAG_SEQ_LEN_RANGE,
                   FLAG_SLOT_RANGE, FLAG_WAIT_TIMEOUT, PkvError, choose_num_splits, lib, lse_merge,
                   paged_gqa_decode, rope_kv_write, status_string, stream_read, validate_indices,
                   validate_indices_static)

__all__ = ["rope_kv_write", "paged_gqa_decode", "lse_merge", "choose_num_splits", "validate_indices",
           "validate_indices_static",
           "status_string", "stream_read", "PkvError", "lib", "EXPORTED", "FLAG_SLOT_RANGE", "FLAG_POSITION_RANGE",
           "FLAG_PAGE_RANGE", "FLAG_SEQ_LEN_RANGE", "FLAG_DUPLICATE_SLOT", "FLAG_WAIT_TIMEOUT"]
