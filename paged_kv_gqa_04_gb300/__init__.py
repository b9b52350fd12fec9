"""Paged-KV GQA decode step for NVIDIA GB300 (sm_103a).

The three calls of one decode step -- fused RoPE + paged-KV write, paged
GQA split-K decode attention, LSE merge -- their split-plan forms (a split
count per sequence), and their NVFP4-cache and MLA (latent cache) forms run
in hand-written CUDA kernels behind the C ABI of include/pkv.h (libpkv.so).
This package is the thin Python binding of that ABI (``_abi``), its build
(``_build``) and the seeded synthetic workload generator (``synth``). The
library is loaded on first use; without it every call raises.
"""
from ._abi import (EXPORTED, FLAG_DUPLICATE_SLOT, FLAG_PAGE_RANGE, FLAG_PLAN_RANGE, FLAG_POSITION_RANGE,
                   FLAG_SEQ_LEN_RANGE, FLAG_SLOT_RANGE, FLAG_WAIT_TIMEOUT, PkvError, choose_num_splits,
                   choose_num_splits_mla, copy, lib, lse_merge, lse_merge_planned, mla_cache_write, paged_gqa_decode,
                   paged_gqa_decode_nvfp4, paged_gqa_decode_planned, paged_mla_decode, paged_mla_decode_planned,
                   plan_splits, plan_splits_mla, rope_kv_write, rope_kv_write_nvfp4, selftest_bounded_wait,
                   status_string, stream_read, validate_indices, validate_indices_static)

__all__ = ["rope_kv_write", "paged_gqa_decode", "lse_merge", "choose_num_splits", "plan_splits",
           "paged_gqa_decode_planned", "lse_merge_planned", "validate_indices", "validate_indices_static",
           "rope_kv_write_nvfp4", "paged_gqa_decode_nvfp4", "mla_cache_write", "paged_mla_decode",
           "choose_num_splits_mla", "plan_splits_mla", "paged_mla_decode_planned", "selftest_bounded_wait", "copy",
           "status_string", "stream_read", "PkvError",
           "lib", "EXPORTED", "FLAG_SLOT_RANGE", "FLAG_POSITION_RANGE", "FLAG_PAGE_RANGE", "FLAG_SEQ_LEN_RANGE",
           "FLAG_DUPLICATE_SLOT", "FLAG_WAIT_TIMEOUT", "FLAG_PLAN_RANGE"]
