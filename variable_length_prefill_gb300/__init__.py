"""GB300-native packed variable-length attention forward (prefill).

The computation is atrex-bench "attention_forward" (page #001, reference.py,
Model.forward): per packed sequence and head, softmax(Q K^T / sqrt(D)) V,
non-causal (or, as an option, causal), bf16 in and out.  It runs in a
hand-written sm_103a CUDA library (TMA, tcgen05 MMA into TMEM,
warp-specialised online softmax) behind the C ABI in include/attn_varlen.h;
the same library holds the paged single-query decode of
include/paged_attn_decode.h and the chunked gated delta-rule output of
include/chunk_delta_rule.h.  This package is a thin ctypes binding.
"""
from ._binding import (AttnVarlenError, SYMBOLS, attn_varlen_fwd, attn_varlen_fwd_noalloc,
                       check, chunk_delta_rule_output, load, paged_attn_decode, strerror,
                       workspace_size)
from .build import build, lib_path
from .shard import head_shard

__all__ = ["AttnVarlenError", "SYMBOLS", "attn_varlen_fwd", "attn_varlen_fwd_noalloc", "build",
           "check", "chunk_delta_rule_output", "head_shard", "lib_path", "load",
           "paged_attn_decode", "strerror", "workspace_size"]
