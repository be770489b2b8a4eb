"""ctypes binding of the C ABI in include/attn_varlen.h.

Argument marshalling only: every step of the attention runs in the CUDA
library.  There is no fallback -- if the in-tree library cannot be built or
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

# Return codes (include/attn_varlen.h)
OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED_DIM = -2
ERR_MISALIGNED = -3
ERR_UNSUPPORTED_DEVICE = -4
ERR_CUDA = -5
ERR_OOM = -6
ERR_DEVICE_TIMEOUT = -7
ERR_WORKSPACE_SMALL = -8
ERR_DRIVER = -9
ERR_NOALLOC_LIMIT = -10
ERR_BAD_BLOCK_TABLE = -11
NOALLOC_MAX_SEQS = 1024

# Every symbol the header declares, with (restype, argtypes).
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SYMBOLS = {
    "attn_varlen_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "attn_varlen_workspace_size": (_SZ, [_I]),
    "attn_varlen_fwd_ws": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "attn_varlen_check": (_I, [_P]),
    "attn_varlen_check_ws": (_I, [_P, _P]),
    "attn_varlen_check_noalloc": (_I, [_P]),
    "attn_varlen_strerror": (ctypes.c_char_p, [_I]),
    "attn_varlen_version": (_I, []),
    "attn_varlen_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "attn_varlen_last_cuda_error": (ctypes.c_char_p, []),
    "attn_varlen_fwd_causal": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "attn_varlen_fwd_heads": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "paged_attn_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "chunk_delta_rule_output": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _P, _P]),
}

_LOCK = threading.Lock()
_LIB = None


class AttnVarlenError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {strerror(code)} (code {code})"
        if code == ERR_CUDA:
            msg += f": {load().attn_varlen_last_cuda_error().decode()}"
        super().__init__(msg)


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the in-tree CUDA library (building it first when absent)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.lib_path()
            if build_if_missing:
                path = _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in SYMBOLS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = lib
        return _LIB


def strerror(code: int) -> str:
    return load().attn_varlen_strerror(int(code)).decode()


def workspace_size(num_seqs: int) -> int:
    return int(load().attn_varlen_workspace_size(int(num_seqs)))


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream))


def _check_inputs(q, k, v, cu_q, cu_k, out):
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bfloat16")
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("q, k, v must be [total_tokens, num_heads, head_dim]; k and v alike")
    if q.shape[1:] != k.shape[1:]:
        raise ValueError("q and k must share num_heads and head_dim")
    for t in (q, k, v, out):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v and out must be contiguous CUDA tensors")
    if cu_q.dtype != torch.int32 or cu_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if cu_q.dim() != 1 or cu_q.shape != cu_k.shape or cu_q.numel() < 1:
        raise ValueError("cu_seqlens_q/k must be 1-D, equal length, >= 1 entry")
    if not cu_q.is_cuda or not cu_k.is_cuda or not cu_q.is_contiguous() or not cu_k.is_contiguous():
        raise ValueError("cu_seqlens must be contiguous CUDA tensors")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must have q's shape and dtype")


def attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, out=None, stream=None,
                    workspace=None, causal=False, heads=None):
    """softmax(q k^T / sqrt(head_dim)) v per packed sequence and head.

    q: bf16 [total_q, H, D]; k, v: bf16 [total_k, H, D]; cu_seqlens_q/k:
    int32 [num_seqs + 1] on the same device.  Returns ``out`` (allocated with
    ``torch.empty_like(q)`` when not given; rows outside every query slice are
    left untouched).  ``workspace``: optional uint8 CUDA tensor of at least
    ``workspace_size(num_seqs)`` bytes, zero-filled before first use.
    ``causal``: row r of a sequence sees keys j <= r + L_k - L_q
    (attn_varlen_fwd_causal; library-owned workspace only).  ``heads``: a
    ``(head_begin, head_count)`` pair to compute only those heads of the
    same tensors in place (attn_varlen_fwd_heads; library-owned workspace).
    """
    import torch
    if out is None:
        out = torch.empty_like(q)
    _check_inputs(q, k, v, cu_seqlens_q, cu_seqlens_k, out)
    lib = load()
    num_seqs = cu_seqlens_q.numel() - 1
    H, D = q.shape[1], q.shape[2]
    s = _stream_handle(stream, q.device)
    if (causal or heads is not None) and workspace is not None:
        raise ValueError("the causal and head-range entry points use the library-owned workspace")
    with torch.cuda.device(q.device):
        if heads is not None:
            rc = lib.attn_varlen_fwd_heads(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                           num_seqs, H, int(heads[0]), int(heads[1]), D,
                                           1 if causal else 0, out.data_ptr(), s)
        elif causal:
            rc = lib.attn_varlen_fwd_causal(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                            num_seqs, H, D, out.data_ptr(), s)
        elif workspace is None:
            rc = lib.attn_varlen_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                     num_seqs, H, D, out.data_ptr(), s)
        else:
            rc = lib.attn_varlen_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                        num_seqs, H, D, out.data_ptr(), workspace.data_ptr(),
                                        workspace.numel() * workspace.element_size(), s)
    if rc != OK:
        raise AttnVarlenError(rc, "attn_varlen_fwd")
    return out


def check(stream=None, device=None, workspace=None, noalloc=False) -> int:
    """Synchronise and return (and clear) the device status; raises on error.

    ``workspace``: the caller-owned workspace to read; ``noalloc``: read the
    status of attn_varlen_fwd_noalloc's fixed scratch instead."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    s = _stream_handle(stream, dev)
    with torch.cuda.device(dev):
        if noalloc:
            rc = load().attn_varlen_check_noalloc(s)
        elif workspace is None:
            rc = load().attn_varlen_check(s)
        else:
            rc = load().attn_varlen_check_ws(workspace.data_ptr(), s)
    if rc != OK:
        raise AttnVarlenError(rc, "attn_varlen_check")
    return rc


def attn_varlen_fwd_noalloc(q, k, v, cu_seqlens_q, cu_seqlens_k, out, stream=None):
    """attn_varlen_fwd through the entry point that allocates nothing.

    For callers that must not allocate device memory at call time; ``out``
    must be given.  Uses the library's fixed scratch (at most
    NOALLOC_MAX_SEQS sequences per call); calls on one device must not
    overlap on the GPU.
    """
    import torch
    _check_inputs(q, k, v, cu_seqlens_q, cu_seqlens_k, out)
    num_seqs = cu_seqlens_q.numel() - 1
    s = _stream_handle(stream, q.device)
    with torch.cuda.device(q.device):
        rc = load().attn_varlen_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                                            num_seqs, q.shape[1], q.shape[2], out.data_ptr(), s)
    if rc != OK:
        raise AttnVarlenError(rc, "attn_varlen_fwd_noalloc")
    return out


def paged_attn_decode(query, k_cache, v_cache, block_tables, seq_lens, out=None, stream=None):
    """One decode step over a paged KV cache (include/paged_attn_decode.h).

    query [num_seqs, Hq, D]; k_cache [num_blocks, Hkv, D/8, 16, 8]; v_cache
    [num_blocks, Hkv, D, 16], all bf16 or all fp16 CUDA tensors;
    block_tables int32 [num_seqs, max_blocks]; seq_lens int32 [num_seqs].
    Returns ``out`` (allocated like ``query`` when not given).
    """
    import torch
    if out is None:
        out = torch.empty_like(query)
    if query.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("query must be bf16 or fp16")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        if t.dtype != query.dtype or not t.is_contiguous() or t.device != query.device:
            raise ValueError(f"{name} must be a contiguous {query.dtype} tensor on {query.device}")
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_contiguous() or t.device != query.device:
            raise ValueError(f"{name} must be a contiguous int32 tensor on {query.device}")
    if query.dim() != 3 or k_cache.dim() != 5 or v_cache.dim() != 4 or block_tables.dim() != 2:
        raise ValueError("query [S, Hq, D], k_cache [B, Hkv, D/8, bs, 8], v_cache [B, Hkv, D, bs], "
                         "block_tables [S, max_blocks]")
    num_seqs, hq, d = query.shape
    num_blocks, hkv, _, bs = v_cache.shape
    lib = load()
    s = _stream_handle(stream, query.device)
    with torch.cuda.device(query.device):
        rc = lib.paged_attn_decode(query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   block_tables.data_ptr(), seq_lens.data_ptr(), num_seqs, hq,
                                   hkv, d, bs, block_tables.shape[1], num_blocks,
                                   1 if query.dtype == torch.float16 else 0, out.data_ptr(), s)
    if rc != OK:
        raise AttnVarlenError(rc, "paged_attn_decode")
    return out


def chunk_delta_rule_output(q, k, v, h, g, chunk_size=64, scale=None, out=None, stream=None):
    """Chunked gated delta-rule output (include/chunk_delta_rule.h).

    q, k bf16 [B, T, Hq, 128]; v bf16 [B, T, Hv, 128]; h bf16
    [B, ceil(T / 64), Hv, 128, 128]; g float32 [B, T, Hv]; all contiguous CUDA
    tensors on one device.  Returns ``out`` (bf16 [B, T, Hv, 128]).
    """
    import torch
    B, T, hq, kd = q.shape
    hv, vd = v.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, T, hv, vd), dtype=torch.bfloat16, device=q.device)
    for name, t in (("q", q), ("k", k), ("v", v), ("h", h), ("out", out)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor on {q.device}")
    if g.dtype != torch.float32 or not g.is_contiguous() or g.device != q.device:
        raise ValueError(f"g must be a contiguous float32 tensor on {q.device}")
    if k.shape != q.shape or v.shape[:2] != (B, T) or g.shape != (B, T, hv) \
            or h.shape != (B, (T + chunk_size - 1) // chunk_size, hv, kd, vd):
        raise ValueError("shapes do not match")
    lib = load()
    s = _stream_handle(stream, q.device)
    with torch.cuda.device(q.device):
        rc = lib.chunk_delta_rule_output(q.data_ptr(), k.data_ptr(), v.data_ptr(), h.data_ptr(),
                                         g.data_ptr(), B, T, hq, hv, kd, vd, int(chunk_size),
                                         float(scale or 0.0), out.data_ptr(), s)
    if rc != OK:
        raise AttnVarlenError(rc, "chunk_delta_rule_output")
    return out
