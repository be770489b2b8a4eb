"""CPU oracle for packed variable-length attention forward (fp64).

TEST INFRASTRUCTURE ONLY.  The product path never imports this package; only
the test suite, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA path: the arithmetic is in ``attn_oracle.c``
(plain C, IEEE double, libm ``exp``), built here with gcc and loaded with
ctypes.

What it computes: atrex-bench "attention_forward" (page #001, reference.py,
Model.forward) -- per non-empty query sequence and head,
``softmax(Q K^T / sqrt(head_dim)) V`` over that sequence's keys.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "paged_oracle.c"), os.path.join(_HERE, "chunk_o_oracle.c")]
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict = {}


def build(mutation: int = 0, out_dir: str | None = None) -> str:
    """Compile the oracle into a shared library and return its path.

    ``mutation`` > 0 builds a copy with one planted mistake (see the
    ``MUT(n)`` hooks in the C file); only the oracle's own pin tests use it.
    """
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "liboracle.so" if mutation == 0 else f"liboracle_mut{mutation}.so"
    path = os.path.join(out_dir, name)
    if (not os.path.exists(path)
            or os.path.getmtime(path) < max(os.path.getmtime(f) for f in _SRCS)):
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, *_SRCS, "-lm"]
        if mutation:
            cmd.insert(1, f"-DORACLE_MUTATION={int(mutation)}")
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def _lib(mutation: int = 0):
    with _LOCK:
        if mutation not in _LIBS:
            lib = ctypes.CDLL(build(mutation))
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_attn_varlen.argtypes = [p, p, p, p, p, i, i, i, i, p, i]
            lib.oracle_attn_varlen.restype = i
            lib.oracle_attn_rows.argtypes = [p, p, p, p, p, i, i, i, i, p,
                                             ctypes.c_int64, p, i]
            lib.oracle_attn_rows.restype = i
            lib.oracle_max_threads.argtypes = [i]
            lib.oracle_max_threads.restype = i
            lib.oracle_paged_decode.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, p]
            lib.oracle_paged_decode.restype = i
            lib.oracle_chunk_o.argtypes = [p, p, p, p, p, i, i, i, i, i, i, i, ctypes.c_double, p]
            lib.oracle_chunk_o.restype = i
            _LIBS[mutation] = lib
        return _LIBS[mutation]


def _prep(q, k, v, cu_q, cu_k):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
    cu_k = np.ascontiguousarray(cu_k, dtype=np.int32)
    if q.ndim != 3 or k.shape != v.shape or k.ndim != 3:
        raise ValueError("q, k, v must be [T, H, D] bf16 bit arrays")
    if q.shape[1:] != k.shape[1:]:
        raise ValueError("q and k/v must share H and D")
    if cu_q.shape != cu_k.shape or cu_q.ndim != 1 or cu_q.size < 1:
        raise ValueError("cu_seqlens_q/k must be 1-D of equal length >= 1")
    return q, k, v, cu_q, cu_k


def max_threads(nthreads: int = 0) -> int:
    """Threads the oracle's parallel loops use for a given request (0 = all)."""
    return int(_lib().oracle_max_threads(int(nthreads)))


def attn_varlen(q, k, v, cu_q, cu_k, nthreads: int = 0, mutation: int = 0,
                fill: float = np.nan, causal: bool = False) -> np.ndarray:
    """All output rows, float64 [total_q, H, D].

    ``q, k, v`` are bf16 bit patterns (uint16) of shape [T, H, D].  Rows that
    no non-empty query sequence covers keep ``fill``.  ``causal``: row r of a
    sequence sees keys j <= r + L_k - L_q (bottom-right aligned mask).
    """
    q, k, v, cu_q, cu_k = _prep(q, k, v, cu_q, cu_k)
    T, H, D = q.shape
    out = np.full((T, H, D), fill, dtype=np.float64)
    rc = _lib(mutation).oracle_attn_varlen(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, cu_q.ctypes.data,
        cu_k.ctypes.data, cu_q.size - 1, H, D, int(bool(causal)), out.ctypes.data,
        int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_varlen failed with {rc}")
    return out


def attn_rows(q, k, v, cu_q, cu_k, rows, nthreads: int = 0,
              mutation: int = 0, causal: bool = False) -> np.ndarray:
    """Selected output rows, float64 [n, D]; ``rows`` is int [n, 2] of (token, head)."""
    q, k, v, cu_q, cu_k = _prep(q, k, v, cu_q, cu_k)
    T, H, D = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 2)
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    rc = _lib(mutation).oracle_attn_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, cu_q.ctypes.data,
        cu_k.ctypes.data, cu_q.size - 1, H, D, int(bool(causal)), rows.ctypes.data,
        rows.shape[0], out.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed with {rc}")
    return out


def paged_decode(query, k_cache, v_cache, block_tables, seq_lens, dtype: str = "bf16",
                 mutation: int = 0) -> np.ndarray:
    """Paged single-query decode, float64 [num_seqs, Hq, D].

    ``query`` [num_seqs, Hq, D], ``k_cache`` [num_blocks, Hkv, D / 8,
    block_size, 8], ``v_cache`` [num_blocks, Hkv, D, block_size]: bit patterns
    (uint16) of ``dtype`` ("bf16" or "fp16"); ``block_tables`` int32
    [num_seqs, max_blocks]; ``seq_lens`` int32 [num_seqs].
    """
    query = np.ascontiguousarray(query, dtype=np.uint16)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n, hq, d = query.shape
    hkv, bs = v_cache.shape[1], v_cache.shape[3]
    if k_cache.shape != (v_cache.shape[0], hkv, d // 8, bs, 8) or v_cache.shape[2] != d:
        raise ValueError("cache shapes do not match the query")
    out = np.zeros((n, hq, d), dtype=np.float64)
    rc = _lib(mutation).oracle_paged_decode(
        query.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data, tables.ctypes.data,
        lens.ctypes.data, n, hq, hkv, d, bs, tables.shape[1] if tables.ndim == 2 else 0,
        1 if dtype == "fp16" else 0, out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_paged_decode failed with {rc}")
    return out


def chunk_o(q, k, v, h, g, chunk_size: int = 64, scale: float | None = None,
            mutation: int = 0) -> np.ndarray:
    """Chunked gated delta-rule output, float64 [B, T, H, V].

    ``q, k`` [B, T, Hq, K], ``v`` [B, T, H, V], ``h`` [B, NC, H, K, V]: bf16
    bit patterns (uint16); ``g`` float32 [B, T, H]; NC = ceil(T / chunk_size).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    g = np.ascontiguousarray(g, dtype=np.float32)
    B, T, Hq, K = q.shape
    H, V = v.shape[2], v.shape[3]
    nc = (T + chunk_size - 1) // chunk_size
    if k.shape != q.shape or v.shape[:2] != (B, T) or h.shape != (B, nc, H, K, V) \
            or g.shape != (B, T, H):
        raise ValueError("shapes do not match")
    out = np.zeros((B, T, H, V), dtype=np.float64)
    rc = _lib(mutation).oracle_chunk_o(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                       h.ctypes.data, g.ctypes.data, B, T, Hq, H, K, V,
                                       int(chunk_size), float(scale or 0.0), out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_chunk_o failed with {rc}")
    return out
