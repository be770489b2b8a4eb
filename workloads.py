"""Seeded synthetic inputs for packed variable-length attention.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds no attention arithmetic: it only draws random
numbers, rounds them to the bf16 input type and builds the ``cu_seqlens``
prefix sums.

What it follows (atrex-bench "attention_forward", page #001, ``input.py``):
q, k and v are drawn i.i.d. N(0, 1) in bf16 with shape
``[total_tokens, num_heads, head_dim]`` and ``cu_seqlens_q = cu_seqlens_k`` is
the prefix sum of the per-sequence lengths.  The page draws unseeded on the
GPU; here every draw is seeded on the host so both sides see identical bits:
``numpy.random.default_rng(seed).standard_normal(..., dtype=float32)`` in the
order q, k, v, each rounded to bf16 by round-to-nearest-even on the bit
pattern.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One attention call: sequence lengths, heads and head size."""

    name: str
    seq_lens_q: tuple
    num_heads: int
    head_dim: int
    seed: int
    seq_lens_k: tuple | None = None   # None: same as seq_lens_q
    cu_offset: int = 0                # rows before the first sequence
    description: str = ""

    @property
    def lens_k(self) -> tuple:
        return self.seq_lens_q if self.seq_lens_k is None else self.seq_lens_k

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_q)

    def cu_seqlens(self):
        """int32 prefix sums (q, k), each of length num_seqs + 1."""
        cu_q = np.zeros(self.num_seqs + 1, dtype=np.int64)
        cu_k = np.zeros(self.num_seqs + 1, dtype=np.int64)
        cu_q[0] = cu_k[0] = self.cu_offset
        cu_q[1:] = self.cu_offset + np.cumsum(self.seq_lens_q)
        cu_k[1:] = self.cu_offset + np.cumsum(self.lens_k)
        return cu_q.astype(np.int32), cu_k.astype(np.int32)

    @property
    def total_q(self) -> int:
        return int(self.cu_offset + sum(self.seq_lens_q))

    @property
    def total_k(self) -> int:
        return int(self.cu_offset + sum(self.lens_k))

    def flops(self) -> float:
        """The metric's FLOP count 4 * sum(L_q * L_k) * H * D (true head_dim)."""
        s = sum(int(a) * int(b) for a, b in zip(self.seq_lens_q, self.lens_k)
                if a > 0 and b > 0)
        return 4.0 * s * self.num_heads * self.head_dim

    def algorithmic_bytes(self) -> int:
        """bf16 bytes of q, k, v read once and out written once."""
        rows_q = sum(max(int(a), 0) for a in self.seq_lens_q)
        rows_k = sum(max(int(b), 0) for a, b in zip(self.seq_lens_q, self.lens_k)
                     if a > 0)
        row = self.num_heads * self.head_dim * 2
        return (2 * rows_q + 2 * rows_k) * row


# The five workloads: four rows of the page's shape table (#4, #8, #9, #11)
# and one packed batch made of rows #11-#17 plus a length-1 and an empty
# sequence.
C1 = Workload("C1_L276_H4_D72", (276,), 4, 72, seed=1,
              description="one sequence L=276, H=4, D=72 (shape-table row #11)")
C2 = Workload("C2_L8136_H16_D72", (8136,), 16, 72, seed=2,
              description="one sequence L=8136, H=16, D=72 (shape-table row #4)")
C3 = Workload("C3_L16742_H32_D128", (16742,), 32, 128, seed=3,
              description="one sequence L=16742, H=32, D=128 (shape-table row #9)")
C4 = Workload("C4_L65556_H16_D72", (65556,), 16, 72, seed=4,
              description="one sequence L=65556, H=16, D=72 (shape-table row #8)")
C5 = Workload("C5_packed9_T31673_H4_D72",
              (1, 276, 600, 1012, 2024, 4100, 8184, 15476, 0), 4, 72, seed=5,
              description="packed batch of 9 sequences (rows #11-#17, a length-1 "
                          "and an empty one), T=31673, H=4, D=72")

CONFIGS = {"C1": C1, "C2": C2, "C3": C3, "C4": C4, "C5": C5}

# head_dim 256 (beyond the page's table, which stops at 128): one long
# sequence, timed beside the five workloads and profiled on its own.
D256 = Workload("D256_L16384_H16", (16384,), 16, 256, seed=6,
                description="one sequence L=16384, H=16, D=256 (head_dim 256)")
EXTRA_CONFIGS = {"D256": D256}


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def make_inputs(w: Workload):
    """Return dict with q, k, v (uint16 bf16 bits, [T, H, D]) and cu_q, cu_k (int32)."""
    rng = np.random.default_rng(w.seed)
    H, D = w.num_heads, w.head_dim
    q = round_to_bf16_bits(rng.standard_normal((w.total_q, H, D), dtype=np.float32))
    k = round_to_bf16_bits(rng.standard_normal((w.total_k, H, D), dtype=np.float32))
    v = round_to_bf16_bits(rng.standard_normal((w.total_k, H, D), dtype=np.float32))
    cu_q, cu_k = w.cu_seqlens()
    return {"q": q, "k": k, "v": v, "cu_q": cu_q, "cu_k": cu_k}


def sample_rows(w: Workload, rows_per_head: int, seed_offset: int = 1000):
    """Seeded subset of (token, head) output rows, drawn independently per head.

    Only tokens that belong to a non-empty query sequence are drawn.  Returns
    an int64 array of shape [n, 2] with columns (token index, head).
    """
    rng = np.random.default_rng(w.seed + seed_offset)
    cu_q, _ = w.cu_seqlens()
    covered = []
    for i in range(w.num_seqs):
        if cu_q[i + 1] > cu_q[i]:
            covered.append(np.arange(cu_q[i], cu_q[i + 1]))
    tokens = np.concatenate(covered) if covered else np.zeros(0, dtype=np.int64)
    out = []
    for h in range(w.num_heads):
        n = min(rows_per_head, tokens.size)
        pick = np.sort(rng.choice(tokens.size, size=n, replace=False))
        out.append(np.stack([tokens[pick], np.full(n, h)], axis=1))
    return np.concatenate(out).astype(np.int64)


# ----------------------------------------------------------- paged decode
# atrex-bench "paged_attention_decode" (page #024, input.py _make_inputs):
# query [num_seqs, Hq, D]; k_cache [num_blocks, Hkv, D / x, block_size, x]
# with x = 16 bytes / element size; v_cache [num_blocks, Hkv, D, block_size];
# block_tables int32 [num_seqs, max_blocks] mapping sequence i's block j to
# physical block i * max_blocks + j; seq_lens = ctx_len for every sequence;
# num_blocks = max_blocks * num_seqs + 16.  Draws are seeded here, in the
# order query, k_cache, v_cache (the page draws unseeded on the GPU).


@dataclass(frozen=True)
class PagedWorkload:
    """One paged-decode call: the page's shape-table parameters."""

    name: str
    num_seqs: int
    ctx_len: int
    num_query_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int = 16
    dtype: str = "bf16"          # "bf16" or "fp16"
    seed: int = 0
    seq_lens: tuple | None = None  # None: ctx_len for every sequence
    shuffle_blocks: bool = False   # permute the physical block ids

    @property
    def max_blocks(self) -> int:
        return (self.ctx_len + self.block_size - 1) // self.block_size

    @property
    def num_blocks(self) -> int:
        return self.max_blocks * self.num_seqs + 16

    @property
    def x(self) -> int:
        return 8  # 16 bytes of a 2-byte type

    def lens(self) -> np.ndarray:
        if self.seq_lens is None:
            return np.full(self.num_seqs, self.ctx_len, dtype=np.int32)
        return np.asarray(self.seq_lens, dtype=np.int32)

    def flops(self) -> float:
        """4 * D per (query head, context token): scores plus weighted sum."""
        return 4.0 * float(np.clip(self.lens(), 0, None).sum()) * self.num_query_heads * self.head_size

    def algorithmic_bytes(self) -> int:
        """K and V of every context token and KV head, query and output once."""
        toks = int(np.clip(self.lens(), 0, None).sum())
        kv = toks * self.num_kv_heads * self.head_size * 2 * 2
        qo = self.num_seqs * self.num_query_heads * self.head_size * 2 * 2
        return kv + qo + self.num_seqs * (self.max_blocks + 1) * 4


def round_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> IEEE half bit patterns (uint16), round to nearest even."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def make_paged_inputs(w: PagedWorkload):
    """Dict of query, k_cache, v_cache (uint16 bits of w.dtype), block_tables,
    seq_lens (int32)."""
    rng = np.random.default_rng(w.seed)
    rnd = round_to_bf16_bits if w.dtype == "bf16" else round_to_f16_bits
    D, bs = w.head_size, w.block_size
    query = rnd(rng.standard_normal((w.num_seqs, w.num_query_heads, D), dtype=np.float32))
    k_cache = rnd(rng.standard_normal((w.num_blocks, w.num_kv_heads, D // w.x, bs, w.x),
                                      dtype=np.float32))
    v_cache = rnd(rng.standard_normal((w.num_blocks, w.num_kv_heads, D, bs), dtype=np.float32))
    tables = (np.arange(w.num_seqs, dtype=np.int32)[:, None] * w.max_blocks
              + np.arange(w.max_blocks, dtype=np.int32)[None, :])
    if w.shuffle_blocks:
        perm = rng.permutation(w.num_blocks).astype(np.int32)
        tables = perm[tables]
    return {"query": query, "k_cache": k_cache, "v_cache": v_cache,
            "block_tables": np.ascontiguousarray(tables, dtype=np.int32), "seq_lens": w.lens()}


# The page's shape table, rows #0-#7.
PAGED_CONFIGS = {
    f"P{i}": PagedWorkload(f"P{i}_s{n}_c{c}_h{hq}_kv{hkv}_d{d}_{dt}", n, c, hq, hkv, d,
                           dtype=dt, seed=60 + i)
    for i, (n, c, hq, hkv, d, dt) in enumerate([
        (256, 64, 16, 16, 128, "bf16"), (1, 128, 16, 2, 256, "bf16"),
        (128, 64, 3, 3, 128, "bf16"), (4, 128, 32, 4, 128, "bf16"),
        (4, 128, 32, 8, 128, "fp16"), (1, 128, 4, 1, 128, "bf16"),
        (4, 128, 40, 8, 128, "fp16"), (4, 128, 64, 8, 128, "fp16")])
}


def f16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """IEEE half bit patterns (uint16) -> exact float64 values."""
    return np.ascontiguousarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------- chunked delta-rule output
# atrex-bench "chunk_delta_rule_output" (page #004, input.py _make_inputs):
# q, k ~ 0.02 N(0,1) bf16 [B, T, Hq, K]; v ~ 0.02 N(0,1) bf16 [B, T, H, V];
# h ~ 0.02 N(0,1) bf16 [B, NC, H, K, V]; g = -U[0,1) float32 [B, T, H].
# Drawn here in the order q, k, v, h, g from one seeded generator.


@dataclass(frozen=True)
class ChunkWorkload:
    """One chunk_delta_rule_output call: the page's shape-table parameters."""

    name: str
    token_count: int
    num_v_heads: int
    value_dim: int
    num_q_heads: int
    chunk_size: int = 64
    key_dim: int = 128
    batch_size: int = 1
    seed: int = 0

    @property
    def num_chunks(self) -> int:
        return (self.token_count + self.chunk_size - 1) // self.chunk_size

    def algorithmic_bytes(self) -> int:
        """q, k, v, h read once, g read once, out written once."""
        B, T = self.batch_size, self.token_count
        qk = 2 * B * T * self.num_q_heads * self.key_dim * 2
        vo = 2 * B * T * self.num_v_heads * self.value_dim * 2
        hh = B * self.num_chunks * self.num_v_heads * self.key_dim * self.value_dim * 2
        return qk + vo + hh + B * T * self.num_v_heads * 4


def make_chunk_inputs(w: ChunkWorkload):
    rng = np.random.default_rng(w.seed)
    B, T, Hq, H = w.batch_size, w.token_count, w.num_q_heads, w.num_v_heads
    K, V = w.key_dim, w.value_dim
    f = lambda *s: (rng.standard_normal(s, dtype=np.float32) * np.float32(0.02))  # noqa: E731
    q = round_to_bf16_bits(f(B, T, Hq, K))
    k = round_to_bf16_bits(f(B, T, Hq, K))
    v = round_to_bf16_bits(f(B, T, H, V))
    h = round_to_bf16_bits(f(B, w.num_chunks, H, K, V))
    g = -rng.random((B, T, H), dtype=np.float32)
    return {"q": q, "k": k, "v": v, "h": h, "g": g}


# The page's shape table, rows #0-#15.
CHUNK_CONFIGS = {
    f"D{i}": ChunkWorkload(f"D{i}_t{t}_h{hv}_q{hq}", t, hv, 128, hq, seed=120 + i)
    for i, (t, hv, hq) in enumerate([
        (64, 32, 16), (128, 32, 16), (256, 32, 16), (512, 32, 16), (1024, 32, 16),
        (2048, 32, 16), (4096, 32, 16), (8192, 32, 16), (704, 16, 8), (1024, 16, 8),
        (2112, 16, 8), (4096, 16, 8), (8256, 16, 8), (4195, 32, 16), (11027, 32, 16),
        (14807, 32, 16)])
}
