"""Pins for the paged-decode oracle: facts fixed by the page and by the
mathematics.  What is computed is atrex-bench "paged_attention_decode"
(page #024, reference.py, Model.forward): one query row per head and
sequence, attending over the sequence's context tokens gathered through its
block table from a split-x key cache and a transposed value cache, each KV
head shared by Hq / Hkv consecutive query heads."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import (PagedWorkload, bf16_bits_to_f64, f16_bits_to_f64, make_paged_inputs,
                       round_to_bf16_bits)


def _decode(x, w, mutation):
    return oracle.paged_decode(x["query"], x["k_cache"], x["v_cache"], x["block_tables"],
                               x["seq_lens"], w.dtype, mutation=mutation)


def _widen(bits, dtype):
    return f16_bits_to_f64(bits) if dtype == "fp16" else bf16_bits_to_f64(bits)


def _gather(x, w, i):
    """Context tokens of sequence i in token order: keys and values [L, Hkv, D],
    written out from the cache layouts (token t: block table entry t // bs,
    position t % bs; key element d at [d // 8][pos][d % 8], value at [d][pos])."""
    L = int(x["seq_lens"][i])
    kc = _widen(x["k_cache"], w.dtype)
    vc = _widen(x["v_cache"], w.dtype)
    keys = np.zeros((L, w.num_kv_heads, w.head_size))
    vals = np.zeros((L, w.num_kv_heads, w.head_size))
    for t in range(L):
        b = x["block_tables"][i, t // w.block_size]
        p = t % w.block_size
        for g in range(w.num_kv_heads):
            keys[t, g] = kc[b, g, :, p, :].reshape(-1)
            vals[t, g] = vc[b, g, :, p]
    return keys, vals


def pin_paged_matches_dense_oracle(mutation=0):
    """Each sequence equals the (separately pinned) dense attention oracle with
    one query row and the gathered context, every KV head repeated for its
    Hq / Hkv query heads."""
    w = PagedWorkload("pin", 3, 9, 6, 2, 16, block_size=4, seed=70, seq_lens=(5, 0, 9),
                      shuffle_blocks=True)
    x = make_paged_inputs(w)
    out = _decode(x, w, mutation)
    qpk = w.num_query_heads // w.num_kv_heads
    for i in range(w.num_seqs):
        L = int(x["seq_lens"][i])
        if L <= 0:
            continue
        keys, vals = _gather(x, w, i)
        kq = np.repeat(keys, qpk, axis=1)  # query head h -> KV head h // qpk
        vq = np.repeat(vals, qpk, axis=1)
        # the gathered values are exact bf16 numbers: re-encode them for the dense oracle
        kb, vb = round_to_bf16_bits(kq.astype(np.float32)), round_to_bf16_bits(vq.astype(np.float32))
        ref = oracle.attn_varlen(x["query"][i:i + 1], kb, vb, np.array([0, 1], np.int32),
                                 np.array([0, L], np.int32))
        np.testing.assert_allclose(out[i], ref[0], rtol=0, atol=1e-12)


def pin_paged_torch_sdpa_gqa(mutation=0):
    """torch's float64 SDPA with enable_gqa (query head h reads KV head
    h // (Hq / Hkv)) on the gathered context, fp16 caches."""
    import torch
    w = PagedWorkload("pin", 2, 21, 8, 2, 32, block_size=8, dtype="fp16", seed=71,
                      seq_lens=(21, 13), shuffle_blocks=True)
    x = make_paged_inputs(w)
    out = _decode(x, w, mutation)
    for i in range(w.num_seqs):
        keys, vals = _gather(x, w, i)
        q = torch.from_numpy(f16_bits_to_f64(x["query"][i]))[None, :, None, :]
        k = torch.from_numpy(keys).permute(1, 0, 2)[None]
        v = torch.from_numpy(vals).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, enable_gqa=True)
        np.testing.assert_allclose(out[i], ref[0, :, 0].numpy(), rtol=0, atol=1e-10)


def pin_paged_block_permutation(mutation=0):
    """Where the blocks physically sit does not matter: shuffling the physical
    block ids (and the table with them) gives the same result."""
    base = PagedWorkload("pin", 2, 37, 4, 4, 16, block_size=8, seed=72, seq_lens=(37, 20))
    a_in = make_paged_inputs(base)
    # the same logical cache, physically permuted
    perm = np.random.default_rng(5).permutation(base.num_blocks)
    b_in = dict(a_in)
    b_in["k_cache"] = np.empty_like(a_in["k_cache"])
    b_in["v_cache"] = np.empty_like(a_in["v_cache"])
    b_in["k_cache"][perm] = a_in["k_cache"]
    b_in["v_cache"][perm] = a_in["v_cache"]
    b_in["block_tables"] = perm[a_in["block_tables"]].astype(np.int32)
    np.testing.assert_array_equal(_decode(a_in, base, mutation), _decode(b_in, base, mutation))


def pin_paged_empty_context(mutation=0):
    """ctx_len <= 0: the sequence is skipped and its rows stay zero."""
    w = PagedWorkload("pin", 3, 5, 2, 1, 8, block_size=4, seed=73, seq_lens=(0, -3, 5))
    x = make_paged_inputs(w)
    out = _decode(x, w, mutation)
    assert np.all(out[0] == 0.0) and np.all(out[1] == 0.0)
    assert np.all(np.isfinite(out[2])) and np.any(out[2] != 0.0)


def pin_paged_single_token(mutation=0):
    """ctx_len = 1: the only weight is 1, so every query head of a group gets
    that token's value row of its KV head."""
    w = PagedWorkload("pin", 2, 1, 6, 3, 16, block_size=4, seed=74, shuffle_blocks=True)
    x = make_paged_inputs(w)
    out = _decode(x, w, mutation)
    vc = _widen(x["v_cache"], w.dtype)
    for i in range(w.num_seqs):
        b = x["block_tables"][i, 0]
        for h in range(w.num_query_heads):
            np.testing.assert_array_equal(out[i, h], vc[b, h // 2, :, 0])


def pin_paged_half_values(mutation=0):
    """fp16 caches are read as IEEE binary16: a single-token context returns
    its value row exactly, including the largest normal, a subnormal and a
    signed zero."""
    w = PagedWorkload("pin", 1, 1, 1, 1, 8, block_size=2, dtype="fp16", seed=75)
    x = make_paged_inputs(w)
    pattern = np.array([0x3C00, 0xC000, 0x7BFF, 0x0001, 0x8400, 0x3555, 0x8000, 0x0400],
                       dtype=np.uint16)
    want = np.array([1.0, -2.0, 65504.0, 2.0 ** -24, -2.0 ** -14, 0.333251953125, -0.0,
                     2.0 ** -14])
    b = x["block_tables"][0, 0]
    x["v_cache"][b, 0, :, 0] = pattern
    out = _decode(x, w, mutation)
    np.testing.assert_array_equal(out[0, 0], want)


PAGED_PINS = [pin_paged_matches_dense_oracle, pin_paged_torch_sdpa_gqa,
              pin_paged_block_permutation, pin_paged_empty_context, pin_paged_single_token,
              pin_paged_half_values]
