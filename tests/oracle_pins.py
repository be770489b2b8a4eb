"""Pins for the CPU oracle: facts fixed by the page and by the mathematics.

Each ``pin_*`` function runs the oracle (optionally a copy with one planted
mistake, ``mutation=n``) on small inputs and raises AssertionError when the
result contradicts a closed form, an invariant or an independent library
routine.  What is computed is atrex-bench "attention_forward" (page #001,
reference.py, Model.forward): per non-empty query sequence and head,
softmax(Q K^T / sqrt(head_dim)) V over that sequence's keys.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
from workloads import bf16_bits_to_f64, round_to_bf16_bits


def _bits(x) -> np.ndarray:
    """Exactly-representable float values -> bf16 bits (asserts exactness)."""
    x = np.asarray(x, dtype=np.float32)
    b = round_to_bf16_bits(x)
    assert np.array_equal(bf16_bits_to_f64(b), x.astype(np.float64)), \
        "test input is not exactly representable in bf16"
    return b


def _rand_bits(rng, shape, scale=1.0):
    return round_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * scale)


def _cu(lens, offset=0):
    return np.concatenate([[offset], offset + np.cumsum(lens)]).astype(np.int32)


def _run(q, k, v, cu_q, cu_k, mutation):
    return oracle.attn_varlen(q, k, v, cu_q, cu_k, mutation=mutation)


def pin_single_key(mutation=0):
    """L_k = 1: the softmax weight is 1, so every output row is that key's v row."""
    rng = np.random.default_rng(11)
    H, D = 2, 8
    q = _rand_bits(rng, (5, H, D))
    k = _rand_bits(rng, (1, H, D))
    v = _rand_bits(rng, (1, H, D))
    out = _run(q, k, v, _cu([5]), _cu([1]), mutation)
    want = np.broadcast_to(bf16_bits_to_f64(v)[0], (5, H, D))
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


def pin_constant_keys(mutation=0):
    """All keys equal: all scores equal, so the output is the mean of V's rows."""
    rng = np.random.default_rng(12)
    H, D, L = 2, 8, 7
    q = _rand_bits(rng, (L, H, D))
    k = np.broadcast_to(_rand_bits(rng, (1, H, D)), (L, H, D)).copy()
    v = _rand_bits(rng, (L, H, D))
    out = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    want = np.broadcast_to(bf16_bits_to_f64(v).mean(axis=0), (L, H, D))
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)


def pin_zero_query(mutation=0):
    """q = 0: all scores are 0, so the output is the mean of V's rows."""
    rng = np.random.default_rng(13)
    H, D, L = 1, 16, 9
    q = _bits(np.zeros((L, H, D)))
    k = _rand_bits(rng, (L, H, D))
    v = _rand_bits(rng, (L, H, D))
    out = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    want = np.broadcast_to(bf16_bits_to_f64(v).mean(axis=0), (L, H, D))
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-12)


def pin_equal_values(mutation=0):
    """All V rows equal: the weights sum to 1, so the output is that row."""
    rng = np.random.default_rng(14)
    H, D, L = 2, 8, 6
    q = _rand_bits(rng, (L, H, D))
    k = _rand_bits(rng, (L, H, D))
    v = np.broadcast_to(_rand_bits(rng, (1, H, D)), (L, H, D)).copy()
    out = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    want = np.broadcast_to(bf16_bits_to_f64(v)[0], (L, H, D))
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-13)


def pin_two_keys(mutation=0):
    """Two keys: o = sigma(s1 - s2) v1 + sigma(s2 - s1) v2, scores set by hand.

    head_dim = 4, so the scale is 4^-1/2 = 1/2.  Query row 0 is (2,0,0,0):
    s1 = (2*1)/2 = 1 against k1 = (1,0,0,1), s2 = 0 against k2 = 0.  Query
    row 1 is (0,0,0,-4): s1 = -4/2 = -2, s2 = 0.
    """
    q = _bits([[[2, 0, 0, 0]], [[0, 0, 0, -4]]])
    k = _bits([[[1, 0, 0, 1]], [[0, 0, 0, 0]]])
    v = _bits([[[1, 0, 2, -1]], [[0, 4, 0, 1]]])
    out = _run(q, k, v, _cu([2]), _cu([2]), mutation)

    def sig(x):
        return 1.0 / (1.0 + math.exp(-x))
    v1 = np.array([1, 0, 2, -1], dtype=np.float64)
    v2 = np.array([0, 4, 0, 1], dtype=np.float64)
    want = np.stack([sig(1.0) * v1 + sig(-1.0) * v2,
                     sig(-2.0) * v1 + sig(2.0) * v2])[:, None, :]
    np.testing.assert_allclose(out, want, rtol=0, atol=1e-15)


def pin_key_permutation(mutation=0):
    """Permuting (k_j, v_j) pairs within a sequence leaves the output unchanged."""
    rng = np.random.default_rng(15)
    H, D, L = 2, 8, 13
    q = _rand_bits(rng, (L, H, D))
    k = _rand_bits(rng, (L, H, D))
    v = _rand_bits(rng, (L, H, D))
    perm = rng.permutation(L)
    a = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    b = _run(q, k[perm], v[perm], _cu([L]), _cu([L]), mutation)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def pin_key_translation(mutation=0):
    """k_j -> k_j + c shifts a row's scores by q.c/sqrt(D): output unchanged."""
    rng = np.random.default_rng(16)
    H, D, L = 1, 8, 10
    q = _bits(rng.integers(-2, 3, (L, H, D)) / 2.0)
    kf = rng.integers(-3, 4, (L, H, D)).astype(np.float64)
    c = rng.integers(-2, 3, (1, H, D)).astype(np.float64)
    v = _rand_bits(rng, (L, H, D))
    a = _run(q, _bits(kf), v, _cu([L]), _cu([L]), mutation)
    b = _run(q, _bits(kf + c), v, _cu([L]), _cu([L]), mutation)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def pin_value_affine(mutation=0):
    """V -> 2 V P + 1 b^T (P a column permutation) maps o -> 2 o P + b."""
    rng = np.random.default_rng(17)
    H, D, L = 1, 8, 9
    q = _rand_bits(rng, (L, H, D))
    k = _rand_bits(rng, (L, H, D))
    vf = rng.integers(-4, 5, (L, H, D)).astype(np.float64)
    b = rng.integers(-3, 4, (D,)).astype(np.float64)
    perm = rng.permutation(D)
    o1 = _run(q, k, _bits(vf), _cu([L]), _cu([L]), mutation)
    o2 = _run(q, k, _bits(2.0 * vf[:, :, perm] + b), _cu([L]), _cu([L]), mutation)
    np.testing.assert_allclose(o2, 2.0 * o1[:, :, perm] + b, rtol=0, atol=1e-12)


def pin_row_independence(mutation=0):
    """Changing one query row changes that output row only."""
    rng = np.random.default_rng(18)
    H, D, L = 2, 8, 11
    q = _rand_bits(rng, (L, H, D))
    k = _rand_bits(rng, (L, H, D))
    v = _rand_bits(rng, (L, H, D))
    a = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    q2 = q.copy()
    q2[4] = _rand_bits(rng, (H, D))
    b = _run(q2, k, v, _cu([L]), _cu([L]), mutation)
    keep = np.ones(L, bool)
    keep[4] = False
    np.testing.assert_array_equal(a[keep], b[keep])
    assert np.abs(a[4] - b[4]).max() > 1e-6


def pin_head_independence(mutation=0):
    """Changing one head's q, k and v changes that head's output only."""
    rng = np.random.default_rng(19)
    H, D, L = 3, 8, 7
    q = _rand_bits(rng, (L, H, D))
    k = _rand_bits(rng, (L, H, D))
    v = _rand_bits(rng, (L, H, D))
    a = _run(q, k, v, _cu([L]), _cu([L]), mutation)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for t in (q2, k2, v2):
        t[:, 1] = _rand_bits(rng, (L, D))
    b = _run(q2, k2, v2, _cu([L]), _cu([L]), mutation)
    np.testing.assert_array_equal(a[:, [0, 2]], b[:, [0, 2]])
    assert np.abs(a[:, 1] - b[:, 1]).max() > 1e-6


def pin_packing(mutation=0):
    """A packed batch equals each sequence run on its own."""
    rng = np.random.default_rng(20)
    H, D = 2, 8
    lens_q = [3, 1, 6, 4]
    lens_k = [5, 2, 6, 1]
    q = _rand_bits(rng, (sum(lens_q), H, D))
    k = _rand_bits(rng, (sum(lens_k), H, D))
    v = _rand_bits(rng, (sum(lens_k), H, D))
    cu_q, cu_k = _cu(lens_q), _cu(lens_k)
    packed = _run(q, k, v, cu_q, cu_k, mutation)
    for i in range(len(lens_q)):
        qs = q[cu_q[i]:cu_q[i + 1]]
        ks, vs = k[cu_k[i]:cu_k[i + 1]], v[cu_k[i]:cu_k[i + 1]]
        alone = _run(qs, ks, vs, _cu([lens_q[i]]), _cu([lens_k[i]]), mutation)
        np.testing.assert_allclose(packed[cu_q[i]:cu_q[i + 1]], alone,
                                   rtol=0, atol=1e-15)


def pin_empty_and_offsets(mutation=0):
    """Empty query slices write nothing, empty key slices give zeros, and rows
    outside [cu_q[0], cu_q[N]) are never written (the page allocates the
    output with empty_like and only fills the covered slices)."""
    rng = np.random.default_rng(21)
    H, D = 2, 8
    off = 3
    lens_q = [2, 0, 3]
    lens_k = [4, 2, 0]
    Tq = off + sum(lens_q) + 2
    Tk = off + sum(lens_k) + 2
    q = _rand_bits(rng, (Tq, H, D))
    k = _rand_bits(rng, (Tk, H, D))
    v = _rand_bits(rng, (Tk, H, D))
    cu_q, cu_k = _cu(lens_q, off), _cu(lens_k, off)
    out = _run(q, k, v, cu_q, cu_k, mutation)
    assert np.isnan(out[:off]).all() and np.isnan(out[cu_q[-1]:]).all()
    assert np.isfinite(out[cu_q[0]:cu_q[-1]]).all()
    np.testing.assert_array_equal(out[cu_q[2]:cu_q[3]], 0.0)


def pin_negative_slices(mutation=0):
    """cu_seqlens that step backwards.  A negative query slice is skipped like
    an empty one (the page's loop runs only while the query length is
    positive), and a negative key slice is an empty key set, so its query rows
    are zeros.  The live sequences must match torch float64 SDPA run on their
    slices alone, and rows no live query slice covers keep the fill value.

    cu_q = [20, 30, 25, 0, 10, 18] gives the query slices [20, 30), [30, 25),
    [25, 0), [0, 10) and [10, 18); cu_k = [0, 50, 40, 60, 5, 33] gives the key
    slices [0, 50), [50, 40), [40, 60), [60, 5) and [5, 33).  So sequences 1
    and 2 are skipped, sequence 3 has a negative key slice, and rows 18, 19
    and 30-39 belong to no sequence."""
    import torch
    rng = np.random.default_rng(24)
    H, D = 2, 8
    cu_q = np.array([20, 30, 25, 0, 10, 18], np.int32)
    cu_k = np.array([0, 50, 40, 60, 5, 33], np.int32)
    q = _rand_bits(rng, (40, H, D))
    k = _rand_bits(rng, (70, H, D))
    v = _rand_bits(rng, (70, H, D))
    out = _run(q, k, v, cu_q, cu_k, mutation)
    qf, kf, vf = (torch.from_numpy(bf16_bits_to_f64(x)) for x in (q, k, v))
    for qs, ks in ((slice(20, 30), slice(0, 50)), (slice(10, 18), slice(5, 33))):
        ref = torch.nn.functional.scaled_dot_product_attention(
            qf[qs].transpose(0, 1)[None], kf[ks].transpose(0, 1)[None],
            vf[ks].transpose(0, 1)[None])
        np.testing.assert_allclose(out[qs], ref[0].transpose(0, 1).numpy(), rtol=0,
                                   atol=1e-10)
    np.testing.assert_array_equal(out[0:10], 0.0)
    assert np.isnan(out[18:20]).all() and np.isnan(out[30:40]).all()


def pin_torch_sdpa(mutation=0):
    """torch's CPU scaled_dot_product_attention in float64, per sequence and
    with its default scale, is an independent implementation of the same
    operation; it must agree to 1e-10 on a packed batch with L_q != L_k."""
    import torch
    rng = np.random.default_rng(22)
    H, D = 3, 72
    lens_q = [1, 17, 40, 5]
    lens_k = [9, 33, 40, 1]
    q = _rand_bits(rng, (sum(lens_q), H, D))
    k = _rand_bits(rng, (sum(lens_k), H, D))
    v = _rand_bits(rng, (sum(lens_k), H, D))
    cu_q, cu_k = _cu(lens_q), _cu(lens_k)
    out = _run(q, k, v, cu_q, cu_k, mutation)
    qf = torch.from_numpy(bf16_bits_to_f64(q))
    kf = torch.from_numpy(bf16_bits_to_f64(k))
    vf = torch.from_numpy(bf16_bits_to_f64(v))
    for i in range(len(lens_q)):
        qs = qf[cu_q[i]:cu_q[i + 1]].transpose(0, 1)[None]
        ks = kf[cu_k[i]:cu_k[i + 1]].transpose(0, 1)[None]
        vs = vf[cu_k[i]:cu_k[i + 1]].transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, is_causal=False)
        ref = ref[0].transpose(0, 1).numpy()
        np.testing.assert_allclose(out[cu_q[i]:cu_q[i + 1]], ref, rtol=0, atol=1e-10)


def pin_rows_match_full(mutation=0):
    """The sampled-rows entry point returns the same rows as the full one."""
    rng = np.random.default_rng(23)
    H, D = 2, 16
    lens = [4, 0, 9, 1]
    q = _rand_bits(rng, (sum(lens), H, D))
    k = _rand_bits(rng, (sum(lens), H, D))
    v = _rand_bits(rng, (sum(lens), H, D))
    cu = _cu(lens)
    full = _run(q, k, v, cu, cu, mutation)
    rows = np.array([[0, 0], [3, 1], [4, 0], [12, 1], [13, 0], [5, 1]])
    part = oracle.attn_rows(q, k, v, cu, cu, rows, mutation=mutation)
    np.testing.assert_array_equal(part, full[rows[:, 0], rows[:, 1]])


# ------------------------------------------------------------------ causal
# The causal variant (not on the page; the common prefill neighbour): row r of
# a sequence sees keys j <= r + L_k - L_q, a mask aligned to the bottom-right
# corner; rows that see no key are zero.


def _run_causal(q, k, v, cu_q, cu_k, mutation):
    return oracle.attn_varlen(q, k, v, cu_q, cu_k, mutation=mutation, causal=True)


def pin_causal_first_and_last_row(mutation=0):
    """L_q = L_k: the first row sees one key, so it is that key's v row; the
    last row sees every key, so it equals the non-causal row."""
    rng = np.random.default_rng(40)
    H, D = 2, 8
    lens = [6, 1, 9]
    q = _rand_bits(rng, (sum(lens), H, D))
    k = _rand_bits(rng, (sum(lens), H, D))
    v = _rand_bits(rng, (sum(lens), H, D))
    cu = _cu(lens, offset=3)
    q = np.concatenate([_rand_bits(rng, (3, H, D)), q])
    k = np.concatenate([_rand_bits(rng, (3, H, D)), k])
    v = np.concatenate([_rand_bits(rng, (3, H, D)), v])
    causal = _run_causal(q, k, v, cu, cu, mutation)
    full = _run(q, k, v, cu, cu, mutation)
    vf = bf16_bits_to_f64(v)
    for i in range(len(lens)):
        first, last = cu[i], cu[i + 1] - 1
        np.testing.assert_allclose(causal[first], vf[first], rtol=0, atol=1e-15)
        np.testing.assert_allclose(causal[last], full[last], rtol=0, atol=1e-12)


def pin_causal_torch_sdpa(mutation=0):
    """L_q = L_k: torch's float64 SDPA with is_causal=True (lower triangle) is an
    independent implementation; it must agree to 1e-10."""
    import torch
    rng = np.random.default_rng(41)
    H, D = 3, 72
    lens = [1, 17, 40, 5]
    q = _rand_bits(rng, (sum(lens), H, D))
    k = _rand_bits(rng, (sum(lens), H, D))
    v = _rand_bits(rng, (sum(lens), H, D))
    cu = _cu(lens)
    out = _run_causal(q, k, v, cu, cu, mutation)
    qf, kf, vf = (torch.from_numpy(bf16_bits_to_f64(x)) for x in (q, k, v))
    for i in range(len(lens)):
        sl = slice(cu[i], cu[i + 1])
        ref = torch.nn.functional.scaled_dot_product_attention(
            qf[sl].transpose(0, 1)[None], kf[sl].transpose(0, 1)[None],
            vf[sl].transpose(0, 1)[None], is_causal=True)
        np.testing.assert_allclose(out[sl], ref[0].transpose(0, 1).numpy(), rtol=0, atol=1e-10)


def pin_causal_bottom_right(mutation=0):
    """L_q != L_k: row r equals the non-causal result over the first
    r + 1 + L_k - L_q keys (the mask's corner sits at the last query and the
    last key); rows with no visible key are zero."""
    rng = np.random.default_rng(42)
    H, D = 2, 8
    for lq, lk in ((5, 12), (9, 4)):
        q = _rand_bits(rng, (lq, H, D))
        k = _rand_bits(rng, (lk, H, D))
        v = _rand_bits(rng, (lk, H, D))
        out = _run_causal(q, k, v, _cu([lq]), _cu([lk]), mutation)
        for r in range(lq):
            n = min(lk, r + 1 + lk - lq)
            if n <= 0:
                np.testing.assert_array_equal(out[r], 0.0)
                continue
            one = _run(q[r:r + 1], k[:n], v[:n], _cu([1]), _cu([n]), mutation)
            np.testing.assert_allclose(out[r], one[0], rtol=0, atol=1e-12)


def pin_causal_rows_match_full(mutation=0):
    """The sampled-rows entry point applies the same causal mask."""
    rng = np.random.default_rng(43)
    H, D = 2, 16
    lens_q, lens_k = [4, 7, 3], [9, 7, 1]
    q = _rand_bits(rng, (sum(lens_q), H, D))
    k = _rand_bits(rng, (sum(lens_k), H, D))
    v = _rand_bits(rng, (sum(lens_k), H, D))
    cu_q, cu_k = _cu(lens_q), _cu(lens_k)
    full = _run_causal(q, k, v, cu_q, cu_k, mutation)
    rows = np.array([[0, 0], [3, 1], [4, 0], [10, 1], [11, 0], [12, 1], [13, 0]])
    part = oracle.attn_rows(q, k, v, cu_q, cu_k, rows, mutation=mutation, causal=True)
    np.testing.assert_array_equal(part, full[rows[:, 0], rows[:, 1]])


PINS = [pin_single_key, pin_constant_keys, pin_zero_query, pin_equal_values,
        pin_two_keys, pin_key_permutation, pin_key_translation,
        pin_value_affine, pin_row_independence, pin_head_independence,
        pin_packing, pin_empty_and_offsets, pin_negative_slices, pin_torch_sdpa, pin_rows_match_full,
        pin_causal_first_and_last_row, pin_causal_torch_sdpa, pin_causal_bottom_right,
        pin_causal_rows_match_full]
