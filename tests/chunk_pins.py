"""Pins for the chunked gated delta-rule output oracle: facts fixed by the
page and by the mathematics.  What is computed is atrex-bench
"chunk_delta_rule_output" (page #004, reference.py, Model.forward): per
64-token chunk, the state part exp(g) * (q h) plus the gated lower-triangular
intra-chunk part bf16(q k^T * exp(g_r - g_j), kept where g_r <= g_j) v, all
times key_dim^-1/2."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import bf16_bits_to_f64, round_to_bf16_bits


def _bf16_round_f64(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bfloat16 value (ties to even), by integer
    arithmetic on the float64 bit pattern: keep 7 explicit fraction bits."""
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.int64)
    drop = 52 - 7
    half = np.int64(1) << (drop - 1)
    lsb = (bits >> drop) & 1
    rounded = ((bits + half - 1 + lsb) >> drop) << drop
    out = rounded.view(np.float64)
    return np.where(np.isfinite(x) & (x != 0), out, x)


def _rand(rng, *shape, s=0.02):
    return round_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(s))


def _inputs(rng, B, T, Hq, H, K, V, cs):
    nc = (T + cs - 1) // cs
    return {"q": _rand(rng, B, T, Hq, K), "k": _rand(rng, B, T, Hq, K),
            "v": _rand(rng, B, T, H, V), "h": _rand(rng, B, nc, H, K, V),
            "g": -rng.random((B, T, H), dtype=np.float32)}


def _run(x, cs, mutation):
    return oracle.chunk_o(x["q"], x["k"], x["v"], x["h"], x["g"], chunk_size=cs,
                          mutation=mutation)


def pin_state_only(mutation=0):
    """k = 0: only the state part is left, scale * exp(g_t) * (q_t h_chunk)."""
    rng = np.random.default_rng(90)
    B, T, Hq, H, K, V, cs = 2, 11, 2, 4, 8, 6, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    x["k"][:] = 0
    out = _run(x, cs, mutation)
    q, hh = bf16_bits_to_f64(x["q"]), bf16_bits_to_f64(x["h"])
    scale = K ** -0.5
    for b in range(B):
        for hd in range(H):
            qh = min(hd // (H // Hq), Hq - 1)
            for t in range(T):
                want = scale * np.exp(float(x["g"][b, t, hd])) * (q[b, t, qh] @ hh[b, t // cs, hd])
                np.testing.assert_allclose(out[b, t, hd], want, rtol=1e-12, atol=1e-18)


def pin_intra_only(mutation=0):
    """h = 0, g = 0: every gate is exp(0) = 1, so the output is
    scale * tril(bf16(Q K^T)) V within each chunk."""
    rng = np.random.default_rng(91)
    B, T, Hq, H, K, V, cs = 1, 9, 1, 2, 8, 5, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    x["h"][:] = 0
    x["g"][:] = 0
    out = _run(x, cs, mutation)
    q, k, v = (bf16_bits_to_f64(x[n]) for n in ("q", "k", "v"))
    scale = K ** -0.5
    for hd in range(H):
        for c0 in range(0, T, cs):
            sl = slice(c0, min(T, c0 + cs))
            a = _bf16_round_f64(np.tril(q[0, sl, 0] @ k[0, sl, 0].T))
            np.testing.assert_allclose(out[0, sl, hd], scale * (a @ v[0, sl, hd]), rtol=1e-12,
                                       atol=1e-18)


def pin_gate_mask(mutation=0):
    """g strictly increasing inside every chunk: g_r > g_j for every j < r, so
    only the diagonal (gate exp(0) = 1) survives the mask."""
    rng = np.random.default_rng(92)
    B, T, Hq, H, K, V, cs = 1, 8, 1, 1, 8, 4, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    x["g"][0, :, 0] = -1.0 + 0.1 * np.arange(T, dtype=np.float32)
    out = _run(x, cs, mutation)
    q, k, v, hh = (bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "h"))
    scale = K ** -0.5
    for t in range(T):
        state = np.exp(float(x["g"][0, t, 0])) * (q[0, t, 0] @ hh[0, t // cs, 0])
        diag = _bf16_round_f64(np.array(q[0, t, 0] @ k[0, t, 0]))
        np.testing.assert_allclose(out[0, t, 0], scale * (state + diag * v[0, t, 0]), rtol=1e-12,
                                   atol=1e-18)


def pin_chunk_independence_and_padding(mutation=0):
    """A chunk reads only its own tokens and state; a padded last chunk gives
    the rows it has the same values as a run over those tokens alone."""
    rng = np.random.default_rng(93)
    B, T, Hq, H, K, V, cs = 1, 10, 1, 2, 8, 4, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    a = _run(x, cs, mutation)
    y = {n: x[n].copy() for n in x}
    y["q"][:, 4:] = _rand(rng, B, T - 4, Hq, K)   # change chunks 1 and 2
    y["v"][:, 4:] = _rand(rng, B, T - 4, H, V)
    y["h"][:, 1:] = _rand(rng, B, 2, H, K, V)
    b = _run(y, cs, mutation)
    np.testing.assert_array_equal(a[:, :4], b[:, :4])
    z = {"q": x["q"][:, :6], "k": x["k"][:, :6], "v": x["v"][:, :6], "h": x["h"][:, :2],
         "g": x["g"][:, :6]}
    np.testing.assert_array_equal(_run(z, cs, mutation), a[:, :6])


def pin_head_map(mutation=0):
    """H = 4 value heads over Hq = 2 query/key heads: heads 0-1 read q/k head
    0, heads 2-3 read head 1; with head 1 zero, heads 2-3 are zero."""
    rng = np.random.default_rng(94)
    B, T, Hq, H, K, V, cs = 1, 6, 2, 4, 8, 4, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    x["q"][:, :, 1] = 0
    x["k"][:, :, 1] = 0
    out = _run(x, cs, mutation)
    assert np.all(out[:, :, 2:] == 0.0)
    assert np.all(np.abs(out[:, :, :2]).max(axis=-1) > 0)


def pin_head_map_clamped(mutation=0):
    """H = 6 value heads over Hq = 4: H / Hq rounds down to 1, so value head
    hd reads q/k head min(hd, 3); heads 3, 4 and 5 all read head 3.  With
    q/k heads 0-2 zero, value heads 0-2 are zero and 3-5 are not."""
    rng = np.random.default_rng(96)
    B, T, Hq, H, K, V, cs = 1, 5, 4, 6, 8, 4, 4
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    x["q"][:, :, :3] = 0
    x["k"][:, :, :3] = 0
    out = _run(x, cs, mutation)
    assert np.all(out[:, :, :3] == 0.0)
    assert np.all(np.abs(out[:, :, 3:]).max(axis=-1) > 0)


CHUNK_PINS = [pin_state_only, pin_intra_only, pin_gate_mask,
              pin_chunk_independence_and_padding, pin_head_map, pin_head_map_clamped]
