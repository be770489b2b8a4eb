"""The chunked delta-rule output oracle against closed forms (state only,
intra-chunk only, the gate mask), chunk independence and padding, the head
map, and a brute-force loop; each planted mistake caught by a pin."""
import math

import numpy as np
import pytest

import oracle
from chunk_pins import CHUNK_PINS, _bf16_round_f64, _inputs
from workloads import CHUNK_CONFIGS, bf16_bits_to_f64, make_chunk_inputs


@pytest.mark.parametrize("pin", CHUNK_PINS, ids=lambda p: p.__name__)
def test_chunk_pin(pin):
    pin(0)


# 30 scale left out   31 the intra-chunk weight not rounded to bf16
# 32 gate mask kept where g_r >= g_j   33 the lower-triangle mask dropped
# 34 value head hd read q/k head hd % Hq
CHUNK_MUTATIONS = [30, 31, 32, 33, 34]


@pytest.mark.parametrize("mutation", CHUNK_MUTATIONS)
def test_chunk_planted_mistake_is_caught(mutation):
    failed = []
    for pin in CHUNK_PINS:
        try:
            pin(mutation)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches planted mistake {mutation}"


def test_chunk_brute_force_tiny():
    """Scalar loops in Python floats, written from the definition."""
    rng = np.random.default_rng(95)
    B, T, Hq, H, K, V, cs = 1, 7, 2, 2, 4, 3, 3
    x = _inputs(rng, B, T, Hq, H, K, V, cs)
    out = oracle.chunk_o(x["q"], x["k"], x["v"], x["h"], x["g"], chunk_size=cs)
    q, k, v, hh = (bf16_bits_to_f64(x[n]) for n in ("q", "k", "v", "h"))
    g = x["g"].astype(np.float64)
    for hd in range(H):
        qh = min(hd // (H // Hq), Hq - 1)
        for t in range(T):
            c, r = divmod(t, cs)
            row = []
            for col in range(V):
                s = sum(q[0, t, qh, i] * hh[0, c, hd, i, col] for i in range(K)) * math.exp(g[0, t, hd])
                for j in range(r + 1):
                    tj = c * cs + j
                    if tj >= T or g[0, t, hd] > g[0, tj, hd]:
                        continue
                    a = sum(q[0, t, qh, i] * k[0, tj, qh, i] for i in range(K))
                    a = float(_bf16_round_f64(np.array(a * math.exp(g[0, t, hd] - g[0, tj, hd]))))
                    s += a * v[0, tj, hd, col]
                row.append(s / math.sqrt(K))
            np.testing.assert_allclose(out[0, t, hd], row, rtol=1e-12, atol=1e-18)


def test_chunk_shapes_follow_the_page():
    """The page's generator: h has one state per chunk, g is in (-1, 0]."""
    for w in list(CHUNK_CONFIGS.values())[:3]:
        x = make_chunk_inputs(w)
        assert x["h"].shape == (1, w.num_chunks, w.num_v_heads, w.key_dim, w.value_dim)
        assert x["g"].dtype == np.float32 and (x["g"] <= 0).all() and (x["g"] > -1).all()
