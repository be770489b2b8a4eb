"""The CPU oracle against closed forms, invariants, torch's float64 SDPA and a
brute-force loop; and each planted mistake caught by at least one pin."""
import math

import numpy as np
import pytest

import oracle
from oracle_pins import PINS
from workloads import C1, C5, bf16_bits_to_f64, make_inputs


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(0)


# Each planted mistake is one a careful reader could make:
#  1 scale 1/D instead of 1/sqrt(D)      3 weights not normalised
#  4 keys located with the query offsets 5 head and dim indices swapped in K
#  6 the last key dropped                7 V row of the query token
#  9 sign of the exponent flipped       10 NaN instead of zeros for L_k = 0
# 11 causal: the diagonal key dropped   12 causal: mask aligned top-left
# 13 a backwards cu_seqlens slice read as the reversed range
MUTATIONS = [1, 3, 4, 5, 6, 7, 9, 10, 11, 12, 13]


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    failed = []
    for pin in PINS:
        try:
            pin(mutation)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches planted mistake {mutation}"


def _brute_force(q, k, v, cu_q, cu_k, H, D, causal=False):
    """Scalar triple loop in Python floats, for tiny inputs.  ``causal``: row
    r of a sequence sees keys j <= r + L_k - L_q."""
    qf, kf, vf = (bf16_bits_to_f64(x) for x in (q, k, v))
    out = {}
    for i in range(len(cu_q) - 1):
        lq, lk = cu_q[i + 1] - cu_q[i], cu_k[i + 1] - cu_k[i]
        for r in range(cu_q[i], cu_q[i + 1]):
            for h in range(H):
                ks = [j for j in range(cu_k[i], cu_k[i + 1])
                      if not causal or (j - cu_k[i]) <= (r - cu_q[i]) + lk - lq]
                if not ks:
                    out[(r, h)] = [0.0] * D
                    continue
                s = [sum(qf[r, h, d] * kf[j, h, d] for d in range(D)) / math.sqrt(D)
                     for j in ks]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                z = sum(w)
                out[(r, h)] = [sum(w[n] * vf[j, h, d] for n, j in enumerate(ks)) / z
                               for d in range(D)]
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [4, 72, 128, 256])
def test_brute_force_tiny(D, causal):
    rng = np.random.default_rng(30 + D)
    from oracle_pins import _cu, _rand_bits
    H = 2
    lens_q, lens_k = [1, 3, 0, 2, 4, 3], [2, 3, 4, 0, 2, 5]
    q = _rand_bits(rng, (sum(lens_q), H, D))
    k = _rand_bits(rng, (sum(lens_k), H, D))
    v = _rand_bits(rng, (sum(lens_k), H, D))
    cu_q, cu_k = _cu(lens_q), _cu(lens_k)
    out = oracle.attn_varlen(q, k, v, cu_q, cu_k, causal=causal)
    ref = _brute_force(q, k, v, cu_q, cu_k, H, D, causal=causal)
    for (r, h), row in ref.items():
        np.testing.assert_allclose(out[r, h], row, rtol=0, atol=1e-12)


def test_c1_against_torch_sdpa_f64():
    """The smallest workload, every row, against torch float64 SDPA."""
    import torch
    x = make_inputs(C1)
    out = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    qf, kf, vf = (torch.from_numpy(bf16_bits_to_f64(x[n])).transpose(0, 1)[None]
                  for n in ("q", "k", "v"))
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf)
    np.testing.assert_allclose(out, ref[0].transpose(0, 1).numpy(), rtol=0, atol=1e-10)


def test_c5_small_members_against_torch_sdpa_f64():
    """The packed batch's short members (and the length-1 one) against torch."""
    import torch
    x = make_inputs(C5)
    cu = x["cu_q"]
    rows = []
    for i in range(4):  # lengths 1, 276, 600, 1012
        rows += [[t, h] for t in range(cu[i], cu[i + 1], 7) for h in range(C5.num_heads)]
    rows = np.array(rows)
    got = oracle.attn_rows(x["q"], x["k"], x["v"], cu, x["cu_k"], rows)
    qf, kf, vf = (torch.from_numpy(bf16_bits_to_f64(x[n])) for n in ("q", "k", "v"))
    for n, (t, h) in enumerate(rows):
        i = int(np.searchsorted(cu, t, side="right") - 1)
        ks = slice(cu[i], cu[i + 1])
        ref = torch.nn.functional.scaled_dot_product_attention(
            qf[t:t + 1, h][None], kf[ks, h][None], vf[ks, h][None])[0, 0].numpy()
        np.testing.assert_allclose(got[n], ref, rtol=0, atol=1e-10)


def test_threads_reported():
    assert oracle.max_threads(1) == 1
    assert oracle.max_threads(0) >= 1
