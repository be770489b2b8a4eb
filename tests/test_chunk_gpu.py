"""Chunked gated delta-rule output (through the C ABI) against the CPU
oracle: the page's sixteen shapes (whole outputs where the oracle takes
seconds, else whole chunks sampled at the start, middle and ragged end),
batches, grouped and ungrouped head maps, one-token and ragged chunks, tied
and monotone gates, an explicit scale, and the empty call.

Tolerance, from the arithmetic: the output is rounded to bf16 (relative
2^-9) after fp32 accumulation, and each gated score is rounded to bf16 on
both sides, where a score whose fp32 and float64 values straddle a rounding
boundary moves by one bf16 step (2^-8 relative) on one of at most 64 terms.
Against the largest output magnitude M that is far below 1e-2 * M for any
element and 1e-3 * M on average, the bounds the tests use."""
import numpy as np
import pytest

import oracle
from workloads import CHUNK_CONFIGS, ChunkWorkload, bf16_bits_to_f64, make_chunk_inputs

pytestmark = pytest.mark.gpu

CS = 64


def _dev(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(vlp, x, scale=None):
    out = vlp.chunk_delta_rule_output(_dev(x["q"]), _dev(x["k"]), _dev(x["v"]), _dev(x["h"]),
                                      _dev(x["g"]), scale=scale)
    vlp.check()
    return out.view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def _assert_close(got_bits, ref, what):
    got = bf16_bits_to_f64(got_bits)
    assert got.shape == ref.shape, what
    m = float(np.abs(ref).max()) if ref.size else 0.0
    if m == 0.0:
        assert np.all(got == 0), what
        return
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    assert err.max() <= 1e-2 * m, f"{what}: max err {err.max():.3e} vs max|ref| {m:.3e}"
    assert err.mean() <= 1e-3 * m, f"{what}: mean err {err.mean():.3e} vs max|ref| {m:.3e}"


def _window(x, c0, c1):
    """Chunks [c0, c1) of every batch: chunks are independent of each other."""
    T = x["q"].shape[1]
    t0, t1 = c0 * CS, min(c1 * CS, T)
    w = {n: x[n][:, t0:t1] for n in ("q", "k", "v", "g")}
    w["h"] = x["h"][:, c0:c1]
    return w


FULL = [n for n, w in CHUNK_CONFIGS.items() if w.token_count <= 2112]
SAMPLED = [n for n in CHUNK_CONFIGS if n not in FULL]


@pytest.mark.parametrize("name", sorted(FULL))
def test_page_shapes_whole(cuda_lib, name):
    w = CHUNK_CONFIGS[name]
    x = make_chunk_inputs(w)
    _assert_close(_run(cuda_lib, x), oracle.chunk_o(**x), w.name)


@pytest.mark.parametrize("name", sorted(SAMPLED))
def test_page_shapes_sampled(cuda_lib, name):
    w = CHUNK_CONFIGS[name]
    x = make_chunk_inputs(w)
    got = _run(cuda_lib, x)
    nc = w.num_chunks
    for c0, c1 in ((0, 1), (nc // 2, nc // 2 + 1), (nc - 2, nc)):
        ref = oracle.chunk_o(**_window(x, c0, c1))
        _assert_close(got[:, c0 * CS:min(c1 * CS, w.token_count)], ref, f"{w.name} chunks {c0}-{c1}")


EXTRA = [
    # batches, value heads not a multiple of query heads (head map clamps)
    ChunkWorkload("b3_t100_h6_q4", 100, 6, 128, 4, batch_size=3, seed=140),
    # fewer value heads than query heads: value head hd reads query head hd
    ChunkWorkload("t130_h2_q4", 130, 2, 128, 4, seed=141),
    # one token; one token short of a chunk; one past a chunk
    ChunkWorkload("t1_h3_q1", 1, 3, 128, 1, seed=142),
    ChunkWorkload("b2_t63_h4_q2", 63, 4, 128, 2, batch_size=2, seed=143),
    ChunkWorkload("t65_h8_q8", 65, 8, 128, 8, seed=144),
]


@pytest.mark.parametrize("w", EXTRA, ids=lambda w: w.name)
def test_extra_shapes(cuda_lib, w):
    x = make_chunk_inputs(w)
    _assert_close(_run(cuda_lib, x), oracle.chunk_o(**x), w.name)


@pytest.mark.parametrize("gates", ["zero", "increasing", "decreasing", "ties"])
def test_gate_patterns(cuda_lib, gates):
    """Gates that keep every earlier key (all equal, or decreasing), none
    but the diagonal (increasing), and blocks of ties."""
    w = ChunkWorkload(f"gates_{gates}", 200, 4, 128, 2, batch_size=2, seed=145)
    x = make_chunk_inputs(w)
    B, T, H = x["g"].shape
    t = np.arange(T, dtype=np.float32)[None, :, None]
    g = {"zero": np.zeros_like(x["g"]),
         "increasing": np.broadcast_to(-2.0 + t / T, (B, T, H)),
         "decreasing": np.broadcast_to(-t / T, (B, T, H)),
         "ties": np.broadcast_to(-np.floor(t / 5) / 40.0, (B, T, H))}[gates]
    x["g"] = np.ascontiguousarray(g, dtype=np.float32)
    _assert_close(_run(cuda_lib, x), oracle.chunk_o(**x), w.name)


def test_explicit_scale(cuda_lib):
    w = ChunkWorkload("scale", 96, 4, 128, 4, seed=146)
    x = make_chunk_inputs(w)
    _assert_close(_run(cuda_lib, x, scale=0.3), oracle.chunk_o(**x, scale=0.3), w.name)


def test_empty_is_a_no_op(cuda_lib):
    w = ChunkWorkload("empty", 0, 4, 128, 2, seed=147)
    x = make_chunk_inputs(w)
    assert _run(cuda_lib, x).shape == (1, 0, 4, 128)


def test_deterministic(cuda_lib):
    x = make_chunk_inputs(CHUNK_CONFIGS["D8"])
    np.testing.assert_array_equal(_run(cuda_lib, x), _run(cuda_lib, x))
