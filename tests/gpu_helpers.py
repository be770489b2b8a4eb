"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
from workloads import bf16_bits_to_f64, make_inputs, sample_rows

# Tolerance on the bf16 output against the fp64 oracle (the unrounded exact
# result): max |err| <= 1e-2 and mean |err| <= 1e-3.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def to_dev(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def device_inputs(x: dict, device):
    import torch
    return ({n: to_dev(x[n], device) for n in ("q", "k", "v")},
            torch.from_numpy(x["cu_q"]).to(device), torch.from_numpy(x["cu_k"]).to(device))


def run_cuda(vlp, x: dict, device="cuda", out_fill: int | None = None):
    """Run the CUDA path; returns the output as bf16 bits (uint16, [T, H, D]).

    ``out_fill``: int16 bit pattern to pre-fill the output with (default:
    torch.empty_like)."""
    import torch
    t, cu_q, cu_k = device_inputs(x, device)
    out = None
    if out_fill is not None:
        out = torch.full(t["q"].shape, out_fill, dtype=torch.int16,
                         device=device).view(torch.bfloat16)
    out = vlp.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out)
    vlp.check()
    return to_bits(out)


def errors(got_bits: np.ndarray, ref: np.ndarray):
    err = np.abs(bf16_bits_to_f64(got_bits) - ref)
    return float(err.max()), float(err.mean())


def assert_close(got_bits, ref, what=""):
    mx, mean = errors(got_bits, ref)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max|err| {mx:.3e}, mean|err| {mean:.3e}"
    return mx, mean


def check_full(vlp, w, device="cuda"):
    """Every output row of workload `w` against the oracle."""
    x = make_inputs(w)
    got = run_cuda(vlp, x, device)
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    cu = x["cu_q"]
    live = np.zeros(got.shape[0], bool)
    for i in range(len(cu) - 1):
        if cu[i + 1] > cu[i]:
            live[cu[i]:cu[i + 1]] = True
    return assert_close(got[live], ref[live], w.name)


def check_sampled(vlp, w, rows_per_head: int, device="cuda"):
    """Seeded sample of output rows of workload `w` against the oracle."""
    x = make_inputs(w)
    got = run_cuda(vlp, x, device)
    rows = sample_rows(w, rows_per_head)
    ref = oracle.attn_rows(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], rows)
    return assert_close(got[rows[:, 0], rows[:, 1]], ref, w.name)
