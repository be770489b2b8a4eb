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
# Where a sequence is so short that its outputs are averages of a handful of
# values of size ~1-4, bf16 arithmetic alone can exceed 1e-2: P is rounded to
# bf16 (unit roundoff 2^-8) before P.V, which moves o by at most
# 2^-8 * sum_j w_j |v_j|, and the output's own rounding adds at most
# 2^-8 * |o|.  An element may exceed MAX_ABS only while it stays inside
# BF16_U * (sum_j w_j |v_j| + |o|) * (1 + BOUND_SLACK); the mean bar always holds.
BF16_U = 2.0 ** -8
BOUND_SLACK = 0.02
REPORT: list = []


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


def run_cuda(vlp, x: dict, device="cuda", out_fill: int | None = None,
             caller_workspace: bool = False, causal: bool = False):
    """Run the CUDA path; returns the output as bf16 bits (uint16, [T, H, D]).

    ``out_fill``: int16 bit pattern to pre-fill the output with (default:
    torch.empty_like).  ``caller_workspace``: pass a caller-owned workspace of
    workspace_size(num_seqs) bytes (that entry point never splits units)."""
    import torch
    t, cu_q, cu_k = device_inputs(x, device)
    out = None
    if out_fill is not None:
        out = torch.full(t["q"].shape, out_fill, dtype=torch.int16,
                         device=device).view(torch.bfloat16)
    if caller_workspace:
        ws = torch.zeros(vlp.workspace_size(len(x["cu_q"]) - 1), dtype=torch.uint8,
                         device=device)
        out = vlp.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out, workspace=ws)
        vlp.check(workspace=ws)
    else:
        out = vlp.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out, causal=causal)
        vlp.check()
    return to_bits(out)


def errors(got_bits: np.ndarray, ref: np.ndarray):
    err = np.abs(bf16_bits_to_f64(got_bits) - ref)
    return float(err.max()), float(err.mean())


def bf16_bound(ref: np.ndarray, ref_absv: np.ndarray) -> np.ndarray:
    """Per-element error bound of bf16 arithmetic (see BF16_U above);
    ref_absv is the oracle applied to |v| (= sum_j w_j |v_j|)."""
    return BF16_U * (ref_absv + np.abs(ref)) * (1.0 + BOUND_SLACK) + 1e-6


def assert_close(got_bits, ref, what="", bound=None):
    """The stated bar; with ``bound``, elements above MAX_ABS must stay inside it.
    ``got_bits``: bf16 bit patterns."""
    return assert_close_values(bf16_bits_to_f64(got_bits), ref, what, bound)


def assert_close_values(got, ref, what="", bound=None):
    """assert_close for outputs already widened to float64."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    REPORT.append((what, err.size, mx, mean))
    assert mean <= MEAN_ABS, f"{what}: mean|err| {mean:.3e} > {MEAN_ABS}"
    if bound is None:
        assert mx <= MAX_ABS, f"{what}: max|err| {mx:.3e} > {MAX_ABS}"
    else:
        over = err > np.maximum(MAX_ABS, bound)
        assert not over.any(), (f"{what}: {int(over.sum())} elements beyond max(1e-2, bf16 bound); "
                                 f"worst err {float(err[over].max()):.3e}")
    return mx, mean


def abs_bits(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of |x|."""
    return bits & np.uint16(0x7FFF)


def check_full(vlp, w, device="cuda", short_sequences=False, x=None, causal=False):
    """Every output row of workload `w` (or of inputs `x`) against the oracle.

    ``short_sequences``: outputs are averages of a handful of values (very
    short sequences, or scores so spread that a few keys dominate), so the
    per-element bf16 bound applies above MAX_ABS (the mean bar still holds).
    """
    x = make_inputs(w) if x is None else x
    got = run_cuda(vlp, x, device, causal=causal)
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal=causal)
    cu = x["cu_q"]
    live = np.zeros(got.shape[0], bool)
    for i in range(len(cu) - 1):
        if cu[i + 1] > cu[i]:
            live[cu[i]:cu[i + 1]] = True
    bound = None
    if short_sequences:
        absv = oracle.attn_varlen(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"],
                                  causal=causal)
        bound = bf16_bound(ref[live], absv[live])
    return assert_close(got[live], ref[live], w.name + (" causal" if causal else ""),
                        bound=bound)


def check_sampled(vlp, w, rows_per_head: int, device="cuda", causal=False):
    """Seeded sample of output rows of workload `w` against the oracle."""
    x = make_inputs(w)
    got = run_cuda(vlp, x, device, causal=causal)
    rows = sample_rows(w, rows_per_head)
    ref = oracle.attn_rows(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], rows, causal=causal)
    bound = None
    if causal:  # the first rows of a sequence average only a few values
        absv = oracle.attn_rows(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"], rows,
                                causal=True)
        bound = bf16_bound(ref, absv)
    return assert_close(got[rows[:, 0], rows[:, 1]], ref,
                        w.name + (" causal" if causal else ""), bound=bound)


def check_rows(vlp, w, rows: np.ndarray, device="cuda", caller_workspace=False, x=None):
    """Given (token, head) output rows of workload `w` against the oracle;
    returns the CUDA output (bf16 bits) for further comparisons."""
    x = make_inputs(w) if x is None else x
    got = run_cuda(vlp, x, device, caller_workspace=caller_workspace)
    ref = oracle.attn_rows(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], rows)
    assert_close(got[rows[:, 0], rows[:, 1]], ref,
                 w.name + (" caller workspace" if caller_workspace else ""))
    return got
