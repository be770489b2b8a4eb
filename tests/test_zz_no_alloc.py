"""attn_varlen_fwd_noalloc, the entry point that allocates nothing.

Some callers cannot allocate device memory when they run attention: a server
that fixes its memory footprint at start-up, a host framework that owns every
allocation of its plug-ins, or a path where cudaMalloc/cudaFree would stall
the device.  This entry point takes its scratch from a fixed array compiled
into the library.  Here it is called through the C ABI on several batches in
a row (they share the one array) and checked three ways: against the CPU
oracle, bit for bit against attn_varlen_fwd_ws (which also runs every unit
whole), and, in a fresh process, for leaving the device's free memory
unchanged.  This file is collected last on purpose.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle
from gpu_helpers import abs_bits, assert_close, bf16_bound, device_inputs, to_bits
from workloads import C1, Workload, make_inputs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _call_noalloc(lib, t, cu_q, cu_k, out, stream):
    q = t["q"]
    return lib.attn_varlen_fwd_noalloc(
        q.data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), cu_q.data_ptr(), cu_k.data_ptr(),
        cu_q.numel() - 1, q.shape[1], q.shape[2], out.data_ptr(),
        ctypes.c_void_p(int(stream.cuda_stream)))


def _live_rows(cu):
    live = np.zeros(int(cu[-1]), bool)
    for i in range(len(cu) - 1):
        if cu[i + 1] > cu[i]:
            live[cu[i]:cu[i + 1]] = True
    return live


BATCHES = [Workload("noalloc_a", (1, 276, 600, 0, 1012, 130), 3, 72, seed=71),
           C1,
           Workload("noalloc_b", (200, 5), 2, 128, seed=72, seq_lens_k=(129, 300))]


def test_noalloc_matches_oracle_and_caller_workspace(cuda_lib):
    import torch
    lib = cuda_lib.load()
    stream = torch.cuda.current_stream()
    for w in BATCHES:  # consecutive calls share the one scratch array
        x = make_inputs(w)
        t, cu_q, cu_k = device_inputs(x, "cuda")
        out = torch.zeros_like(t["q"])
        assert _call_noalloc(lib, t, cu_q, cu_k, out, stream) == 0
        assert lib.attn_varlen_check_noalloc(ctypes.c_void_p(int(stream.cuda_stream))) == 0
        got = to_bits(out)
        live = _live_rows(x["cu_q"])
        ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
        absv = oracle.attn_varlen(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"])
        assert_close(got[live], ref[live], w.name + " no-alloc",
                     bound=bf16_bound(ref[live], absv[live]))
        ws = torch.zeros(cuda_lib.workspace_size(w.num_seqs), dtype=torch.uint8, device="cuda")
        want = cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, workspace=ws)
        cuda_lib.check(workspace=ws)
        np.testing.assert_array_equal(got[live], to_bits(want)[live])


def test_noalloc_rejects_too_many_sequences(cuda_lib):
    import torch
    from variable_length_prefill_gb300._binding import ERR_NOALLOC_LIMIT, NOALLOC_MAX_SEQS
    lib = cuda_lib.load()
    n = NOALLOC_MAX_SEQS + 1
    q = torch.zeros(n, 1, 128, dtype=torch.bfloat16, device="cuda")
    cu = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    rc = _call_noalloc(lib, {"q": q, "k": q, "v": q}, cu, cu, out, torch.cuda.current_stream())
    assert rc == ERR_NOALLOC_LIMIT
    assert "1024" in cuda_lib.strerror(rc)
    torch.cuda.synchronize()
    assert (out == 0).all()


# Run in a fresh process, where the library has no workspace of its own yet.
# The kernels are loaded eagerly and launched once through the caller-
# workspace entry point first, so neither module loading nor the driver's
# first local-memory reservation can move the free-memory figure; then the
# first no-alloc calls must leave it exactly where it was.
_CHILD = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, sys.argv[1])
    import numpy as np, torch
    import variable_length_prefill_gb300 as vlp
    from gpu_helpers import device_inputs
    from workloads import C1, Workload, make_inputs
    lib = vlp.load()
    s = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    batches = [C1, Workload("noalloc_c", (300, 1, 40), 2, 72, seed=73)]
    ins = [device_inputs(make_inputs(w), "cuda") for w in batches]
    outs = [torch.empty_like(t["q"]) for t, _, _ in ins]
    for (t, cq, ck), o in zip(ins, outs):
        ws = torch.zeros(vlp.workspace_size(cq.numel() - 1), dtype=torch.uint8, device="cuda")
        vlp.attn_varlen_fwd(t["q"], t["k"], t["v"], cq, ck, out=o, workspace=ws)
        vlp.check(workspace=ws)
    torch.cuda.synchronize()
    before = torch.cuda.mem_get_info()[0]
    for (t, cq, ck), o in zip(ins, outs):
        rc = lib.attn_varlen_fwd_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                         cq.data_ptr(), ck.data_ptr(), cq.numel() - 1,
                                         t["q"].shape[1], t["q"].shape[2], o.data_ptr(), s)
        assert rc == 0, rc
    assert lib.attn_varlen_check_noalloc(s) == 0
    after = torch.cuda.mem_get_info()[0]
    print("FREE_DELTA", before - after)
""")


def test_noalloc_leaves_free_memory_unchanged(cuda_lib):
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _CHILD, os.path.join(ROOT, "tests")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    deltas = [int(line.split()[1]) for line in r.stdout.splitlines()
              if line.startswith("FREE_DELTA")]
    assert deltas == [0], r.stdout + r.stderr
