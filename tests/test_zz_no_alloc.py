"""attn_varlen_fwd_noalloc, the entry point that allocates nothing.

Some callers cannot allocate device memory when they run attention (a server
that fixes its memory footprint at start-up, a host framework that owns every
allocation of its plug-ins, a path where cudaMalloc/cudaFree would stall the
device).  This entry point takes its scratch from a fixed array compiled into
the library.  Here it is called through the C ABI, twice in a row on
different batches, and its output is compared with attn_varlen_fwd's within
the tolerance the parity tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import MAX_ABS, MEAN_ABS, device_inputs, to_bits
from workloads import C1, Workload, bf16_bits_to_f64, make_inputs

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, t, cu_q, cu_k, out, stream):
    q = t["q"]
    return lib.attn_varlen_fwd_noalloc(
        q.data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), cu_q.data_ptr(), cu_k.data_ptr(),
        cu_q.numel() - 1, q.shape[1], q.shape[2], out.data_ptr(),
        ctypes.c_void_p(int(stream.cuda_stream)))


def test_noalloc_matches_allocating_entry_point(cuda_lib):
    import torch
    lib = cuda_lib.load()
    stream = torch.cuda.current_stream()
    batches = [Workload("noalloc_a", (1, 276, 600, 0, 1012, 130), 3, 72, seed=71),
               C1,
               Workload("noalloc_b", (200, 5), 2, 128, seed=72, seq_lens_k=(129, 300))]
    for w in batches:  # consecutive calls share the one scratch array
        x = make_inputs(w)
        t, cu_q, cu_k = device_inputs(x, "cuda")
        want = to_bits(cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k))
        cuda_lib.check()
        out = torch.zeros_like(t["q"])
        assert _call_noalloc(lib, t, cu_q, cu_k, out, stream) == 0
        torch.cuda.synchronize()
        got = to_bits(out)
        cu = x["cu_q"]
        live = np.zeros(got.shape[0], bool)
        for i in range(len(cu) - 1):
            if cu[i + 1] > cu[i]:
                live[cu[i]:cu[i + 1]] = True
        err = np.abs(bf16_bits_to_f64(got[live]) - bf16_bits_to_f64(want[live]))
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (w.name, err.max(), err.mean())


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
