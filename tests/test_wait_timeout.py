"""The bounded-wait give-up path of the attention kernel, run on purpose.

Every wait in the attention kernel gives up after a time limit: it records a
bit in the status word of the call's workspace, makes the CTA's other roles
stop waiting, lets the copies and MMAs it already issued finish (again with a
bound), frees TMEM and returns, so the context stays usable.  The product
library waits 4 s.  This test loads a separate test build (build variant
"testhooks") that waits 50 ms and can withhold CTA 0's first K/V tile: that
tile is neither copied nor announced to its barrier, so the MMA warp's wait on
it runs out while no copy is in flight on that slot.  Each workspace kind (the
library's own, a caller's, the no-alloc scratch) must then report
ATTN_VARLEN_ERR_DEVICE_TIMEOUT once, and the next normal call on the device
must meet the parity bar against the oracle.
"""
import ctypes
import time

import pytest

import oracle
from gpu_helpers import assert_close, device_inputs, to_bits
from workloads import C1, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def waitlib(cuda_lib):
    from variable_length_prefill_gb300 import _binding
    lib = ctypes.CDLL(cuda_lib.build(variant="testhooks"))
    for name, (res, args) in _binding.SYMBOLS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    lib.attn_varlen_test_withhold.argtypes = [ctypes.c_int]
    lib.attn_varlen_test_withhold.restype = None
    yield lib
    lib.attn_varlen_test_withhold(0)


def _inputs():
    import torch
    x = make_inputs(C1)
    t, cu_q, cu_k = device_inputs(x, "cuda")
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    return x, t, cu_q, cu_k, torch.zeros_like(t["q"]), ref


def _run(lib, kind, t, cu_q, cu_k, out, s, ws=None):
    args = (t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(), cu_q.data_ptr(),
            cu_k.data_ptr(), cu_q.numel() - 1, t["q"].shape[1], t["q"].shape[2], out.data_ptr())
    if kind == "owned":
        return lib.attn_varlen_fwd(*args, s)
    if kind == "caller":
        return lib.attn_varlen_fwd_ws(*args, ws.data_ptr(), ws.numel(), s)
    return lib.attn_varlen_fwd_noalloc(*args, s)


def _check(lib, kind, s, ws=None):
    if kind == "owned":
        return lib.attn_varlen_check(s)
    if kind == "caller":
        return lib.attn_varlen_check_ws(ws.data_ptr(), s)
    return lib.attn_varlen_check_noalloc(s)


@pytest.mark.parametrize("kind", ["owned", "caller", "noalloc"])
def test_wait_runs_out_and_is_reported(waitlib, kind):
    import torch
    from variable_length_prefill_gb300._binding import ERR_DEVICE_TIMEOUT
    _, t, cu_q, cu_k, out, ref = _inputs()
    s = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda") if kind == "caller" else None
    # a normal call first: module loaded, result right, status clear
    assert _run(waitlib, kind, t, cu_q, cu_k, out, s, ws) == 0
    assert _check(waitlib, kind, s, ws) == 0
    assert_close(to_bits(out), ref, f"testhooks build, {kind} workspace")

    waitlib.attn_varlen_test_withhold(1)
    try:
        t0 = time.perf_counter()
        assert _run(waitlib, kind, t, cu_q, cu_k, out, s, ws) == 0
        assert _check(waitlib, kind, s, ws) == ERR_DEVICE_TIMEOUT
        elapsed = time.perf_counter() - t0
    finally:
        waitlib.attn_varlen_test_withhold(0)
    # a 50 ms wait, then a 50 ms drain of the withheld slot
    assert elapsed < 1.0, elapsed
    # the bit was read and cleared; the other workspaces never saw it
    assert _check(waitlib, kind, s, ws) == 0
    for other in ("owned", "noalloc"):
        if other != kind:
            assert _check(waitlib, other, s) == 0

    out.zero_()
    assert _run(waitlib, kind, t, cu_q, cu_k, out, s, ws) == 0
    assert _check(waitlib, kind, s, ws) == 0
    assert_close(to_bits(out), ref, f"testhooks build after a timeout, {kind} workspace")


def test_split_counters_recover_after_a_timeout(waitlib):
    """A call whose plan splits units along keys (the library's own
    workspace) and that times out in CTA 0 can leave the split region's row
    counters part-counted (a chunk CTA 0 claimed is never run).  The CTA that
    gave up marks them dirty, and the next call's plan zeroes them: that call
    must meet the parity bar on every row.  6000 tokens over 7 heads: 168
    units, the 16 of the second wave cut into 2 key chunks each."""
    import torch
    from variable_length_prefill_gb300._binding import ERR_DEVICE_TIMEOUT
    w = Workload("timeout_split", (6000,), 7, 72, seed=113)
    x = make_inputs(w)
    t, cu_q, cu_k = device_inputs(x, "cuda")
    out = torch.zeros_like(t["q"])
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    s = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    assert _run(waitlib, "owned", t, cu_q, cu_k, out, s) == 0
    assert _check(waitlib, "owned", s) == 0
    assert_close(to_bits(out), ref, "testhooks build, split units")
    waitlib.attn_varlen_test_withhold(1)
    try:
        assert _run(waitlib, "owned", t, cu_q, cu_k, out, s) == 0
        assert _check(waitlib, "owned", s) == ERR_DEVICE_TIMEOUT
    finally:
        waitlib.attn_varlen_test_withhold(0)
    for _ in range(2):
        out.zero_()
        assert _run(waitlib, "owned", t, cu_q, cu_k, out, s) == 0
        assert _check(waitlib, "owned", s) == 0
        assert_close(to_bits(out), ref, "testhooks build after a timeout, split units")


def test_product_library_has_no_test_hook(cuda_lib):
    """The withholding hook exists only in the test build."""
    assert not hasattr(cuda_lib.load(), "attn_varlen_test_withhold")
