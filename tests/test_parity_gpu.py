"""CUDA path (through the C ABI) against the CPU oracle, element by element on
seeded inputs: the five workloads, ragged tiles, varlen edge cases, and
properties that hold at any size."""
import numpy as np
import pytest

import oracle
from gpu_helpers import (abs_bits, assert_close, bf16_bound, check_full, check_rows,
                         check_sampled, device_inputs, run_cuda, to_bits)
from workloads import C1, C2, C3, C4, C5, Workload, make_inputs

pytestmark = pytest.mark.gpu

SMALL = [
    # (lens_q, lens_k or None, heads, head_dim)
    ((1,), None, 1, 72), ((1,), None, 1, 128),
    ((127,), None, 2, 72), ((128,), None, 2, 128), ((129,), None, 2, 72),
    ((255,), None, 2, 128), ((256,), None, 2, 72), ((257,), None, 2, 128),
    ((300,), None, 2, 72), ((513,), None, 2, 128), ((700,), None, 3, 72),
    ((5, 130, 0, 257, 1, 64), None, 3, 72), ((5, 130, 0, 257, 1, 64), None, 3, 128),
    ((100, 300, 7), (257, 64, 1000), 2, 72), ((100, 300, 7), (257, 64, 1000), 2, 128),
    ((10, 5, 3), (0, 7, 0), 2, 72),
    # one Q tile against many key tiles, two Q tiles against fewer key tiles
    # than score buffers: the score/P buffer rotation must not lap a barrier
    ((7,), (1000,), 2, 72), ((7,), (1000,), 2, 128), ((130,), (1000,), 1, 72),
    ((300, 1, 200), (64, 2000, 30), 2, 72), ((300, 1, 200), (64, 2000, 30), 2, 128),
    # key counts on both sides of the head_dim-72 key tile (112 keys) and its
    # multiples, with one and two Q tiles
    ((200,), (111,), 2, 72), ((200,), (112,), 2, 72), ((129,), (113,), 2, 72),
    ((300,), (224,), 1, 72), ((257,), (225,), 2, 72), ((112, 113, 224), None, 2, 72),
    # head_dim 64 (128-key tiles), 80 (112-key tiles) and 96 (96-key tiles)
    ((1,), None, 2, 64), ((200,), (127,), 2, 64), ((129,), (129,), 2, 64),
    ((5, 130, 0, 257, 1, 64), None, 3, 64), ((300,), (1000,), 2, 64),
    ((1,), None, 2, 80), ((200,), (111,), 2, 80), ((257,), (113,), 2, 80),
    ((5, 130, 0, 257, 1, 64), None, 3, 80), ((100, 300, 7), (257, 64, 1000), 2, 80),
    ((1,), None, 2, 96), ((200,), (95,), 2, 96), ((129,), (97,), 2, 96), ((300,), (193,), 1, 96),
    ((5, 130, 0, 257, 1, 64), None, 3, 96), ((100, 300, 7), (257, 64, 1000), 2, 96),
    # head_dim 256 (its own kernel: 64-key tiles, the two Q tiles of a unit in turn)
    ((1,), None, 2, 256), ((200,), (63,), 2, 256), ((129,), (65,), 2, 256),
    ((128,), (128,), 1, 256), ((256,), (192,), 2, 256), ((64,), (256,), 1, 256),
    ((300,), (1000,), 1, 256), ((5, 130, 0, 257, 1, 64), None, 3, 256),
    ((100, 300, 7), (257, 64, 1000), 2, 256), ((10, 5, 3), (0, 7, 0), 2, 256),
]


@pytest.mark.parametrize("lens_q,lens_k,H,D", SMALL)
def test_small_ragged_shapes(cuda_lib, lens_q, lens_k, H, D):
    w = Workload(f"small_{lens_q}_{lens_k}_{H}_{D}", lens_q, H, D, seed=100 + sum(lens_q) + D,
                 seq_lens_k=lens_k)
    check_full(cuda_lib, w)


def test_c1_all_rows(cuda_lib):
    check_full(cuda_lib, C1)


def test_c5_all_rows(cuda_lib):
    check_full(cuda_lib, C5)


def test_c2_all_rows(cuda_lib):
    """Every output row of C2 (130176 rows of 8136 keys; a few seconds of the
    oracle on the host cores)."""
    check_full(cuda_lib, C2)


def test_c3_all_rows(cuda_lib):
    """Every output row of C3 (535744 rows of 16742 keys; about two minutes of
    the oracle on 16 host cores)."""
    check_full(cuda_lib, C3)


@pytest.mark.parametrize("w,rows", [(C2, 512), (C3, 512), (C4, 512)], ids=lambda x: getattr(x, "name", str(x)))
def test_full_size_sampled_rows(cuda_lib, w, rows):
    check_sampled(cuda_lib, w, rows)


def test_lk_zero_gives_zero_rows(cuda_lib):
    w = Workload("lk0", (10, 5, 3), 2, 72, seed=41, seq_lens_k=(0, 7, 0))
    x = make_inputs(w)
    got = run_cuda(cuda_lib, x)
    assert (got[0:10] == 0).all() and (got[15:18] == 0).all()
    assert (got[10:15] != 0).any()


@pytest.mark.parametrize("D", [64, 72, 80, 96, 128, 256])
def test_rows_outside_sequences_untouched(cuda_lib, D):
    """cu_seqlens starting past row 0, an empty sequence, and rows after the
    last sequence: a sentinel pattern there must survive bit for bit (the
    epilogue's tiled stores end at each sequence's last row, for every box
    width: one 64-column box, an 8-column box B, a 64-column box B cut at
    head_dim)."""
    w = Workload(f"offsets_{D}", (40, 0, 200, 3), 2, D, seed=42, cu_offset=7)
    x = make_inputs(w)
    # two extra trailing rows beyond cu_q[-1]
    for n in ("q", "k", "v"):
        x[n] = np.concatenate([x[n], np.ones((2,) + x[n].shape[1:], np.uint16)])
    sentinel = 0x7FC1  # a NaN payload the kernel never produces
    got = run_cuda(cuda_lib, x, out_fill=sentinel)
    cu = x["cu_q"]
    assert (got[:cu[0]] == sentinel).all()
    assert (got[cu[-1]:] == sentinel).all()
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    assert_close(got[cu[0]:cu[-1]], ref[cu[0]:cu[-1]], f"offsets D={D}")


@pytest.mark.parametrize("D,causal,ws", [(72, False, False), (128, False, True),
                                         (72, True, False), (128, True, False)])
def test_backwards_cu_seqlens(cuda_lib, D, causal, ws):
    """cu_seqlens that step backwards, every offset inside the buffers.  Query
    slices [600, 900), [900, 750), [750, 0), [0, 300), [300, 540); key slices
    [0, 1500), [1500, 1200), [1200, 1800), [1800, 150), [150, 990).  The two
    backwards query slices are skipped, the backwards key slice of the fourth
    sequence gives zero rows, and rows 540-599 and 900-999 belong to no
    sequence: a sentinel there must survive bit for bit."""
    from workloads import round_to_bf16_bits
    rng = np.random.default_rng(48 + D)
    H = 2
    x = {"q": round_to_bf16_bits(rng.standard_normal((1000, H, D), dtype=np.float32)),
         "k": round_to_bf16_bits(rng.standard_normal((2000, H, D), dtype=np.float32)),
         "v": round_to_bf16_bits(rng.standard_normal((2000, H, D), dtype=np.float32)),
         "cu_q": np.array([600, 900, 750, 0, 300, 540], np.int32),
         "cu_k": np.array([0, 1500, 1200, 1800, 150, 990], np.int32)}
    sentinel = 0x7FC1
    if ws:
        got = run_cuda(cuda_lib, x, out_fill=sentinel, caller_workspace=True)
    else:
        got = run_cuda(cuda_lib, x, out_fill=sentinel, causal=causal)
    assert (got[540:600] == sentinel).all() and (got[900:] == sentinel).all()
    assert (got[0:300] == 0).all()
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal=causal)
    live = np.r_[300:540, 600:900]
    bound = None
    if causal:  # the first rows of a causal sequence average only a few values
        absv = oracle.attn_varlen(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"],
                                  causal=True)
        bound = bf16_bound(ref[live], absv[live])
    assert_close(got[live], ref[live], f"backwards cu_seqlens D={D} causal={causal}",
                 bound=bound)


@pytest.mark.parametrize("D,causal", [(72, False), (128, False), (64, True), (80, False),
                                     (96, True)])
def test_head_shards_in_place(cuda_lib, D, causal):
    """attn_varlen_fwd_heads on the shards of a 5-head batch: one shard
    leaves the other heads' rows untouched (a sentinel survives bit for bit),
    and the three shards of a 3-way split together meet the bar against the
    oracle on every head."""
    import torch
    from variable_length_prefill_gb300 import head_shard
    w = Workload(f"heads_{D}", (300, 1, 0, 700), 5, D, seed=95 + D, seq_lens_k=(300, 40, 3, 700))
    x = make_inputs(w)
    t, cu_q, cu_k = device_inputs(x, "cuda")
    sentinel = 0x7FC1
    out = torch.full(t["q"].shape, sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    b, c = head_shard(5, 1, 2)
    cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out, causal=causal,
                             heads=(b, c))
    cuda_lib.check()
    got = to_bits(out)
    live = np.zeros(got.shape[0], bool)
    cu = x["cu_q"]
    for i in range(len(cu) - 1):
        live[cu[i]:cu[i + 1]] = cu[i + 1] > cu[i]
    others = [h for h in range(5) if not b <= h < b + c]
    assert (got[:, others] == sentinel).all()
    assert (got[live][:, b:b + c] != sentinel).all()
    cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out, causal=causal,
                             heads=(2, 0))  # an empty range writes nothing
    for r in range(3):
        cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, out=out, causal=causal,
                                 heads=head_shard(5, r, 3))
    cuda_lib.check()
    got = to_bits(out)
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"], causal=causal)
    absv = oracle.attn_varlen(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"],
                              causal=causal)
    assert_close(got[live], ref[live], f"head shards D={D} causal={causal}",
                 bound=bf16_bound(ref[live], absv[live]))


def test_num_seqs_zero_is_a_noop(cuda_lib):
    import torch
    q = torch.zeros(4, 2, 72, dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    cuda_lib.attn_varlen_fwd(q, q, q, cu, cu, out=out)
    cuda_lib.check()
    assert (out == 3.0).all()


def test_packing_invariance_bitwise(cuda_lib):
    """The packed batch equals each member run alone, bit for bit (tiles
    start at sequence starts, so every row sees the same arithmetic).  Run
    with caller-owned workspaces, which never split a unit's key range: the
    library-owned workspace may split the units of the grid's last partial
    wave, and which units those are depends on the whole batch."""
    x = make_inputs(C5)
    packed = run_cuda(cuda_lib, x, caller_workspace=True)
    cu = x["cu_q"]
    for i in range(len(cu) - 1):
        if cu[i + 1] <= cu[i]:
            continue
        sl = slice(cu[i], cu[i + 1])
        alone = {"q": x["q"][sl], "k": x["k"][sl], "v": x["v"][sl],
                 "cu_q": np.array([0, cu[i + 1] - cu[i]], np.int32),
                 "cu_k": np.array([0, cu[i + 1] - cu[i]], np.int32)}
        np.testing.assert_array_equal(run_cuda(cuda_lib, alone, caller_workspace=True),
                                      packed[sl])


def test_deterministic(cuda_lib):
    x = make_inputs(C5)
    np.testing.assert_array_equal(run_cuda(cuda_lib, x), run_cuda(cuda_lib, x))


def test_many_short_sequences(cuda_lib):
    """300 sequences (some empty) plus one long one: longest-first order and
    the unit search over many sequences."""
    rng = np.random.default_rng(43)
    lens = tuple(int(v) for v in rng.integers(0, 5, 300)) + (1500,)
    check_full(cuda_lib, Workload("many_short", lens, 2, 72, seed=44), short_sequences=True)


def test_more_sequences_than_sorted_limit(cuda_lib):
    """Beyond the longest-first limit the natural order is used."""
    rng = np.random.default_rng(45)
    lens = tuple(int(v) for v in rng.integers(0, 4, 2500))
    check_full(cuda_lib, Workload("very_many", lens, 1, 128, seed=46), short_sequences=True)


def _scale_keys(x, scale_of_key):
    """k rows times a per-key factor, rounded back to bf16 (test input only)."""
    from workloads import bf16_bits_to_f64, round_to_bf16_bits
    cu = x["cu_k"]
    k = bf16_bits_to_f64(x["k"])
    for i in range(len(cu) - 1):
        for j in range(cu[i + 1] - cu[i]):
            k[cu[i] + j] *= scale_of_key(j)
    x["k"] = round_to_bf16_bits(k.astype(np.float32))
    return x


@pytest.mark.parametrize("D", [72, 128, 256])
def test_running_max_rises_every_tile(cuda_lib, D):
    """Key norms step up every 128 keys, so a row's running max rises by more
    than the rescale threshold at tile starts: the O/l rescale runs."""
    w = Workload(f"rising_tiles_{D}", (700, 300), 2, D, seed=51)
    x = _scale_keys(make_inputs(w), lambda j: 1.0 + 2.5 * (j // 128))
    check_full(cuda_lib, w, x=x, short_sequences=True)


@pytest.mark.parametrize("D", [72, 128, 256])
def test_running_max_rises_in_second_half(cuda_lib, D):
    """Only the second 64 keys of each tile step up, so the first half's P is
    computed against the old max and must be rescaled with O and l."""
    w = Workload(f"rising_halves_{D}", (640, 200), 2, D, seed=52)
    x = _scale_keys(make_inputs(w), lambda j: 1.0 + 3.0 * (j // 128) + (2.5 if j % 128 >= 64 else 0.0))
    check_full(cuda_lib, w, x=x, short_sequences=True)


@pytest.mark.parametrize("D", [72, 128, 256])
def test_running_max_huge_jump(cuda_lib, D):
    """A jump far beyond the exp2 range of the old max (scores x60 from key
    300 on): no overflow leaks into the result."""
    w = Workload(f"huge_jump_{D}", (520,), 2, D, seed=53)
    x = _scale_keys(make_inputs(w), lambda j: 60.0 if j >= 300 else 1.0)
    check_full(cuda_lib, w, x=x, short_sequences=True)


def test_caller_workspace_on_two_streams(cuda_lib):
    """Two calls with their own workspaces on two streams agree bit for bit
    with a single caller-workspace call (the default entry point may split C1's
    units along keys, so it is compared with the oracle elsewhere)."""
    import torch
    x = make_inputs(C1)
    want = run_cuda(cuda_lib, x, caller_workspace=True)
    t, cu_q, cu_k = device_inputs(x, "cuda")
    outs = []
    for _ in range(2):
        s = torch.cuda.Stream()
        ws = torch.zeros(cuda_lib.workspace_size(1), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(s):
            out = cuda_lib.attn_varlen_fwd(t["q"], t["k"], t["v"], cu_q, cu_k, workspace=ws)
        outs.append((s, ws, out))
    for s, ws, out in outs:
        cuda_lib.check(stream=s, workspace=ws)
        np.testing.assert_array_equal(to_bits(out), want)


def test_errors_raise(cuda_lib):
    import torch
    from variable_length_prefill_gb300 import AttnVarlenError
    q = torch.zeros(8, 2, 48, dtype=torch.bfloat16, device="cuda")  # head_dim 48: not built
    cu = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    with pytest.raises(AttnVarlenError) as e:
        cuda_lib.attn_varlen_fwd(q, q, q, cu, cu)
    assert e.value.code == -2


def _tail_rows(w, extra_per_head=48, seed=11):
    """The last 8 query rows of every head plus a seeded sample."""
    cu_q, _ = w.cu_seqlens()
    end = int(cu_q[-1])
    rng = np.random.default_rng(seed)
    rows = []
    for h in range(w.num_heads):
        last = np.arange(max(int(cu_q[0]), end - 8), end)
        pick = rng.choice(np.arange(int(cu_q[0]), end), size=extra_per_head, replace=False)
        toks = np.unique(np.concatenate([last, pick]))
        rows.append(np.stack([toks, np.full(toks.size, h)], axis=1))
    return np.concatenate(rows).astype(np.int64)


@pytest.mark.parametrize("D", [72, 128])
def test_tail_split_one_unit_over_the_grid(cuda_lib, D):
    """152 full units plus one more: on a 152-SM GB300 the last unit (7
    query rows against all 38919 keys) is cut into many key chunks whose
    partials are merged; the caller-workspace path computes it whole."""
    w = Workload(f"tail_153_units_D{D}", (152 * 256 + 7,), 1, D, seed=31 + D)
    rows = _tail_rows(w)
    x = make_inputs(w)
    # both meet the bar against the oracle; they may differ in the last bits
    # where the fp32 sums were taken in another order
    check_rows(cuda_lib, w, rows, x=x)
    check_rows(cuda_lib, w, rows, x=x, caller_workspace=True)


@pytest.mark.parametrize("D", [72, 128])
def test_tail_split_equal_tail_units(cuda_lib, D):
    """One sequence of 10000 tokens over 5 heads: 200 units, so on a 152-SM
    GB300 the second wave's 48 units (equal key ranges) are the late ones and
    are each cut into floor(152 / 48) = 3 key chunks (the plan's closed-form
    budget for a short tail of equal units) and merged.  Every row against
    the oracle."""
    w = Workload(f"tail_equal_D{D}", (10000,), 5, D, seed=41 + D)
    check_full(cuda_lib, w)


def test_tail_split_mixed_batch(cuda_lib):
    """Fewer units than SMs, so every unit is late in the plan's schedule:
    units of 81, 54, 45, 19, 1 and 0 key tiles (head_dim 72) are cut into 3,
    2, 2 and 1 chunks of at most 32 key tiles.  Every row against the oracle,
    through both entry points."""
    lens_q = (3000, 1, 700, 0, 2048, 5, 300)
    lens_k = (6000, 9000, 0, 9, 2048, 5000, 1)
    w = Workload("tail_mixed", lens_q, 2, 72, seed=77, seq_lens_k=lens_k)
    x = make_inputs(w)
    check_full(cuda_lib, w, x=x, short_sequences=True)
    got = run_cuda(cuda_lib, x, caller_workspace=True)
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["cu_q"], x["cu_k"])
    live = np.zeros(got.shape[0], bool)
    cu = x["cu_q"]
    for i in range(len(cu) - 1):
        live[cu[i]:cu[i + 1]] = True
    absv = oracle.attn_varlen(x["q"], x["k"], abs_bits(x["v"]), x["cu_q"], x["cu_k"])
    assert_close(got[live], ref[live], "tail_mixed caller workspace",
                 bound=bf16_bound(ref[live], absv[live]))


@pytest.mark.parametrize("D", [64, 80, 96, 256])
def test_other_head_dims_sampled(cuda_lib, D):
    """A longer sequence at every extra head_dim: 512 rows per head."""
    w = Workload(f"L4500_H8_D{D}", (4500,), 8, D, seed=50 + D)
    check_sampled(cuda_lib, w, 512)


# ------------------------------------------------------------------ causal
CAUSAL = [
    # (lens_q, lens_k or None, heads, head_dim): L_q = L_k across tile and
    # unit boundaries, L_q < L_k (a cached prefix), L_q > L_k (leading rows
    # that see no key), L_k = 0, every head_dim
    ((1,), None, 2, 72), ((127,), None, 2, 72), ((129,), None, 2, 128), ((300,), None, 2, 72),
    ((513,), None, 2, 128), ((700,), None, 3, 64), ((5, 130, 0, 257, 1, 64), None, 3, 72),
    ((100, 7), (257, 1000), 2, 72), ((300,), (1000,), 2, 128), ((300,), (100,), 2, 72),
    ((257,), (5,), 2, 128), ((400, 3), (0, 3), 2, 72), ((300,), None, 2, 96),
    ((200, 31), (250, 600), 2, 80), ((640,), (113,), 1, 72), ((129,), (1,), 2, 64),
    ((300,), None, 2, 256), ((100, 7), (257, 1000), 2, 256), ((300,), (100,), 2, 256),
]


@pytest.mark.parametrize("lens_q,lens_k,H,D", CAUSAL)
def test_causal_ragged_shapes(cuda_lib, lens_q, lens_k, H, D):
    w = Workload(f"causal_{lens_q}_{lens_k}_{H}_{D}", lens_q, H, D,
                 seed=300 + sum(lens_q) + D, seq_lens_k=lens_k)
    check_full(cuda_lib, w, short_sequences=True, causal=True)


@pytest.mark.parametrize("w", [C2, C3, C5], ids=lambda w: w.name)
def test_causal_workloads_sampled(cuda_lib, w):
    """The page's workloads under the causal mask: 256 seeded rows per head."""
    check_sampled(cuda_lib, w, 256, causal=True)


def test_causal_deterministic(cuda_lib):
    x = make_inputs(C5)
    a = run_cuda(cuda_lib, x, causal=True)
    b = run_cuda(cuda_lib, x, causal=True)
    np.testing.assert_array_equal(a, b)


def test_causal_last_row_equals_non_causal(cuda_lib):
    """The bottom-right-aligned mask hides nothing from a sequence's last row."""
    x = make_inputs(C1)
    a = run_cuda(cuda_lib, x, causal=True)
    b = run_cuda(cuda_lib, x)
    last = int(x["cu_q"][-1]) - 1
    np.testing.assert_array_equal(a[last], b[last])
