"""Paged single-query decode (through the C ABI) against the CPU oracle,
element by element: the page's eight shapes, ragged and empty contexts,
shuffled physical blocks, every head size, grouped heads beyond one CTA's
share, a long context, and the bad-block-id check."""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close_values
from workloads import (PAGED_CONFIGS, PagedWorkload, bf16_bits_to_f64, f16_bits_to_f64,
                       make_paged_inputs)

pytestmark = pytest.mark.gpu


def _run(vlp, x, dtype):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    dev = {n: torch.from_numpy(x[n].view(np.int16)).view(tdt).cuda()
           for n in ("query", "k_cache", "v_cache")}
    tables = torch.from_numpy(x["block_tables"]).cuda()
    lens = torch.from_numpy(x["seq_lens"]).cuda()
    out = vlp.paged_attn_decode(dev["query"], dev["k_cache"], dev["v_cache"], tables, lens)
    vlp.check()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def _check(vlp, w):
    x = make_paged_inputs(w)
    got = _run(vlp, x, w.dtype)
    ref = oracle.paged_decode(x["query"], x["k_cache"], x["v_cache"], x["block_tables"],
                              x["seq_lens"], w.dtype)
    widen = f16_bits_to_f64 if w.dtype == "fp16" else bf16_bits_to_f64
    assert_close_values(widen(got), ref, w.name)
    return got


@pytest.mark.parametrize("name", sorted(PAGED_CONFIGS))
def test_page_shapes(cuda_lib, name):
    _check(cuda_lib, PAGED_CONFIGS[name])


EXTRA = [
    # ragged and empty contexts, shuffled blocks
    PagedWorkload("ragged_bf16", 7, 100, 8, 2, 128, seed=80, shuffle_blocks=True,
                  seq_lens=(0, 1, 15, 16, 17, 100, -2)),
    PagedWorkload("ragged_fp16", 5, 65, 12, 4, 128, dtype="fp16", seed=81, shuffle_blocks=True,
                  seq_lens=(65, 33, 1, 0, 48)),
    # every head size
    PagedWorkload("d64", 6, 200, 8, 8, 64, seed=82, shuffle_blocks=True),
    PagedWorkload("d256_fp16", 3, 300, 16, 4, 256, dtype="fp16", seed=83),
    # 16 query heads per KV head: two CTAs per (sequence, KV head)
    PagedWorkload("gqa16", 3, 150, 32, 2, 128, seed=84, shuffle_blocks=True),
    # a long context: each warp walks many blocks
    PagedWorkload("long_ctx", 2, 4100, 8, 1, 128, seed=85, shuffle_blocks=True),
    # Short tables (at most 8 blocks) with at least four pairs per SM run one
    # consumer warp per (sequence, KV head, head group) pair: ragged and empty
    # contexts, head groups of 4 and 2, fp16, head sizes 64 and 256
    PagedWorkload("wpp_ragged", 700, 100, 4, 1, 128, seed=87, shuffle_blocks=True,
                  seq_lens=tuple((i * 37) % 106 - 5 for i in range(700))),
    PagedWorkload("wpp_fp16_g2", 320, 128, 4, 2, 128, dtype="fp16", seed=88, shuffle_blocks=True),
    PagedWorkload("wpp_d64", 640, 33, 1, 1, 64, seed=89, shuffle_blocks=True,
                  seq_lens=tuple(33 - i % 34 for i in range(640))),
    PagedWorkload("wpp_d256", 160, 50, 8, 4, 256, seed=90, shuffle_blocks=True),
]


@pytest.mark.parametrize("w", EXTRA, ids=lambda w: w.name)
def test_extra_shapes(cuda_lib, w):
    _check(cuda_lib, w)


def test_deterministic(cuda_lib):
    w = PAGED_CONFIGS["P0"]
    x = make_paged_inputs(w)
    np.testing.assert_array_equal(_run(cuda_lib, x, w.dtype), _run(cuda_lib, x, w.dtype))


def test_bad_block_id_is_reported(cuda_lib):
    """A table entry outside [0, num_blocks) is not read; the check call
    reports it."""
    from variable_length_prefill_gb300 import AttnVarlenError
    w = PagedWorkload("bad", 2, 40, 4, 2, 128, seed=86)
    x = make_paged_inputs(w)
    x["block_tables"][1, 1] = w.num_blocks + 1000
    with pytest.raises(AttnVarlenError) as e:
        _run(cuda_lib, x, w.dtype)
    assert e.value.code == -11
    cuda_lib.check()  # the status word was cleared


def test_bad_block_id_warp_per_pair(cuda_lib):
    """The same check in the warp-per-pair form (short tables, many pairs):
    the bad block is skipped, every other row still matches the oracle."""
    from variable_length_prefill_gb300 import AttnVarlenError
    w = PagedWorkload("bad_wpp", 640, 40, 2, 2, 128, seed=91)
    x = make_paged_inputs(w)
    x["block_tables"][5, 1] = -7
    with pytest.raises(AttnVarlenError) as e:
        _run(cuda_lib, x, w.dtype)
    assert e.value.code == -11
    cuda_lib.check()
    ok = np.ones(w.num_seqs, dtype=bool)
    ok[5] = False
    x2 = {k: (v[ok] if k in ("query", "block_tables", "seq_lens") else v) for k, v in x.items()}
    got = _run(cuda_lib, x2, w.dtype)
    ref = oracle.paged_decode(x2["query"], x2["k_cache"], x2["v_cache"], x2["block_tables"],
                              x2["seq_lens"], w.dtype)
    assert_close_values(bf16_bits_to_f64(got), ref, w.name)
