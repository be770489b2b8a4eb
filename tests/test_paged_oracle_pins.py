"""The paged-decode oracle against the dense oracle, torch's float64 SDPA with
grouped KV heads, layout invariants and closed forms; each planted mistake
caught by at least one pin."""
import pytest

from paged_pins import PAGED_PINS
from workloads import PAGED_CONFIGS, make_paged_inputs


@pytest.mark.parametrize("pin", PAGED_PINS, ids=lambda p: p.__name__)
def test_paged_pin(pin):
    pin(0)


# 20 query head h read KV head h % Hkv instead of h / (Hq / Hkv)
# 21 token t read at flat index t, ignoring the block table
# 22 keys read in the value cache's [D][block_size] layout
# 23 fp16 caches decoded as bf16
PAGED_MUTATIONS = [20, 21, 22, 23]


@pytest.mark.parametrize("mutation", PAGED_MUTATIONS)
def test_paged_planted_mistake_is_caught(mutation):
    failed = []
    for pin in PAGED_PINS:
        try:
            pin(mutation)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches planted mistake {mutation}"


def test_paged_shapes_follow_the_page():
    """The page's input generator: identity block tables, num_blocks =
    max_blocks * num_seqs + 16, x = 8 elements of 2 bytes."""
    for w in PAGED_CONFIGS.values():
        x = make_paged_inputs(w)
        assert x["k_cache"].shape == (w.max_blocks * w.num_seqs + 16, w.num_kv_heads,
                                      w.head_size // 8, w.block_size, 8)
        assert x["v_cache"].shape == (w.num_blocks, w.num_kv_heads, w.head_size, w.block_size)
        assert (x["block_tables"][:, 0] == [i * w.max_blocks for i in range(w.num_seqs)]).all()
