"""The synthetic workloads against the page's shape table, and the metric's
FLOP count against the page's T_SOL column."""
import os

import numpy as np

from workloads import C1, C2, C3, C4, C5, CONFIGS, make_inputs, round_to_bf16_bits, \
    bf16_bits_to_f64, sample_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "shape_table_attention_forward.txt")


def _table():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            r, h, d, L, tsol, tprod, s = line.split()
            rows.append(dict(row=int(r), H=int(h), D=int(d), L=int(L),
                             tsol=float(tsol), tprod=float(tprod), s=float(s)))
    return rows


def test_configs_are_rows_of_the_shape_table():
    t = {r["row"]: r for r in _table()}
    for w, row in ((C1, 11), (C2, 4), (C3, 9), (C4, 8)):
        assert (w.num_heads, w.head_dim, w.seq_lens_q[0]) == (t[row]["H"], t[row]["D"], t[row]["L"])
    # the packed batch holds rows #11-#17 plus a length-1 and an empty sequence
    members = [t[r]["L"] for r in range(11, 18)]
    assert [x for x in C5.seq_lens_q if x > 1] == members
    assert 1 in C5.seq_lens_q and 0 in C5.seq_lens_q
    assert all(t[r]["H"] == C5.num_heads and t[r]["D"] == C5.head_dim for r in range(11, 18))
    assert C5.total_q == 31673


def test_flop_count_matches_page_speed_of_light():
    """T_SOL on the page is a pure compute bound: T_SOL / (4 L^2 H D) must be
    the same on every row (within the table's printed rounding), which fixes
    the metric's FLOP count at 4 L^2 H D with the true head_dim."""
    rates = []
    for r in _table():
        if r["tsol"] < 1.0:   # 0.00 and 0.38 us rows carry too few digits
            continue
        flops = 4.0 * r["L"] ** 2 * r["H"] * r["D"]
        rates.append(flops / (r["tsol"] * 1e-6))
    rates = np.array(rates)
    assert rates.max() / rates.min() < 1.01
    # with a padded head_dim of 80 the d=72 and d=128 rows would disagree
    padded = []
    for r in _table():
        if r["tsol"] < 1.0:
            continue
        dp = 80 if r["D"] == 72 else r["D"]
        padded.append(4.0 * r["L"] ** 2 * r["H"] * dp / (r["tsol"] * 1e-6))
    assert max(padded) / min(padded) > 1.05


def test_speedup_column_is_tsol_over_tprod():
    for r in _table():
        if r["tprod"] > 0 and r["tsol"] >= 1.0:
            assert abs(100.0 * r["tsol"] / r["tprod"] - r["s"]) < 0.15


def test_flops_method():
    assert C3.flops() == 4.0 * 16742 ** 2 * 32 * 128
    assert C5.flops() == 4.0 * sum(L * L for L in C5.seq_lens_q) * 4 * 72


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-40, 3.0e38],
                 dtype=np.float32)
    b = round_to_bf16_bits(x)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins;
    # 1+3*2^-8 ties between 1+2^-7 and 1+2^-6: the even one is 1+2^-6
    np.testing.assert_array_equal(bf16_bits_to_f64(b)[:4], [1.0, 1.0, 1.0 + 2 ** -6, -2.5])


def test_generator_is_seeded_and_shaped():
    a, b = make_inputs(C1), make_inputs(C1)
    for n in ("q", "k", "v"):
        assert a[n].shape == (276, 4, 72) and a[n].dtype == np.uint16
        np.testing.assert_array_equal(a[n], b[n])
    f = bf16_bits_to_f64(a["q"])
    assert abs(f.mean()) < 0.02 and abs(f.std() - 1.0) < 0.02
    np.testing.assert_array_equal(a["cu_q"], [0, 276])
    cu_q, cu_k = C5.cu_seqlens()
    np.testing.assert_array_equal(cu_q, [0, 1, 277, 877, 1889, 3913, 8013, 16197, 31673, 31673])
    np.testing.assert_array_equal(cu_q, cu_k)


def test_sample_rows_cover_only_live_tokens():
    rows = sample_rows(C5, 64)
    assert rows.shape == (64 * C5.num_heads, 2)
    cu, _ = C5.cu_seqlens()
    assert rows[:, 0].min() >= 0 and rows[:, 0].max() < cu[-1]
    for h in range(C5.num_heads):
        assert len(set(rows[rows[:, 1] == h, 0])) == 64
    assert set(CONFIGS) == {"C1", "C2", "C3", "C4", "C5"}
