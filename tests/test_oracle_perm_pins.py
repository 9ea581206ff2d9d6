"""Pins of the oracle's channel-permutation search ("Channel Permutations for
N:M Sparsity", abstract; "Accelerating Sparse Deep Neural Networks",
Sec. 4.1) to facts outside the oracle: hand-computed metrics, invariances of
the metric, the magnitude pruning of the mask layer's own pinned functions,
the fixed-point bounds, brute force over swaps and over all partitions of
small matrices.  CPU only.
"""
import itertools

import numpy as np
import pytest

import oracle as orc


def bf16(x):
    """float array -> bf16 bit patterns (round to nearest even), via the
    oracle's pinned single-rounding conversion."""
    x = np.asarray(x, np.float64)
    return np.array([orc.double_to_bf16(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)


def rand_w(rows, cols, seed, sigma=0.02):
    rng = np.random.default_rng(seed)
    return bf16(rng.normal(0.0, sigma, (rows, cols)))


def swapped(perm, a, b):
    p = np.array(perm, np.int32)
    p[a], p[b] = p[b], p[a]
    return p


HAND = bf16([[0.5, -1.0, 0.25, 2.0, 3.0, 0.0, -0.125, 1.0]])


def test_metric_hand_case():
    # kept: group (0.5, -1, 0.25, 2) -> 2 + 1; group (3, 0, -0.125, 1) -> 3 + 1
    ident = np.arange(8, dtype=np.int32)
    assert orc.perm_metric(HAND, ident) == 7.0
    assert orc.perm_shift(HAND) == 30           # 1 row, max 3: 31 - 0 - 1
    assert orc.perm_metric_fixed(HAND, ident, 30) == 7 << 30
    # channels 3 and 4 exchanged: (0.5, -1, 0.25, 3) -> 4; (2, 0, -0.125, 1) -> 3
    assert orc.perm_metric(HAND, [0, 1, 2, 4, 3, 5, 6, 7]) == 7.0
    # (2, 3, 0.5, -1) -> 5; (0.25, 0, -0.125, 1) -> 1.25
    assert orc.perm_metric(HAND, [3, 4, 0, 1, 2, 5, 6, 7]) == 6.25
    assert orc.perm_metric_fixed(HAND, [3, 4, 0, 1, 2, 5, 6, 7], 30) == 25 << 28


def test_metric_invariances_and_magnitude_pruning():
    rows, cols = 8, 64
    W = rand_w(rows, cols, 1)
    rng = np.random.default_rng(2)
    perm = rng.permutation(cols).astype(np.int32)
    k = orc.perm_shift(W)
    m, mq = orc.perm_metric(W, perm), orc.perm_metric_fixed(W, perm, k)
    # reordering slots inside each group, or whole groups, keeps the metric
    inner = perm.reshape(-1, 4)[:, rng.permutation(4)].ravel()
    blocks = perm.reshape(-1, 4)[rng.permutation(cols // 4)].ravel()
    for p in (inner, blocks):
        assert orc.perm_metric(W, p) == m
        assert orc.perm_metric_fixed(W, p, k) == mq
    # identity metric = the magnitude that the mask layer's magnitude prior +
    # hard mask keep (the two largest of four, "Accelerating Sparse Deep
    # Neural Networks" Sec. 4.1)
    L = orc.prior_init(W, 1.0)
    vals, _, _ = orc.hard_compress(W, L)
    kept = np.abs(orc.bf16_to_f64(vals)).sum()
    assert orc.perm_metric(W, np.arange(cols, dtype=np.int32)) == pytest.approx(kept, rel=1e-15)


@pytest.mark.parametrize("sigma", [1e-3, 0.02, 3.0, 1e3])
@pytest.mark.parametrize("rows", [1, 7, 64, 100])
def test_shift_keeps_column_sums_in_32_bits(sigma, rows):
    W = rand_w(rows, 32, rows, sigma)
    k = orc.perm_shift(W)
    qmax = max(orc.perm_fixed(int(w), k) for w in W.ravel())
    assert rows * qmax < 2 ** 32
    assert rows * qmax >= 2 ** 30        # and wastes at most two bits


def test_shift_special_cases():
    assert orc.perm_shift(np.zeros((4, 32), np.uint16)) == 0
    W = np.zeros((2, 32), np.uint16)
    W[1, 5] = 0x7F80                      # +inf
    assert orc.perm_shift(W) == orc.PERM_NONFINITE
    W[1, 5] = 0xFFC1                      # NaN
    assert orc.perm_shift(W) == orc.PERM_NONFINITE
    W[1, 5] = 0x0003                      # largest magnitude 3 * 2^-133 (subnormal)
    k = orc.perm_shift(W)
    assert k == 31 - 1 - (-132)
    assert orc.perm_fixed(0x0003, k) == 3 << 29   # 3 * 2^(162 - 133)


def test_fixed_point_is_truncation():
    assert orc.perm_fixed(bf16(1.5), 1) == 3
    assert orc.perm_fixed(bf16(-1.5), 1) == 3
    assert orc.perm_fixed(bf16(0.75), 0) == 0
    assert orc.perm_fixed(bf16(1.75), 0) == 1
    assert orc.perm_fixed(0x0001, 133) == 1     # 2^-133
    assert orc.perm_fixed(0x0001, 132) == 0


def test_fixed_metric_bounds_the_exact_metric():
    rows, cols = 16, 96
    W = rand_w(rows, cols, 3)
    perm = np.random.default_rng(4).permutation(cols).astype(np.int32)
    k = orc.perm_shift(W)
    exact = orc.perm_metric(W, perm) * 2.0 ** k
    fixed = orc.perm_metric_fixed(W, perm, k)
    assert 0 <= exact - fixed < rows * cols // 2     # one truncation per kept value
    # values on the fixed-point grid: no truncation at all
    Wi = bf16(np.random.default_rng(5).integers(-200, 200, (rows, cols)))
    ki = orc.perm_shift(Wi)
    assert orc.perm_metric_fixed(Wi, perm, ki) == int(orc.perm_metric(Wi, perm)) << ki


def test_swap_gain_is_the_metric_difference():
    rows, cols = 6, 32
    W = rand_w(rows, cols, 6)
    perm = np.random.default_rng(7).permutation(cols).astype(np.int32)
    k = orc.perm_shift(W)
    base = orc.perm_metric_fixed(W, perm, k)
    for a in range(cols):
        for b in range(cols):
            want = orc.perm_metric_fixed(W, swapped(perm, a, b), k) - base
            assert orc.perm_swap_gain(W, perm, k, a, b) == want
            if a // 4 == b // 4:
                assert want == 0


def test_search_is_steepest_ascent_to_a_local_optimum():
    rows, cols = 8, 32
    W = rand_w(rows, cols, 8)
    start = np.random.default_rng(9).permutation(cols).astype(np.int32)
    k = orc.perm_shift(W)
    final, swaps, gains = orc.perm_search(W, start, k, 1000)
    assert sorted(final) == list(range(cols))
    assert len(swaps) > 0
    cur = start.copy()
    for (a, b), g in zip(swaps, gains):
        base = orc.perm_metric_fixed(W, cur, k)
        every = {(x, y): orc.perm_metric_fixed(W, swapped(cur, x, y), k) - base
                 for x in range(cols) for y in range(x + 1, cols)}
        best = max(every.values())
        assert g == best > 0
        assert (a, b) == min(p for p, v in every.items() if v == best)
        cur = swapped(cur, a, b)
    assert np.array_equal(cur, final)
    base = orc.perm_metric_fixed(W, final, k)
    assert all(orc.perm_metric_fixed(W, swapped(final, x, y), k) <= base
               for x in range(cols) for y in range(x + 1, cols))
    assert base - orc.perm_metric_fixed(W, start, k) == int(gains.sum())
    assert orc.perm_metric(W, final) > orc.perm_metric(W, start)


def test_search_tie_rule_hand_case():
    # four equal weights in one group, zeros in the other: every cross swap
    # gains 8; the first pair wins each time, and two swaps reach 8+8 / 8+8
    W = bf16([[8.0, 8.0, 8.0, 8.0, 0.0, 0.0, 0.0, 0.0]])
    k = orc.perm_shift(W)
    final, swaps, gains = orc.perm_search(W, np.arange(8, dtype=np.int32), k, 10)
    assert swaps.tolist() == [[0, 4], [1, 5]]
    assert gains.tolist() == [8 << k, 8 << k]
    assert final.tolist() == [4, 5, 2, 3, 0, 1, 6, 7]
    assert orc.perm_metric(W, final) == 32.0


def test_search_respects_max_swaps():
    W = rand_w(4, 32, 10)
    k = orc.perm_shift(W)
    start = np.random.default_rng(11).permutation(32).astype(np.int32)
    _, s0, _ = orc.perm_search(W, start, k, 0)
    p1, s1, g1 = orc.perm_search(W, start, k, 1)
    _, s5, g5 = orc.perm_search(W, start, k, 5)
    assert len(s0) == 0 and len(s1) == 1
    assert s5[:1].tolist() == s1.tolist() and g5[0] == g1[0]
    assert np.array_equal(p1, swapped(start, *s1[0]))


def test_search_against_every_partition_of_eight_channels():
    # two groups of four: 35 distinct partitions; the search ends no higher
    # than the best of them and at a partition no single swap improves
    for seed in range(5):
        W = rand_w(4, 8, 20 + seed)
        k = orc.perm_shift(W)
        ident = np.arange(8, dtype=np.int32)
        best = max(orc.perm_metric_fixed(W, list(g) + [c for c in range(8) if c not in g], k)
                   for g in itertools.combinations(range(8), 4))
        final, _, _ = orc.perm_search(W, ident, k, 100)
        got = orc.perm_metric_fixed(W, final, k)
        assert orc.perm_metric_fixed(W, ident, k) <= got <= best
        assert all(orc.perm_swap_gain(W, final, k, a, b) <= 0
                   for a in range(4) for b in range(4, 8))
