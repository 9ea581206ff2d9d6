"""GPU parity of the channel-permutation entry points against the oracle
("Accelerating Sparse Deep Neural Networks", Sec. 4.1; "Channel Permutations
for N:M Sparsity", abstract).  Every quantity here is an integer (fixed-point
magnitudes, gains, slots), so every comparison is exact.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as W
from tests._helpers import bits16

pytestmark = pytest.mark.gpu

INT32_MIN = -(2 ** 31)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


def weights(rows, cols, seed, sigma=0.02):
    return W.normal_bf16(rows, cols, sigma, seed, device="cuda")


def start_perm(cols, seed):
    if seed is None:
        return torch.arange(cols, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(cols, generator=g).to(torch.int32).cuda()


def host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("rows,cols,sigma", [(1, 32, 0.02), (33, 64, 3.0), (300, 544, 1e-3),
                                             (4096, 128, 0.02)])
def test_shift(rows, cols, sigma):
    Wt = weights(rows, cols, rows + cols, sigma)
    got = int(mk.maskllm_perm_shift(Wt).item())
    assert got == orc.perm_shift(bits16(Wt))


def test_shift_special_values():
    Wt = torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")
    assert int(mk.maskllm_perm_shift(Wt).item()) == 0
    b = Wt.view(torch.int16)
    b[2, 7] = 3                       # 3 * 2^-133, subnormal
    assert int(mk.maskllm_perm_shift(Wt).item()) == orc.perm_shift(bits16(Wt))
    b[1, 9] = 0x7F80                  # +inf
    assert int(mk.maskllm_perm_shift(Wt).item()) == INT32_MIN
    b[1, 9] = -63                     # 0xFFC1: NaN
    assert int(mk.maskllm_perm_shift(Wt).item()) == INT32_MIN


@pytest.mark.parametrize("rows,cols,seed", [(37, 96, 1), (256, 1024, 2), (5, 32, None)])
def test_metric(rows, cols, seed):
    Wt = weights(rows, cols, 10 + rows)
    p = start_perm(cols, seed)
    shift = mk.maskllm_perm_shift(Wt)
    got = int(mk.maskllm_perm_metric(Wt, p, shift).item())
    want = orc.perm_metric_fixed(bits16(Wt), host(p), int(shift.item()))
    assert got == want


def test_permute_columns():
    rows, cols = 70, 352
    Wt = weights(rows, cols, 3)
    p = start_perm(cols, 4)
    out = mk.maskllm_permute_columns(Wt, p)
    assert np.array_equal(bits16(out), bits16(Wt)[:, host(p)])
    assert mk.maskllm_device_status() == 0
    # an entry out of range reads as +0 and is reported, nothing else changes
    bad = p.clone()
    bad[5] = cols + 3
    out = mk.maskllm_permute_columns(Wt, bad)
    got = bits16(out)
    assert (got[:, 5] == 0).all()
    keep = np.arange(cols) != 5
    assert np.array_equal(got[:, keep], bits16(Wt)[:, host(p)][:, keep])
    assert mk.maskllm_device_status() == 1     # MASKLLM_ERR_INVALID_ARG
    assert mk.maskllm_device_status() == 0


@pytest.mark.parametrize("rows,cols,seed", [(5, 32, 1), (33, 64, None), (40, 160, 2),
                                            (70, 288, 3)])
def test_swap_gains(rows, cols, seed):
    Wt = weights(rows, cols, 20 + cols)
    p = start_perm(cols, seed)
    gains, info, shift = mk.maskllm_perm_swap_gains(Wt, p)
    assert int(info.item()) == 0
    k = int(shift.item())
    assert k == orc.perm_shift(bits16(Wt))
    want = orc.perm_swap_gains(bits16(Wt), host(p), k)
    assert np.array_equal(host(gains), want)


def test_swap_gains_bad_inputs():
    Wt = weights(8, 64, 5)
    p = start_perm(64, 6)
    dup = p.clone()
    dup[3] = dup[4]
    _, info, _ = mk.maskllm_perm_swap_gains(Wt, dup)
    assert int(info.item()) == mk.PERM_BAD_PERMUTATION
    neg = p.clone()
    neg[0] = -1
    _, info, _ = mk.maskllm_perm_swap_gains(Wt, neg)
    assert int(info.item()) == mk.PERM_BAD_PERMUTATION
    Wn = Wt.clone()
    Wn.view(torch.int16)[2, 2] = 0x7F80
    _, info, _ = mk.maskllm_perm_swap_gains(Wn, p)
    assert int(info.item()) == mk.PERM_NONFINITE


def run_search(Wt, p, max_swaps):
    n, swaps, gains, shift = mk.maskllm_perm_search(Wt, p, max_swaps)
    n = int(n.item())
    return n, host(swaps)[:max(n, 0)], host(gains)[:max(n, 0)], int(shift.item())


@pytest.mark.parametrize("rows,cols,seed,max_swaps", [(24, 64, 7, 500), (16, 128, None, 500),
                                                      (33, 96, 8, 500), (24, 64, 7, 5),
                                                      (48, 192, 9, 12)])
def test_search_matches_oracle_exactly(rows, cols, seed, max_swaps):
    Wt = weights(rows, cols, 30 + rows + cols)
    p = start_perm(cols, seed)
    p0 = host(p).copy()
    n, swaps, gains, k = run_search(Wt, p, max_swaps)
    want_p, want_s, want_g = orc.perm_search(bits16(Wt), p0, orc.perm_shift(bits16(Wt)), max_swaps)
    assert k == orc.perm_shift(bits16(Wt))
    assert n == len(want_s)
    assert np.array_equal(swaps, want_s)
    assert np.array_equal(gains, want_g)
    assert np.array_equal(host(p), want_p)


def test_search_tie_rule_and_stop():
    # four equal weights in group 0, zeros elsewhere: the first pair wins each
    # step, two swaps, then nothing gains
    Wt = torch.zeros((1, 32), dtype=torch.bfloat16, device="cuda")
    Wt[0, :4] = 8.0
    p = start_perm(32, None)
    n, swaps, gains, k = run_search(Wt, p, 10)
    assert n == 2
    assert swaps.tolist() == [[0, 4], [1, 5]]
    assert gains.tolist() == [8 << k, 8 << k]
    assert host(p)[:8].tolist() == [4, 5, 2, 3, 0, 1, 6, 7]


def test_search_edge_cases():
    Wt = weights(12, 64, 40)
    p = start_perm(64, 41)
    p0 = p.clone()
    n, _, _, _ = run_search(Wt, p, 0)
    assert n == 0 and torch.equal(p, p0)
    dup = p0.clone()
    dup[1] = dup[0]
    n, _, _, _ = run_search(Wt, dup, 10)
    assert n == mk.PERM_BAD_PERMUTATION
    Wn = Wt.clone()
    Wn.view(torch.int16)[0, 0] = -63      # NaN
    q = p0.clone()
    n, _, _, _ = run_search(Wn, q, 10)
    assert n == mk.PERM_NONFINITE and torch.equal(q, p0)
    # all-zero weights: nothing to gain
    z = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    n, _, _, k = run_search(z, p0.clone(), 10)
    assert n == 0 and k == 0


@pytest.mark.slow
def test_search_full_size_q_proj():
    """The q projection of the LLaMA-2-7B block (4096 x 4096): 64 steps; every
    logged gain is the oracle's gain of that swap in that state, the metric
    moves by their sum, and sampled entries of the gain table are exact."""
    wl = W.WORKLOADS["llama2_7b_block"]
    Wt = W.matrix_inputs(wl, 0, 0, device="cuda", with_grad=False).W
    Wb = bits16(Wt)
    cols = Wt.shape[1]
    p = start_perm(cols, None)
    gains_t, info, shift = mk.maskllm_perm_swap_gains(Wt, p)
    k = int(shift.item())
    assert int(info.item()) == 0 and k == orc.perm_shift(Wb)
    rng = np.random.default_rng(0)
    ident = np.arange(cols, dtype=np.int32)
    table = host(gains_t)
    for a, b in rng.integers(0, cols, (64, 2)):
        assert table[a, b] == orc.perm_swap_gain(Wb, ident, k, int(a), int(b))
    # the search's first swap is the table's best pair (first one on ties)
    upper = np.triu(table, 1)
    best = upper.max()
    first = np.argwhere(upper == best)[0]
    del gains_t, table, upper
    n, swaps, gains, k2 = run_search(Wt, p, 64)
    assert k2 == k and n == 64
    assert swaps[0].tolist() == first.tolist() and gains[0] == best
    cur = ident.copy()
    for (a, b), g in zip(swaps, gains):
        assert a < b and a // 4 != b // 4 and g > 0
        assert g == orc.perm_swap_gain(Wb, cur, k, int(a), int(b))
        cur[a], cur[b] = cur[b], cur[a]
    assert np.array_equal(host(p), cur)
    assert (orc.perm_metric_fixed(Wb, cur, k) - orc.perm_metric_fixed(Wb, ident, k)
            == int(gains.sum()))


def test_search_steps_are_the_best_of_fresh_gain_tables():
    """A longer search (each slot's list of best swaps is carried from step to
    step): every step's swap is the best pair of a gain table computed from
    scratch for that step's permutation (the tables themselves match the
    oracle above)."""
    rows, cols, steps = 200, 512, 120
    Wt = weights(rows, cols, 77)
    p = start_perm(cols, 78)
    cur = p.clone()
    n, swaps, gains, _ = run_search(Wt, p, steps)
    assert n == steps
    upper = np.triu(np.ones((cols, cols), bool), 1)
    for (a, b), g in zip(swaps, gains):
        table, info, _ = mk.maskllm_perm_swap_gains(Wt, cur)
        t = np.where(upper, host(table), np.iinfo(np.int64).min)
        best = t.max()
        assert g == best > 0
        assert [a, b] == np.argwhere(t == best)[0].tolist()
        cur[a], cur[b] = cur[b].clone(), cur[a].clone()
    assert torch.equal(cur, p)
