"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something the pages, the mathematics or an
independent library fix: printed numbers (golden fixtures), closed forms,
invariants, textbook identities, brute force on tiny inputs, finite
differences, and a library implementation of the same RNG.
"""
import ctypes
import itertools
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EULER_GAMMA = 0.57721566490153286061


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# Candidates and the metadata codes
# --------------------------------------------------------------------------

def test_candidates_match_golden_and_enumeration(orc):
    rows = _golden_rows("candidates.txt")
    pairs = orc.candidate_pairs()
    assert pairs == [(int(r[1]), int(r[2])) for r in rows]
    # lexicographic enumeration of the 2-subsets of {0,1,2,3}
    assert pairs == list(itertools.combinations(range(4), 2))
    lib = orc.lib()
    for c, r in enumerate(rows):
        keeps = [lib.orc_candidate_keeps(c, j) for j in range(4)]
        assert "".join(str(k) for k in keeps) == r[3]
        assert sum(keeps) == 2   # 2:4 -- two kept, at least two zeros of four
        i, j = pairs[c]
        assert i | (j << 2) == int(r[4], 16)


# --------------------------------------------------------------------------
# Philox4x32-10 against cuRAND's host implementation of the same generator
# --------------------------------------------------------------------------

def _curand():
    for name in ("libcurand.so.10", "libcurand.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def _curand_host_philox(cur, seed, n, offset):
    gen = ctypes.c_void_p()
    assert cur.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
    try:
        assert cur.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert cur.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        buf = (ctypes.c_uint * n)()
        assert cur.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
        return np.frombuffer(buf, dtype=np.uint32).copy().reshape(-1, 4)
    finally:
        cur.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF, 20240917])
def test_philox_matches_curand_host_generator(orc, seed):
    """cuRAND's host Philox4x32-10 stream, default ordering, lays its output out
    in blocks of 4 words: block b is the bijection at counter
    (x0 + b // 65536, y0, b % 65536, 0), where the generator offset (in words)
    sets x0 + 2^32 y0 = offset / (4 * 65536).  Our noise words of group
    x + 2^32 y at step z and tensor id 0 must equal that block."""
    cur = _curand()
    if cur is None:
        pytest.skip("libcurand not available")
    S = 65536
    for base in (0, 7, (5 << 32) + 11):
        blocks = _curand_host_philox(cur, seed, 4 * 2 * S, offset=4 * S * base)
        for b in list(range(0, 2 * S, 977)) + [S - 1, S, 2 * S - 1]:
            group = base + b // S
            step = b % S
            mine = orc.noise_words(seed, step, 0, group, 1)[0]
            assert (mine == blocks[b]).all(), (seed, base, b)


def test_noise_words_are_the_bijection_at_the_group_counter(orc):
    seed, step, tid = 0xDEADBEEFCAFEF00D, 17, 1234
    g0 = (3 << 32) + 5
    words = orc.noise_words(seed, step, tid, g0, 4)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for i in range(4):
        g = g0 + i
        ctr = np.array([g & 0xFFFFFFFF, g >> 32, step, tid], np.uint32)
        assert (orc.philox4x32_10(key, ctr) == words[i]).all()
    # distinct steps and tensor ids give unrelated words
    a = orc.noise_words(seed, 0, 0, 0, 64)
    b = orc.noise_words(seed, 1, 0, 0, 64)
    c = orc.noise_words(seed, 0, 1, 0, 64)
    assert (a != b).mean() > 0.99 and (a != c).mean() > 0.99


def test_philox_bits_are_balanced(orc):
    w = orc.noise_words(7, 0, 0, 0, 1 << 15)
    bits = np.unpackbits(w.view(np.uint8))
    n = bits.size
    assert abs(bits.mean() - 0.5) < 5.0 * 0.5 / math.sqrt(n)


# --------------------------------------------------------------------------
# Gumbel noise
# --------------------------------------------------------------------------

def test_gumbel_cell_hand_case(orc):
    words = np.array([0x89ABCDEF, 0x01234567, 0xFEDCBA98, 0x76543210], np.uint32)
    expect = [0x337B, 0x226A, 0x1159, 0x0048, 0x2EA6, 0x3FB7]
    assert [orc.gumbel_cell(words, c) for c in range(6)] == expect


def test_gumbel_table_moments_and_shape(orc):
    T = orc.gumbel_table().astype(np.float64)
    assert T.size == 1 << 14
    assert np.all(np.diff(T) > 0)                  # a quantile function is increasing
    # Gumbel(0,1): mean = Euler's gamma, variance = pi^2/6.  The table is the
    # midpoint rule over 2^14 cells; its error sits in the two end cells where
    # the quantile is logarithmic: about 2e-5 on the mean and 5e-4 on the
    # variance, so these bounds leave a factor of a few.
    assert abs(T.mean() - EULER_GAMMA) < 1e-4
    assert abs(T.var() - math.pi ** 2 / 6) < 3e-3
    # the quantile at u = 1/e is exactly 0; the cell holding 1/e is within one
    # cell width times the slope (e) of zero
    i = int(math.floor((1 / math.e) * (1 << 14)))
    assert abs(T[i]) <= math.e / (1 << 14)
    # support of the quantised noise
    assert -2.4 < T[0] < -2.3 and 10.3 < T[-1] < 10.5


def test_gumbel_max_samples_softmax(orc):
    """Gumbel-max: argmax_c(x_c + g_c) with i.i.d. Gumbel g is distributed as
    softmax(x).  Checked with a chi-square test over 300k groups, using the
    oracle's noise for every group and the oracle's own forward at a tiny tau
    (which turns p into the one-hot of argmax(z))."""
    x = np.array([0.5, -0.3, 1.2, 0.0, -1.0, 0.8], np.float32)
    n = 300_000
    g = orc.gumbel_noise(42, 3, 9, 0, n)
    winners = np.argmax(x[None, :] + g, axis=1)
    counts = np.bincount(winners, minlength=6)
    expect = np.exp(x.astype(np.float64)) / np.exp(x.astype(np.float64)).sum() * n
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert chi2 < 35.0, (counts, expect, chi2)     # 5 dof; P(chi2 > 35) < 2e-6

    # the same through the oracle's forward: tau -> 0 makes p one-hot
    rows, cols = 50, 4 * 400
    L = np.broadcast_to(x, (rows, cols // 4, 6)).copy()
    W = np.full((rows, cols), 0x3F80, np.uint16)
    _, _, probs, _ = orc.forward(W, L, 1e-4, 1.0, 42, 3, 9, want_probs=True)
    fw = probs.reshape(-1, 6).argmax(1)
    assert (fw == winners[: rows * cols // 4]).all()
    # near-ties (|dz| < ~1e-3) keep a few groups from being one-hot
    assert (probs.reshape(-1, 6).max(1) > 1 - 1e-6).mean() > 0.995


# --------------------------------------------------------------------------
# Softmax and soft mask of one group
# --------------------------------------------------------------------------

def _random_groups(n, seed):
    rng = np.random.default_rng(seed)
    L = rng.normal(0, 1, (n, 6)).astype(np.float32)
    g = rng.gumbel(0, 1, (n, 6)).astype(np.float32)
    return L, g


def test_probs_invariants_and_log_ratios(orc):
    L, g = _random_groups(200, 1)
    for kappa, tau in [(1.0, 1.0), (3.0, 0.7), (0.0, 2.0), (100.0, 4.0)]:
        for n in range(200):
            p, _ = orc.group_probs(L[n], g[n], kappa, tau, exact=True)
            assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()
            # softmax's defining property: log-ratios are logit differences
            k64, t64 = float(np.float32(kappa)), float(np.float32(tau))   # fp32 arguments
            y = (k64 * L[n].astype(np.float64) + g[n].astype(np.float64)) / t64
            keep = p > 1e-200
            ratios = np.log(p[keep][:, None] / p[keep][None, :])
            diffs = y[keep][:, None] - y[keep][None, :]
            assert np.allclose(ratios, diffs, rtol=1e-10, atol=1e-9)


def test_fp32_logit_path_is_within_rounding_of_exact(orc):
    L, g = _random_groups(500, 2)
    for n in range(500):
        _, z32 = orc.group_probs(L[n], g[n], 300.0, 1.0, exact=False)
        _, z64 = orc.group_probs(L[n], g[n], 300.0, 1.0, exact=True)
        # three fp32 roundings: half an ulp of kappa*L and of kappa*L + g (both
        # then scaled by 1/tau = 1), and half an ulp of z
        a = 300.0 * L[n].astype(np.float64)
        s = a + g[n].astype(np.float64)
        sp = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)
        bound = 0.5 * (sp(a) + sp(s) + sp(z64)) * 1.01
        assert (np.abs(z32 - z64) <= bound).all()


def test_tau_to_zero_gives_one_hot(orc):
    L, g = _random_groups(100, 3)
    for n in range(100):
        p, z = orc.group_probs(L[n], g[n], 2.0, 1e-5, exact=True)
        c = int(np.argmax(2.0 * L[n].astype(np.float64) + g[n]))
        assert p[c] > 1 - 1e-9


def test_soft_mask_brute_force_and_invariants(orc):
    # candidate masks by brute force: all 4-bit vectors with exactly two ones,
    # ordered by their kept index pair
    S = sorted((tuple(j for j in range(4) if (b >> j) & 1), b) for b in range(16)
               if bin(b).count("1") == 2)
    S = np.array([[(b >> j) & 1 for j in range(4)] for _, b in S], np.float64)
    L, g = _random_groups(300, 4)
    for n in range(300):
        p, _ = orc.group_probs(L[n], g[n], 1.5, 0.8, exact=True)
        M = orc.soft_mask(p)
        assert np.allclose(M, p @ S, rtol=0, atol=1e-15)
        assert abs(M.sum() - 2.0) < 1e-12
        assert (M >= 0).all() and (M <= 1 + 1e-15).all()


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_on_float32_values(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([orc.double_to_bf16(float(v)) for v in f], np.uint16)
    assert (mine == ref).all()


def test_bf16_rounding_hand_cases(orc):
    assert orc.double_to_bf16(1.0 + 2 ** -8) == 0x3F80            # tie -> even (down)
    assert orc.double_to_bf16(1.0 + 3 * 2 ** -8) == 0x3F82        # tie -> even (up)
    # just above a tie: one rounding from double goes up, where rounding
    # through float32 first would have hit the tie and gone down
    assert orc.double_to_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert orc.double_to_bf16(-0.0) == 0x8000
    assert orc.double_to_bf16(1e39) == 0x7F80
    assert orc.double_to_bf16(-1e39) == 0xFF80
    assert orc.double_to_bf16(2.0 ** -133) == 0x0001              # smallest subnormal
    assert orc.double_to_bf16(2.0 ** -135) == 0x0000              # below half of it
    assert orc.double_to_bf16(3 * 2.0 ** -135) == 0x0001


# --------------------------------------------------------------------------
# Magnitude prior
# --------------------------------------------------------------------------

def test_prior_hand_cases(orc):
    W = np.array([[0x3F80, 0xC000, 0x4040, 0xC080] * 8], np.uint16)   # 1, -2, 3, -4
    L = orc.prior_init(W, 0.5)
    assert (L[0, 0] == np.array([1.5, 2.0, 2.5, 2.5, 3.0, 3.5], np.float32)).all()
    # fp32 rounding order: |w_i| + |w_j| is rounded to fp32 before the scale.
    # 1 + 2^-24 ties to 1.0; times (1 + 2^-23) gives 1 + 2^-23 exactly.  One
    # rounding of the exact product would give 1 + 2^-22 instead.
    W = np.array([[0x3F80, 0x3380, 0x0000, 0x0000] * 8], np.uint16)
    s = np.frombuffer(np.uint32(0x3F800001).tobytes(), np.float32)[0]
    L = orc.prior_init(W, float(s))
    assert L[0, 0, 0].view(np.uint32) == 0x3F800001


def test_prior_argmax_is_magnitude_pruning(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = rng.normal(0, 0.02, (64, 256)).astype(np.float32)
    W = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mag = np.abs(orc.bf16_to_f64(W)).reshape(64, 64, 4)
    srt = np.sort(mag, axis=2)
    tie_free = (np.diff(srt, axis=2) > 0).all(axis=2)
    L = orc.prior_init(W, 300.0)
    pairs = orc.candidate_pairs()
    for r in range(64):
        for k in range(64):
            if not tie_free[r, k]:
                continue
            top2 = tuple(sorted(np.argsort(mag[r, k])[-2:]))
            assert pairs[int(np.argmax(L[r, k]))] == top2


# --------------------------------------------------------------------------
# Forward over matrices
# --------------------------------------------------------------------------

def test_forward_one_hot_limit_keeps_weights_exactly(orc):
    rng = np.random.default_rng(7)
    rows, cols = 8, 64
    W = rng.integers(0x3C00, 0x4000, (rows, cols), dtype=np.uint16)
    W[::2] |= 0x8000
    L = rng.normal(0, 1, (rows, cols // 4, 6)).astype(np.float32)
    Wo, sq, probs, M = orc.forward(W, L, 1e-6, 1.0, 11, want_probs=True, want_masks=True)
    assert set(np.unique(M)) <= {0.0, 1.0}
    w = orc.bf16_to_f64(W)
    assert (orc.bf16_to_f64(Wo) == w * M).all()
    assert np.allclose(sq, (w * w * M).sum(1), rtol=1e-15)
    # kept positions are those of the sampled candidate
    pairs = orc.candidate_pairs()
    c = probs.argmax(2)
    for r in range(rows):
        for k in range(cols // 4):
            kept = [j for j in range(4) if M[r, 4 * k + j] == 1.0]
            assert tuple(kept) == pairs[c[r, k]]


def test_forward_generic_properties(orc):
    torch = pytest.importorskip("torch")
    from semi_structured_sparsity_gb300 import workloads as wl
    W, L, _ = wl.random_case(16, 96, seed=3)
    Wb = wl.bf16_bits(W)
    Wo, sq, probs, M = orc.forward(Wb, L.numpy(), 4.0, 100.0, 0, want_probs=True,
                                   want_masks=True)
    w = orc.bf16_to_f64(Wb)
    wo = orc.bf16_to_f64(Wo)
    assert (np.abs(wo) <= np.abs(w)).all()
    assert ((np.sign(wo) == np.sign(w)) | (wo == 0)).all()
    assert np.allclose(M.reshape(16, 24, 4).sum(2), 2.0, atol=1e-12)
    assert np.allclose(probs.sum(2), 1.0, atol=1e-12)
    expect = np.array([orc.double_to_bf16(v) for v in (w * M).ravel()], np.uint16)
    assert (Wo.ravel() == expect).all()
    assert np.allclose(sq, ((w * M) ** 2).sum(1), rtol=1e-13)


def test_row_begin_addresses_the_same_groups(orc):
    from semi_structured_sparsity_gb300 import workloads as wl
    W, L, G = wl.random_case(6, 64, seed=4)
    Wb, Gb, Ln = wl.bf16_bits(W), wl.bf16_bits(G), L.numpy()
    full = orc.forward(Wb, Ln, 1.0, 30.0, 5, 2, 3, want_probs=True)
    dfull = orc.backward(Wb, Ln, Gb, 1.0, 30.0, 5, 2, 3, 0.1)
    for r in range(6):
        one = orc.forward(Wb[r:r + 1], Ln[r:r + 1], 1.0, 30.0, 5, 2, 3, row_begin=r,
                          want_probs=True)
        assert (one[0][0] == full[0][r]).all() and (one[2][0] == full[2][r]).all()
        d = orc.backward(Wb[r:r + 1], Ln[r:r + 1], Gb[r:r + 1], 1.0, 30.0, 5, 2, 3, 0.1,
                         row_begin=r)
        assert (d[0] == dfull[r]).all()


# --------------------------------------------------------------------------
# Backward: finite differences
# --------------------------------------------------------------------------

@pytest.mark.parametrize("reg", [0.0, 0.37, -0.2])
def test_backward_matches_finite_differences(orc, reg):
    rng = np.random.default_rng(8)
    rows, cols = 2, 32
    W = np.array([orc.double_to_bf16(v) for v in rng.normal(0, 0.5, rows * cols)],
                 np.uint16).reshape(rows, cols)
    G = np.array([orc.double_to_bf16(v) for v in rng.normal(0, 1.0, rows * cols)],
                 np.uint16).reshape(rows, cols)
    L = rng.normal(0, 0.5, (rows, cols // 4, 6)).astype(np.float32)
    kappa, tau, seed = 3.0, 2.0, 99
    grad = orc.backward(W, L, G, tau, kappa, seed, 1, 2, reg, exact=True)
    h = np.float32(1e-3)
    flat = L.reshape(-1)
    for i in range(flat.size):
        Lp, Lm = flat.copy(), flat.copy()
        Lp[i] = flat[i] + h
        Lm[i] = flat[i] - h
        step = float(Lp[i]) - float(Lm[i])
        lp = orc.loss_exact(W, Lp, G, tau, kappa, seed, 1, 2, reg)
        lm = orc.loss_exact(W, Lm, G, tau, kappa, seed, 1, 2, reg)
        fd = (lp - lm) / step
        g = grad.reshape(-1)[i]
        # central differences: truncation ~ h^2 * (kappa/tau)^3 * |dl| / 6
        assert abs(fd - g) <= 1e-6 * max(1.0, abs(g)) + 1e-8, (i, fd, g)
    # the softmax Jacobian annihilates constants: gradients sum to zero per group
    assert np.allclose(grad.sum(2), 0.0, atol=1e-15)


def test_backward_fp32_definition_close_to_exact(orc):
    from semi_structured_sparsity_gb300 import workloads as wl
    W, L, G = wl.random_case(8, 64, seed=9)
    Wb, Gb, Ln = wl.bf16_bits(W), wl.bf16_bits(G), L.numpy()
    a = orc.backward(Wb, Ln, Gb, 4.0, 100.0, 0, exact=False)
    b = orc.backward(Wb, Ln, Gb, 4.0, 100.0, 0, exact=True)
    assert np.allclose(a, b, rtol=1e-4, atol=1e-9)


# --------------------------------------------------------------------------
# Hard mask and compressed storage
# --------------------------------------------------------------------------

def test_hard_index_hand_cases(orc):
    nan, inf = float("nan"), float("inf")
    cases = [
        ([1, 2, 3, 3, 2, 1], 2),              # tie: lowest index wins
        ([nan, 1, nan, 5, 5, nan], 3),        # NaN never wins
        ([nan] * 6, 0),                       # all NaN: candidate 0
        ([-inf] * 6, 0),
        ([-0.0, 0.0, -1, -1, -1, -1], 0),     # -0 == +0: a tie
        ([1, inf, 2, inf, nan, 3], 1),
        ([8, 0, 0, 0, 0, 8], 0),
        ([0, 0, 0, 0, 0, 8], 5),
    ]
    for logits, c in cases:
        assert orc.hard_index(np.array(logits, np.float32)) == c, logits


def test_hard_index_is_first_argmax(orc):
    rng = np.random.default_rng(10)
    L = rng.integers(-3, 4, (5000, 6)).astype(np.float32)   # many ties
    for n in range(5000):
        assert orc.hard_index(L[n]) == int(np.argmax(L[n]))   # numpy: first max


def test_metadata_hand_case(orc):
    rows = dict((r[0], r[1:]) for r in _golden_rows("metadata_hand_case.txt"))
    winners = [int(v) for v in rows["winners"]]
    W = (0x3F80 + np.arange(32)).astype(np.uint16).reshape(1, 32)
    L = np.zeros((1, 8, 6), np.float32)
    for k, c in enumerate(winners):
        L[0, k, c] = 1.0
    vals, meta, idx = orc.hard_compress(W, L)
    assert meta[0, 0] == int(rows["meta"][0], 16)
    assert [int(v) for v in vals[0]] == [int(v, 16) for v in rows["values"]]
    assert list(idx[0]) == winners


def test_compress_round_trip(orc):
    rng = np.random.default_rng(11)
    rows, cols = 12, 160
    W = rng.integers(0, 1 << 16, (rows, cols), dtype=np.uint64).astype(np.uint16)
    L = rng.integers(-2, 3, (rows, cols // 4, 6)).astype(np.float32)
    vals, meta, idx = orc.hard_compress(W, L)
    D = orc.decompress(vals, meta, rows, cols)
    pairs = orc.candidate_pairs()
    expect = np.zeros_like(W)
    for r in range(rows):
        for k in range(cols // 4):
            assert idx[r, k] == int(np.argmax(L[r, k]))
            for j in pairs[idx[r, k]]:
                expect[r, 4 * k + j] = W[r, 4 * k + j]
    assert (D == expect).all()            # select(mask, W, +0): bit-exact


def test_storage_savings_match_the_page(orc):
    for elem_bits, percent in _golden_rows("storage_savings.txt"):
        eb = int(elem_bits) // 8
        rows, cols = 4096, 4096
        dense = rows * cols * eb
        comp = orc.compressed_bytes(rows, cols, eb)
        saving = 1.0 - comp / dense
        assert round(100 * saving) == int(percent), (elem_bits, saving)
    # the exact closed forms: 16-bit -> 56.25% of dense, 8-bit -> 62.5%
    assert orc.compressed_bytes(64, 64, 2) * 10000 == 5625 * 64 * 64 * 2
    assert orc.compressed_bytes(64, 64, 1) * 1000 == 625 * 64 * 64


# --------------------------------------------------------------------------
# Prior from a given mask (Table 2) and the convergence diagnostics (Fig. 5)
# --------------------------------------------------------------------------

def test_prior_from_mask_hand_case_and_invalid_codes(orc):
    rows = dict((r[0], r[1:]) for r in _golden_rows("metadata_hand_case.txt"))
    winners = [int(v) for v in rows["winners"]]
    meta = np.array([[int(rows["meta"][0], 16)]], np.uint32)
    L = orc.prior_from_mask(meta, 1, 32, 5.0, -1.0)
    assert (L[0].argmax(1) == winners).all()
    assert (L[0].max(1) == 5.0).all() and ((L[0] == -1.0).sum(1) == 5).all()
    # codes that name no candidate (i >= j): every candidate gets `low`
    meta = np.array([[0x00000000 | (0x5 << 4) | (0xF << 8) | (0x1 << 12)]], np.uint32)
    L = orc.prior_from_mask(meta, 1, 32, 5.0, -1.0)
    assert (L[0, :4] == -1.0).all()
    assert [orc.candidate_of_code(c) for c in (0x4, 0x8, 0xC, 0x9, 0xD, 0xE)] == list(range(6))


def test_prior_from_mask_round_trips_hard_compress(orc):
    rng = np.random.default_rng(21)
    rows, cols = 9, 96
    W = rng.integers(0, 1 << 16, (rows, cols), dtype=np.uint64).astype(np.uint16)
    L = rng.normal(0, 1, (rows, cols // 4, 6)).astype(np.float32)
    _, meta, idx = orc.hard_compress(W, L)
    P = orc.prior_from_mask(meta, rows, cols, 3.0, 0.0)
    assert (P.argmax(2) == idx).all()
    _, meta2, idx2 = orc.hard_compress(W, P)
    assert (meta2 == meta).all() and (idx2 == idx).all()


def test_mask_stats_large_kappa_freezes_the_samples(orc):
    """Fig. 5: an inappropriately large kappa suppresses exploration -- the
    sampled mask is the hard mask at every step and the mask difference
    between adjacent steps is zero."""
    rng = np.random.default_rng(22)
    rows, cols = 16, 256
    L = rng.normal(0, 1, (rows, cols // 4, 6)).astype(np.float32)
    hard = np.array([[orc.hard_index(L[r, k]) for k in range(cols // 4)] for r in range(rows)])
    prev, _, _ = orc.mask_stats(L, rows, cols, 1.0, 1e6, 5, step=0)
    cur, l1, mp = orc.mask_stats(L, rows, cols, 1.0, 1e6, 5, step=1, prev_idx=prev)
    assert (prev == hard).all() and (cur == hard).all()
    assert (l1 == 0).all()
    assert np.allclose(mp, cols // 4, rtol=1e-9)       # max probability -> 1 per group


def test_mask_stats_zero_kappa_is_uniform_random(orc):
    """kappa = 0: every candidate equally likely at every step (Gumbel-max over
    equal logits), so the sample is uniform and independent across steps.
    Two independent uniform candidates differ in L1 by 0 (same, p = 1/6), 2
    (one shared position, p = 4/6) or 4 (complementary pairs, p = 1/6): the
    expected distance is exactly 2 per group; the maximum probability is
    exactly 1/6."""
    rows, cols = 100, 1600
    G = rows * cols // 4
    L = np.random.default_rng(23).normal(0, 1, (rows, cols // 4, 6)).astype(np.float32)
    prev, _, _ = orc.mask_stats(L, rows, cols, 1.0, 0.0, 9, step=10)
    cur, l1, mp = orc.mask_stats(L, rows, cols, 1.0, 0.0, 9, step=11, prev_idx=prev)
    mean = l1.sum() / G
    assert abs(mean - 2.0) < 5 * math.sqrt(4.0 / 3.0 / G)
    counts = np.bincount(cur.ravel(), minlength=6)
    chi2 = ((counts - G / 6) ** 2 / (G / 6)).sum()
    assert chi2 < 35.0
    assert np.allclose(mp, (cols // 4) / 6.0, rtol=1e-12)


def test_mask_stats_l1_hand_cases(orc):
    """Force the samples with a large kappa on one-hot logits: candidate 0
    (0,1) then 5 (2,3) differ in all four positions; 0 then 1 (0,2) in two."""
    rows, cols = 1, 32
    def onehot(cands):
        L = np.full((1, 8, 6), -10.0, np.float32)
        for k, c in enumerate(cands):
            L[0, k, c] = 10.0
        return L
    a = [0, 0, 1, 2, 3, 4, 5, 2]
    b = [5, 1, 1, 3, 2, 1, 0, 4]
    want = [4, 2, 0, 4, 4, 4, 4, 2]   # (0,1)|(2,3) (0,1)|(0,2) same (0,3)|(1,2) ... (1,3)|(0,2) ...
    prev, _, _ = orc.mask_stats(onehot(a), rows, cols, 1.0, 1e4, 0)
    cur, l1, _ = orc.mask_stats(onehot(b), rows, cols, 1.0, 1e4, 0, step=1, prev_idx=prev)
    assert list(prev[0]) == a and list(cur[0]) == b
    assert l1[0] == sum(want)


def test_mask_stats_sample_is_the_forward_argmax(orc):
    from semi_structured_sparsity_gb300 import workloads as wl
    W, L, _ = wl.random_case(8, 128, seed=24)
    Wb, Ln = wl.bf16_bits(W), L.numpy()
    _, _, probs, _ = orc.forward(Wb, Ln, 0.5, 30.0, 3, 4, 5, want_probs=True)
    idx, _, _ = orc.mask_stats(Ln, 8, 128, 0.5, 30.0, 3, step=4, tensor_id=5)
    assert (idx == probs.argmax(2)).all()
