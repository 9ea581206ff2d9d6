"""Pins of the oracle's 2:4 sparse x dense product ("Accelerating Sparse Deep
Neural Networks", Sec. 3.1 storage, Sec. 3.2 sparse tensor core product):
a hand case, a pure-Python triple loop, and the masked dense product built
without the compressed format.  CPU only."""
import numpy as np

import oracle as orc

PAIRS = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


def bf16(x):
    x = np.asarray(x, np.float64)
    return np.array([orc.double_to_bf16(float(v)) for v in x.ravel()], np.uint16).reshape(x.shape)


def test_hand_case_recovers_the_sparse_rows():
    # one row, K = 32: group g keeps 1 + g at its first kept position and
    # -(1 + g) at its second; B = the identity (N = 32) gives A back
    W = np.zeros((1, 32))
    L = np.full((1, 8, 6), -1.0, np.float32)
    for g in range(8):
        c = g % 6
        i, j = PAIRS[c]
        W[0, 4 * g + i], W[0, 4 * g + j] = 1 + g, -(1 + g)
        L[0, g, c] = 1.0
    vals, meta, _ = orc.hard_compress(bf16(W), L)
    C, S = orc.spmm(vals, meta, 1, 32, bf16(np.eye(32)))
    assert np.array_equal(C, W)
    assert np.array_equal(S, np.abs(W))


def test_small_integers_against_a_triple_loop():
    rng = np.random.default_rng(0)
    M, K, N = 5, 64, 7
    W = bf16(rng.integers(-8, 9, (M, K)))
    L = rng.normal(size=(M, K // 4, 6)).astype(np.float32)
    B = bf16(rng.integers(-8, 9, (N, K)))
    vals, meta, idx = orc.hard_compress(W, L)
    C, _ = orc.spmm(vals, meta, M, K, B)
    Wf, Bf = orc.bf16_to_f64(W), orc.bf16_to_f64(B)
    for m in range(M):
        for n in range(N):
            s = 0.0
            for g in range(K // 4):
                i, j = PAIRS[idx[m, g]]
                s += Wf[m, 4 * g + i] * Bf[n, 4 * g + i] + Wf[m, 4 * g + j] * Bf[n, 4 * g + j]
            assert C[m, n] == s


def test_equals_the_masked_dense_product():
    # the hard mask built directly (first maximum of the raw logits), applied
    # to W, multiplied densely: no compressed format involved
    rng = np.random.default_rng(1)
    M, K, N = 16, 128, 24
    W = bf16(rng.normal(0, 0.02, (M, K)))
    L = rng.normal(size=(M, K // 4, 6)).astype(np.float32)
    B = bf16(rng.normal(0, 1, (N, K)))
    keep = np.zeros((6, 4))
    for c, (i, j) in enumerate(PAIRS):
        keep[c, i] = keep[c, j] = 1
    mask = keep[np.argmax(L, axis=-1)].reshape(M, K)
    want = (orc.bf16_to_f64(W) * mask) @ orc.bf16_to_f64(B).T
    vals, meta, _ = orc.hard_compress(W, L)
    C, S = orc.spmm(vals, meta, M, K, B)
    assert np.allclose(C, want, rtol=0, atol=1e-15)
    assert (S >= np.abs(C)).all()
