"""Comparison helpers shared by the GPU parity tests.

Tolerances (stated once, used everywhere):
  * noise words, argmax indices, metadata, compressed values, decompressed
    weights, prior logits: bit-exact;
  * W' (bf16): within 1 bf16 ulp, compared as ordered integers;
  * p and dlogits: |got - want| <= 1e-6 + 1e-4 * |want|;
  * row_sq: relative 1e-4 (the reduction order differs from the oracle's).
"""
import numpy as np
import torch

P_RTOL, P_ATOL = 1e-4, 1e-6
ROWSQ_RTOL = 1e-4
W_ULPS = 1


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_bf16_ulps(got_bits, want_bits, ulps=W_ULPS, what="W'"):
    d = np.abs(bf16_ordered(got_bits) - bf16_ordered(want_bits))
    if d.size and d.max() > ulps:
        i = np.unravel_index(np.argmax(d), d.shape)
        raise AssertionError("%s differs by %d bf16 ulps at %s (got 0x%04X want 0x%04X); "
                             "%d elements beyond %d ulp" % (what, d[i], i, got_bits[i],
                                                            want_bits[i], (d > ulps).sum(), ulps))


def assert_close(got, want, rtol=P_RTOL, atol=P_ATOL, what="value"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    excess = np.abs(got - want) - (atol + rtol * np.abs(want))
    if excess.size and excess.max() > 0:
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError("%s mismatch at %s: got %.9g want %.9g (|diff| %.3g, allowed %.3g); "
                             "%d elements out of tolerance" % (
                                 what, i, got[i], want[i], abs(got[i] - want[i]),
                                 atol + rtol * abs(want[i]), (excess > 0).sum()))


def assert_bits_equal(got, want, what="bits"):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = got != want
    if bad.any():
        i = np.unravel_index(np.argmax(bad), bad.shape)
        raise AssertionError("%s differ at %s (got %r want %r); %d differing" % (
            what, i, got[i], want[i], bad.sum()))


def sampled_rows(rows: int, every: int = 64):
    r = list(range(0, rows, every))
    if r[-1] != rows - 1:
        r.append(rows - 1)
    return r
