"""Plain CPU oracle of the MaskLLM 2:4 mask layer (ctypes wrapper over the C code).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The product path (the CUDA library
and its binding) never imports this package, and this package imports nothing
from the product.

All array arguments are numpy arrays on the host.  bf16 tensors travel as
``uint16`` bit patterns.  Float outputs of the oracle are float64 (it computes
in double after the fp32 logit arithmetic that defines z; see the C header).
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import _build

NCAND = 6
TABLE_BITS = 14
TABLE_SIZE = 1 << TABLE_BITS

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
        i64, u64, u32, f32 = C.c_int64, C.c_uint64, C.c_uint32, C.c_float
        vp = C.c_void_p
        L.orc_candidate_pair.argtypes = [C.c_int, C.c_int]
        L.orc_candidate_pair.restype = C.c_int
        L.orc_candidate_keeps.argtypes = [C.c_int, C.c_int]
        L.orc_candidate_keeps.restype = C.c_int
        L.orc_bf16_to_double.argtypes = [C.c_uint16]
        L.orc_bf16_to_double.restype = C.c_double
        L.orc_double_to_bf16.argtypes = [C.c_double]
        L.orc_double_to_bf16.restype = C.c_uint16
        L.orc_philox4x32_10.argtypes = [u32p, u32p, u32p]
        L.orc_philox4x32_10.restype = None
        L.orc_noise_words.argtypes = [u64, u32, u32, i64, i64, u32p]
        L.orc_noise_words.restype = None
        L.orc_gumbel_table.argtypes = [f32p]
        L.orc_gumbel_table.restype = None
        L.orc_gumbel_noise.argtypes = [u64, u32, u32, i64, i64, f32p]
        L.orc_gumbel_noise.restype = None
        L.orc_gumbel_cell.argtypes = [u32p, C.c_int]
        L.orc_gumbel_cell.restype = C.c_int
        L.orc_group_probs.argtypes = [f32p, f32p, f32, f32, C.c_int, f64p, vp]
        L.orc_group_probs.restype = None
        L.orc_soft_mask.argtypes = [f64p, f64p]
        L.orc_soft_mask.restype = None
        L.orc_group_backward.argtypes = [f64p, f64p, f64p, C.c_double, f64p]
        L.orc_group_backward.restype = None
        L.orc_prior_init.argtypes = [u16p, i64, i64, f32, f32p]
        L.orc_prior_init.restype = None
        L.orc_forward.argtypes = [u16p, f32p, i64, i64, i64, f32, f32, u64, u32, u32,
                                  u16p, vp, vp, vp]
        L.orc_forward.restype = None
        L.orc_backward.argtypes = [u16p, f32p, u16p, i64, i64, i64, f32, f32, u64, u32,
                                   u32, f32, C.c_int, f64p]
        L.orc_backward.restype = None
        L.orc_loss_exact.argtypes = [u16p, f32p, u16p, i64, i64, i64, f32, f32, u64, u32,
                                     u32, f32]
        L.orc_loss_exact.restype = C.c_double
        L.orc_hard_index.argtypes = [f32p]
        L.orc_hard_index.restype = C.c_int
        L.orc_hard_compress.argtypes = [u16p, f32p, i64, i64, u16p, u32p, vp]
        L.orc_hard_compress.restype = None
        L.orc_decompress.argtypes = [u16p, u32p, i64, i64, u16p]
        L.orc_decompress.restype = None
        L.orc_compressed_bytes.argtypes = [i64, i64, i64]
        L.orc_compressed_bytes.restype = i64
        i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
        L.orc_candidate_of_code.argtypes = [u32]
        L.orc_candidate_of_code.restype = C.c_int
        L.orc_prior_from_mask.argtypes = [u32p, i64, i64, f32, f32, f32p]
        L.orc_prior_from_mask.restype = None
        L.orc_mask_stats.argtypes = [f32p, i64, i64, i64, f32, f32, u64, u32, u32, vp, vp, vp, vp]
        L.orc_mask_stats.restype = None
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        i32 = C.c_int32
        L.orc_perm_shift.argtypes = [u16p, i64, i64]
        L.orc_perm_shift.restype = i32
        L.orc_perm_fixed.argtypes = [C.c_uint16, i32]
        L.orc_perm_fixed.restype = u32
        L.orc_perm_metric_fixed.argtypes = [u16p, i64, i64, i32p, i32]
        L.orc_perm_metric_fixed.restype = u64
        L.orc_perm_metric.argtypes = [u16p, i64, i64, i32p]
        L.orc_perm_metric.restype = C.c_double
        L.orc_perm_swap_gain.argtypes = [u16p, i64, i64, i32p, i32, i64, i64]
        L.orc_perm_swap_gain.restype = i64
        L.orc_perm_search.argtypes = [u16p, i64, i64, i32p, i32, i32, vp, vp]
        L.orc_perm_search.restype = i32
        _ = (u8p, i64p)
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def candidate_pairs():
    """The six kept index pairs in the oracle's candidate order."""
    return [(lib().orc_candidate_pair(c, 0), lib().orc_candidate_pair(c, 1))
            for c in range(NCAND)]


def bf16_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def double_to_bf16(x: float) -> int:
    return int(lib().orc_double_to_bf16(float(x)))


def philox4x32_10(key, ctr):
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_c(key, np.uint32), _c(ctr, np.uint32), out)
    return out


def noise_words(seed: int, step: int, tensor_id: int, group_begin: int, n: int):
    out = np.zeros((n, 4), np.uint32)
    lib().orc_noise_words(seed, step, tensor_id, group_begin, n, out)
    return out


def gumbel_table():
    t = np.zeros(TABLE_SIZE, np.float32)
    lib().orc_gumbel_table(t)
    return t


def gumbel_noise(seed: int, step: int, tensor_id: int, group_begin: int, n: int):
    out = np.zeros((n, NCAND), np.float32)
    lib().orc_gumbel_noise(seed, step, tensor_id, group_begin, n, out)
    return out


def gumbel_cell(words, c: int) -> int:
    return int(lib().orc_gumbel_cell(_c(words, np.uint32), c))


def group_probs(logits, gumbel, kappa: float, tau: float, exact: bool = False):
    p = np.zeros(NCAND, np.float64)
    z = np.zeros(NCAND, np.float64)
    lib().orc_group_probs(_c(logits, np.float32), _c(gumbel, np.float32), kappa, tau,
                          int(exact), p, _ptr(z))
    return p, z


def soft_mask(p):
    m = np.zeros(4, np.float64)
    lib().orc_soft_mask(_c(p, np.float64), m)
    return m


def group_backward(p, w, t, dz_dlogit: float):
    out = np.zeros(NCAND, np.float64)
    lib().orc_group_backward(_c(p, np.float64), _c(w, np.float64), _c(t, np.float64),
                             float(dz_dlogit), out)
    return out


def prior_init(W, scale: float):
    W = _c(W, np.uint16)
    rows, cols = W.shape
    out = np.zeros((rows, cols // 4, NCAND), np.float32)
    lib().orc_prior_init(W, rows, cols, scale, out)
    return out


def forward(W, L, tau, kappa, seed, step=0, tensor_id=0, row_begin=0,
            want_probs=False, want_masks=False):
    """Returns (W_out bf16 bits [rows, cols], row_sq f64 [rows], probs|None, masks|None)."""
    W = _c(W, np.uint16)
    rows, cols = W.shape
    L = _c(L, np.float32).reshape(rows, cols // 4, NCAND)
    W_out = np.zeros((rows, cols), np.uint16)
    row_sq = np.zeros(rows, np.float64)
    probs = np.zeros((rows, cols // 4, NCAND), np.float64) if want_probs else None
    masks = np.zeros((rows, cols), np.float64) if want_masks else None
    lib().orc_forward(W, L, rows, cols, row_begin, tau, kappa, seed, step, tensor_id,
                      W_out, _ptr(row_sq), _ptr(probs), _ptr(masks))
    return W_out, row_sq, probs, masks


def backward(W, L, G, tau, kappa, seed, step=0, tensor_id=0, reg_coeff=0.0, row_begin=0,
             exact=False):
    W = _c(W, np.uint16)
    rows, cols = W.shape
    L = _c(L, np.float32).reshape(rows, cols // 4, NCAND)
    G = _c(G, np.uint16)
    out = np.zeros((rows, cols // 4, NCAND), np.float64)
    lib().orc_backward(W, L, G, rows, cols, row_begin, tau, kappa, seed, step, tensor_id,
                       reg_coeff, int(exact), out)
    return out


def loss_exact(W, L, G, tau, kappa, seed, step=0, tensor_id=0, reg_coeff=0.0, row_begin=0):
    W = _c(W, np.uint16)
    rows, cols = W.shape
    L = _c(L, np.float32).reshape(rows, cols // 4, NCAND)
    G = _c(G, np.uint16)
    return lib().orc_loss_exact(W, L, G, rows, cols, row_begin, tau, kappa, seed, step,
                                tensor_id, reg_coeff)


def hard_index(logits6) -> int:
    return int(lib().orc_hard_index(_c(logits6, np.float32)))


def hard_compress(W, L):
    """Returns (values bf16 bits [rows, cols/2], meta u32 [rows, cols/32], idx u8 [rows, cols/4])."""
    W = _c(W, np.uint16)
    rows, cols = W.shape
    L = _c(L, np.float32).reshape(rows, cols // 4, NCAND)
    vals = np.zeros((rows, cols // 2), np.uint16)
    meta = np.zeros((rows, cols // 32), np.uint32)
    idx = np.zeros((rows, cols // 4), np.uint8)
    lib().orc_hard_compress(W, L, rows, cols, vals, meta, _ptr(idx))
    return vals, meta, idx


def decompress(vals, meta, rows: int, cols: int):
    out = np.zeros((rows, cols), np.uint16)
    lib().orc_decompress(_c(vals, np.uint16), _c(meta, np.uint32), rows, cols, out)
    return out


def compressed_bytes(rows: int, cols: int, elem_bytes: int) -> int:
    return int(lib().orc_compressed_bytes(rows, cols, elem_bytes))


def candidate_of_code(code: int) -> int:
    return int(lib().orc_candidate_of_code(code))


def prior_from_mask(meta, rows: int, cols: int, high: float, low: float):
    out = np.zeros((rows, cols // 4, NCAND), np.float32)
    lib().orc_prior_from_mask(_c(meta, np.uint32).reshape(rows, cols // 32), rows, cols, high, low,
                              out)
    return out


def mask_stats(L, rows, cols, tau, kappa, seed, step=0, tensor_id=0, prev_idx=None, row_begin=0):
    """Returns (idx u8 [rows, cols/4], l1 int64 [rows] or None, maxprob f64 [rows])."""
    L = _c(L, np.float32).reshape(rows, cols // 4, NCAND)
    idx = np.zeros((rows, cols // 4), np.uint8)
    l1 = np.zeros(rows, np.int64) if prev_idx is not None else None
    mp = np.zeros(rows, np.float64)
    prev = None if prev_idx is None else _c(prev_idx, np.uint8).reshape(rows, cols // 4)
    lib().orc_mask_stats(L, rows, cols, row_begin, tau, kappa, seed, step, tensor_id, _ptr(prev),
                         _ptr(idx), _ptr(l1), _ptr(mp))
    return idx, l1, mp


# ---------------------------------------------------------------------------
# channel permutation before pruning
# ---------------------------------------------------------------------------

PERM_NONFINITE = -(2 ** 31)   # orc_perm_shift's answer for a non-finite weight


def perm_shift(W) -> int:
    W = _c(W, np.uint16)
    return int(lib().orc_perm_shift(W, W.shape[0], W.shape[1]))


def perm_fixed(w_bits: int, shift: int) -> int:
    return int(lib().orc_perm_fixed(int(w_bits), int(shift)))


def perm_metric_fixed(W, perm, shift: int) -> int:
    W = _c(W, np.uint16)
    return int(lib().orc_perm_metric_fixed(W, W.shape[0], W.shape[1], _c(perm, np.int32), shift))


def perm_metric(W, perm) -> float:
    W = _c(W, np.uint16)
    return float(lib().orc_perm_metric(W, W.shape[0], W.shape[1], _c(perm, np.int32)))


def perm_swap_gain(W, perm, shift: int, a: int, b: int) -> int:
    W = _c(W, np.uint16)
    p = np.array(perm, np.int32)
    return int(lib().orc_perm_swap_gain(W, W.shape[0], W.shape[1], p, shift, a, b))


def perm_swap_gains(W, perm, shift: int):
    """[cols, cols] int64: the fixed-point gain of every swap (0 within a group)."""
    W = _c(W, np.uint16)
    cols = W.shape[1]
    out = np.zeros((cols, cols), np.int64)
    for a in range(cols):
        for b in range(a + 1, cols):
            out[a, b] = out[b, a] = perm_swap_gain(W, perm, shift, a, b)
    return out


def perm_search(W, perm, shift: int, max_swaps: int):
    """Returns (perm after the search, swaps int32 [n, 2], gains int64 [n])."""
    W = _c(W, np.uint16)
    p = np.array(perm, np.int32)
    swaps = np.zeros((max(max_swaps, 1), 2), np.int32)
    gains = np.zeros(max(max_swaps, 1), np.int64)
    n = int(lib().orc_perm_search(W, W.shape[0], W.shape[1], p, shift, max_swaps, _ptr(swaps),
                                  _ptr(gains)))
    return p, swaps[:n].copy(), gains[:n].copy()


# ---------------------------------------------------------------------------
# 2:4 sparse x dense product
# ---------------------------------------------------------------------------

def spmm(values, meta, M: int, K: int, B):
    """C = A B^T in float64, A the [M, K] matrix stored as 2:4 values [M, K/2]
    (bf16 bits) + metadata [M, K/32] (the orc_hard_compress layout), B dense
    bf16 bits [N, K] ("Accelerating Sparse Deep Neural Networks", Sec. 3.2:
    the sparse tensor core multiplies a 2:4 sparse first operand by a dense
    second operand into a dense result).  Returns (C, S) with S = sum over k
    of |A[m,k] B[n,k]|, the scale of the rounding error of any summation
    order.  The product itself is numpy's float64 matmul of the decompressed
    matrix: every bf16 product is exact in binary64 and the sums are rounded
    only at binary64 precision, far below the fp32 accumulation error of any
    single-precision kernel."""
    A = bf16_to_f64(decompress(values, meta, M, K))
    Bf = bf16_to_f64(np.asarray(B, np.uint16).reshape(-1, K))
    return A @ Bf.T, np.abs(A) @ np.abs(Bf).T
