"""Thin Python binding of libmaskllm (include/maskllm.h), via ctypes.

Argument marshalling only: every function checks the torch tensors it is given
(device, dtype, shape, contiguity), allocates outputs that were not passed in
(PyTorch is the device allocator), and calls the C entry point of the same
name on the current CUDA stream.  No step of the computation runs here.  If
``libmaskllm.so`` has not been built, ``lib()`` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmaskllm.so")

MASKLLM_OK = 0
STATUS = {0: "MASKLLM_OK", 1: "MASKLLM_ERR_INVALID_ARG", 2: "MASKLLM_ERR_SHAPE",
          3: "MASKLLM_ERR_ALIGNMENT", 4: "MASKLLM_ERR_ALIAS", 5: "MASKLLM_ERR_CUDA",
          6: "MASKLLM_ERR_TIMEOUT"}

# The entry points of include/maskllm.h.
EXPORTS = ("maskllm_prior_init", "maskllm_forward", "maskllm_backward",
           "maskllm_hard_compress", "maskllm_decompress", "maskllm_noise_words",
           "maskllm_prior_init_batched", "maskllm_forward_batched", "maskllm_backward_batched",
           "maskllm_hard_compress_batched", "maskllm_prior_from_mask",
           "maskllm_prior_from_mask_batched", "maskllm_mask_stats",
           "maskllm_perm_shift", "maskllm_perm_metric", "maskllm_permute_columns",
           "maskllm_perm_swap_gains", "maskllm_perm_search", "maskllm_perm_search_static",
           "maskllm_spmm", "maskllm_forward_stats", "maskllm_mask_stats_batched",
           "maskllm_forward_stats_batched", "maskllm_backward_stats",
           "maskllm_backward_stats_batched",
           "maskllm_set_wait_timeout",
           "maskllm_test_withhold_loads", "maskllm_test_spmm_tile_n", "maskllm_device_status",
           "maskllm_status_string",
           "maskllm_last_cuda_error", "maskllm_perm_workspace_bytes")
MAX_BATCH = 16
PERM_BAD_PERMUTATION = -1   # maskllm_perm_search / maskllm_perm_swap_gains outcome codes
PERM_NONFINITE = -2
PERM_SEARCH_STATIC_BYTES = 32 * 1024 * 1024   # the library-held scratch of the no-allocation search


class maskllm_rng(C.Structure):
    _fields_ = [("seed", C.c_uint64), ("step", C.c_uint32), ("tensor_id", C.c_uint32)]


class maskllm_matrix(C.Structure):
    _fields_ = [("W", C.c_void_p), ("logits", C.c_void_p), ("grad_W_out", C.c_void_p),
                ("rows", C.c_int64), ("cols", C.c_int64), ("tensor_id", C.c_uint32),
                ("logits_out", C.c_void_p), ("W_out", C.c_void_p), ("row_sq_out", C.c_void_p),
                ("probs_out", C.c_void_p), ("dlogits_out", C.c_void_p),
                ("values_out", C.c_void_p), ("meta_out", C.c_void_p), ("idx_out", C.c_void_p),
                ("meta", C.c_void_p), ("prev_idx", C.c_void_p), ("l1_row_out", C.c_void_p),
                ("maxprob_row_out", C.c_void_p)]


class MaskLLMError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        msg = "%s returned %s" % (fn, STATUS.get(status, str(status)))
        super().__init__(msg + (": " + detail if detail else ""))


_lib = None


def lib() -> C.CDLL:
    """Load libmaskllm.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmaskllm.so is not built (%s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        L = C.CDLL(LIB_PATH)
        vp, i64, f32, st = C.c_void_p, C.c_int64, C.c_float, C.c_int
        L.maskllm_prior_init.argtypes = [vp, i64, i64, f32, vp, vp]
        L.maskllm_forward.argtypes = [vp, vp, i64, i64, f32, f32, maskllm_rng, vp, vp, vp, vp]
        L.maskllm_backward.argtypes = [vp, vp, vp, i64, i64, f32, f32, maskllm_rng, f32, vp, vp]
        L.maskllm_hard_compress.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp]
        L.maskllm_decompress.argtypes = [vp, vp, i64, i64, vp, vp]
        L.maskllm_noise_words.argtypes = [maskllm_rng, i64, i64, vp, vp]
        L.maskllm_device_status.argtypes = [vp]
        mp = C.POINTER(maskllm_matrix)
        i32, u64, u32 = C.c_int32, C.c_uint64, C.c_uint32
        L.maskllm_prior_init_batched.argtypes = [mp, i32, f32, vp]
        L.maskllm_forward_batched.argtypes = [mp, i32, f32, f32, u64, u32, vp]
        L.maskllm_backward_batched.argtypes = [mp, i32, f32, f32, u64, u32, f32, vp]
        L.maskllm_hard_compress_batched.argtypes = [mp, i32, vp]
        L.maskllm_prior_from_mask.argtypes = [vp, i64, i64, f32, f32, vp, vp]
        L.maskllm_prior_from_mask_batched.argtypes = [mp, i32, f32, f32, vp]
        L.maskllm_mask_stats.argtypes = [vp, vp, i64, i64, f32, f32, maskllm_rng, vp, vp, vp, vp]
        L.maskllm_set_wait_timeout.argtypes = [u64]
        L.maskllm_test_withhold_loads.argtypes = [i32]
        L.maskllm_test_spmm_tile_n.argtypes = [i32]
        L.maskllm_perm_shift.argtypes = [vp, i64, i64, vp, vp]
        L.maskllm_perm_metric.argtypes = [vp, i64, i64, vp, vp, vp, vp]
        L.maskllm_permute_columns.argtypes = [vp, i64, i64, vp, vp, vp]
        L.maskllm_perm_swap_gains.argtypes = [vp, i64, i64, vp, vp, i64, vp, vp, vp, vp]
        L.maskllm_perm_search.argtypes = [vp, i64, i64, vp, i32, vp, i64, vp, vp, vp, vp, vp]
        L.maskllm_perm_search_static.argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp]
        L.maskllm_spmm.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp]
        L.maskllm_forward_stats.argtypes = [vp, vp, vp, i64, i64, f32, f32, maskllm_rng, vp, vp,
                                            vp, vp, vp, vp]
        L.maskllm_mask_stats_batched.argtypes = [mp, i32, f32, f32, u64, u32, vp]
        L.maskllm_forward_stats_batched.argtypes = [mp, i32, f32, f32, u64, u32, vp]
        L.maskllm_backward_stats.argtypes = [vp, vp, vp, vp, i64, i64, f32, f32, maskllm_rng, f32,
                                             vp, vp, vp, vp, vp]
        L.maskllm_backward_stats_batched.argtypes = [mp, i32, f32, f32, u64, u32, f32, vp]
        for fn in EXPORTS[:-3]:
            getattr(L, fn).restype = st
        L.maskllm_perm_workspace_bytes.argtypes = [i64, i64]
        L.maskllm_perm_workspace_bytes.restype = i64
        L.maskllm_status_string.argtypes = [st]
        L.maskllm_status_string.restype = C.c_char_p
        L.maskllm_last_cuda_error.argtypes = []
        L.maskllm_last_cuda_error.restype = C.c_char_p
        _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != MASKLLM_OK:
        detail = lib().maskllm_last_cuda_error().decode() if status == 5 else ""
        raise MaskLLMError(fn, status, detail)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _out(t, name, dtype, shape, like):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return _need(t, name, dtype, shape)


def _rng(rng) -> maskllm_rng:
    if isinstance(rng, maskllm_rng):
        return rng
    seed, step, tensor_id = rng
    return maskllm_rng(seed, step, tensor_id)


def maskllm_prior_init(W, scale, logits_out=None, stream=None):
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    logits_out = _out(logits_out, "logits_out", torch.float32, (rows, cols // 4, 6), W)
    _check("maskllm_prior_init", lib().maskllm_prior_init(
        _ptr(W), rows, cols, scale, _ptr(logits_out), _stream(stream)))
    return logits_out


def maskllm_forward(W, logits, tau, kappa, rng, W_out=None, row_sq_out=None, probs_out=None,
                    want_row_sq=True, stream=None):
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _need(logits, "logits", torch.float32, (rows, cols // 4, 6))
    W_out = _out(W_out, "W_out", torch.bfloat16, (rows, cols), W)
    if row_sq_out is None and want_row_sq:
        row_sq_out = torch.empty((rows,), dtype=torch.float32, device=W.device)
    elif row_sq_out is not None:
        _need(row_sq_out, "row_sq_out", torch.float32, (rows,))
    if probs_out is not None:
        _need(probs_out, "probs_out", torch.float32, (rows, cols // 4, 6))
    _check("maskllm_forward", lib().maskllm_forward(
        _ptr(W), _ptr(logits), rows, cols, tau, kappa, _rng(rng), _ptr(W_out),
        _ptr(row_sq_out), _ptr(probs_out), _stream(stream)))
    return W_out, row_sq_out, probs_out


def maskllm_backward(W, logits, grad_W_out, tau, kappa, rng, reg_coeff=0.0, dlogits_out=None,
                     stream=None):
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _need(logits, "logits", torch.float32, (rows, cols // 4, 6))
    _need(grad_W_out, "grad_W_out", torch.bfloat16, (rows, cols))
    dlogits_out = _out(dlogits_out, "dlogits_out", torch.float32, (rows, cols // 4, 6), W)
    _check("maskllm_backward", lib().maskllm_backward(
        _ptr(W), _ptr(logits), _ptr(grad_W_out), rows, cols, tau, kappa, _rng(rng), reg_coeff,
        _ptr(dlogits_out), _stream(stream)))
    return dlogits_out


def maskllm_hard_compress(W, logits, values_out=None, meta_out=None, idx_out=None,
                          want_idx=False, stream=None):
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _need(logits, "logits", torch.float32, (rows, cols // 4, 6))
    values_out = _out(values_out, "values_out", torch.bfloat16, (rows, cols // 2), W)
    meta_out = _out(meta_out, "meta_out", torch.int32, (rows, cols // 32), W)
    if idx_out is None and want_idx:
        idx_out = torch.empty((rows, cols // 4), dtype=torch.uint8, device=W.device)
    elif idx_out is not None:
        _need(idx_out, "idx_out", torch.uint8, (rows, cols // 4))
    _check("maskllm_hard_compress", lib().maskllm_hard_compress(
        _ptr(W), _ptr(logits), rows, cols, _ptr(values_out), _ptr(meta_out), _ptr(idx_out),
        _stream(stream)))
    return values_out, meta_out, idx_out


def maskllm_decompress(values, meta, rows, cols, W_out=None, stream=None):
    _need(values, "values", torch.bfloat16, (rows, cols // 2))
    _need(meta, "meta", torch.int32, (rows, cols // 32))
    W_out = _out(W_out, "W_out", torch.bfloat16, (rows, cols), values)
    _check("maskllm_decompress", lib().maskllm_decompress(
        _ptr(values), _ptr(meta), rows, cols, _ptr(W_out), _stream(stream)))
    return W_out


def maskllm_noise_words(rng, group_begin, n, out4=None, device="cuda", stream=None):
    if out4 is None:
        out4 = torch.empty((n, 4), dtype=torch.int32, device=device)
    else:
        _need(out4, "out4", torch.int32, (n, 4))
    _check("maskllm_noise_words", lib().maskllm_noise_words(
        _rng(rng), group_begin, n, _ptr(out4), _stream(stream)))
    return out4


def maskllm_device_status(stream=None) -> int:
    return int(lib().maskllm_device_status(_stream(stream)))


def maskllm_status_string(status: int) -> str:
    return lib().maskllm_status_string(status).decode()


# ---------------------------------------------------------------------------
# Batched calls.  `mats` is a list of dicts with tensor entries named like the
# fields of maskllm_matrix (W, logits, grad_W_out, logits_out, W_out,
# row_sq_out, probs_out, dlogits_out, values_out, meta_out, idx_out, meta) and
# an optional int tensor_id.  The shape comes from W (bf16 [rows, cols]), or
# from meta (int32 [rows, cols/32]) when there is no W.
# ---------------------------------------------------------------------------

_TENSOR_FIELDS = ("W", "logits", "grad_W_out", "logits_out", "W_out", "row_sq_out",
                  "probs_out", "dlogits_out", "values_out", "meta_out", "idx_out", "meta",
                  "prev_idx", "l1_row_out", "maxprob_row_out")


def matrix_array(mats):
    arr = (maskllm_matrix * len(mats))()
    for a, m in zip(arr, mats):
        W = m.get("W")
        if W is None and m.get("meta") is not None:
            meta = m["meta"]
            if not (isinstance(meta, torch.Tensor) and meta.dtype == torch.int32
                    and meta.dim() == 2):
                raise ValueError("meta must be a 2-D int32 CUDA tensor")
            a.rows, a.cols = meta.shape[0], 32 * meta.shape[1]
        elif W is None and m.get("logits") is not None:
            lg = m["logits"]
            if not (isinstance(lg, torch.Tensor) and lg.dtype == torch.float32
                    and lg.dim() == 3 and lg.shape[2] == 6):
                raise ValueError("logits must be a float32 CUDA tensor [rows, cols/4, 6]")
            a.rows, a.cols = lg.shape[0], 4 * lg.shape[1]
        else:
            if not (isinstance(W, torch.Tensor) and W.is_cuda and W.dtype == torch.bfloat16
                    and W.dim() == 2 and W.is_contiguous()):
                raise ValueError("W must be a contiguous 2-D bf16 CUDA tensor")
            a.rows, a.cols = W.shape
        a.tensor_id = int(m.get("tensor_id", 0))
        for f in _TENSOR_FIELDS:
            t = m.get(f)
            if t is not None:
                if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
                    raise ValueError("%s must be a contiguous CUDA tensor" % f)
                setattr(a, f, t.data_ptr())
    return arr


def maskllm_prior_init_batched(mats, scale, stream=None):
    arr = matrix_array(mats)
    _check("maskllm_prior_init_batched",
           lib().maskllm_prior_init_batched(arr, len(mats), scale, _stream(stream)))


def maskllm_forward_batched(mats, tau, kappa, seed, step, stream=None):
    arr = matrix_array(mats)
    _check("maskllm_forward_batched", lib().maskllm_forward_batched(
        arr, len(mats), tau, kappa, seed, step, _stream(stream)))


def maskllm_backward_batched(mats, tau, kappa, seed, step, reg_coeff=0.0, stream=None):
    arr = matrix_array(mats)
    _check("maskllm_backward_batched", lib().maskllm_backward_batched(
        arr, len(mats), tau, kappa, seed, step, reg_coeff, _stream(stream)))


def maskllm_hard_compress_batched(mats, stream=None):
    arr = matrix_array(mats)
    _check("maskllm_hard_compress_batched",
           lib().maskllm_hard_compress_batched(arr, len(mats), _stream(stream)))


def maskllm_prior_from_mask_batched(mats, high, low, stream=None):
    arr = matrix_array(mats)
    _check("maskllm_prior_from_mask_batched", lib().maskllm_prior_from_mask_batched(
        arr, len(mats), high, low, _stream(stream)))


def maskllm_mask_stats_batched(mats, tau, kappa, seed, step, stream=None):
    """maskllm_mask_stats over a batch: per matrix `logits`, `prev_idx` (u8
    [rows, cols/4], optional) in; `idx_out`, `l1_row_out` (int32 [rows],
    needs prev_idx), `maxprob_row_out` (fp32 [rows]) out, all optional."""
    arr = matrix_array(mats)
    _check("maskllm_mask_stats_batched", lib().maskllm_mask_stats_batched(
        arr, len(mats), tau, kappa, seed, step, _stream(stream)))


def maskllm_forward_stats_batched(mats, tau, kappa, seed, step, stream=None):
    """maskllm_forward_stats over a batch: the forward's fields (`W`,
    `logits`, `W_out`, `row_sq_out`) and the diagnostics' fields of
    maskllm_mask_stats_batched."""
    arr = matrix_array(mats)
    _check("maskllm_forward_stats_batched", lib().maskllm_forward_stats_batched(
        arr, len(mats), tau, kappa, seed, step, _stream(stream)))


def maskllm_backward_stats_batched(mats, tau, kappa, seed, step, reg_coeff=0.0, stream=None):
    """maskllm_backward_stats over a batch: the backward's fields (`W`,
    `logits`, `grad_W_out`, `dlogits_out`) and the diagnostics' fields of
    maskllm_mask_stats_batched."""
    arr = matrix_array(mats)
    _check("maskllm_backward_stats_batched", lib().maskllm_backward_stats_batched(
        arr, len(mats), tau, kappa, seed, step, reg_coeff, _stream(stream)))


def maskllm_set_wait_timeout(nanoseconds: int) -> None:
    _check("maskllm_set_wait_timeout", lib().maskllm_set_wait_timeout(int(nanoseconds)))


def maskllm_test_withhold_loads(enable: bool) -> None:
    _check("maskllm_test_withhold_loads", lib().maskllm_test_withhold_loads(int(bool(enable))))


def maskllm_test_spmm_tile_n(n: int) -> None:
    """Force the sparse product's tile width (128..256, a multiple of 32), or
    restore the per-call choice with 0 (test hook)."""
    _check("maskllm_test_spmm_tile_n", lib().maskllm_test_spmm_tile_n(int(n)))


def maskllm_prior_from_mask(meta, rows, cols, high, low, logits_out=None, stream=None):
    _need(meta, "meta", torch.int32, (rows, cols // 32))
    logits_out = _out(logits_out, "logits_out", torch.float32, (rows, cols // 4, 6), meta)
    _check("maskllm_prior_from_mask", lib().maskllm_prior_from_mask(
        _ptr(meta), rows, cols, high, low, _ptr(logits_out), _stream(stream)))
    return logits_out


def maskllm_mask_stats(logits, tau, kappa, rng, prev_idx=None, idx_out=None, want_idx=True,
                       want_l1=None, want_maxprob=True, stream=None):
    """Returns (idx u8 [rows, cols/4] | None, l1 int32 [rows] | None, maxprob f32 [rows] | None).
    The L1 row sums are uint32 values carried in an int32 tensor."""
    rows, g, six = logits.shape
    cols = 4 * g
    _need(logits, "logits", torch.float32, (rows, g, 6))
    if prev_idx is not None:
        _need(prev_idx, "prev_idx", torch.uint8, (rows, g))
    if idx_out is None and want_idx:
        idx_out = torch.empty((rows, g), dtype=torch.uint8, device=logits.device)
    elif idx_out is not None:
        _need(idx_out, "idx_out", torch.uint8, (rows, g))
    if want_l1 is None:
        want_l1 = prev_idx is not None
    l1 = torch.empty((rows,), dtype=torch.int32, device=logits.device) if want_l1 else None
    mp = torch.empty((rows,), dtype=torch.float32, device=logits.device) if want_maxprob else None
    _check("maskllm_mask_stats", lib().maskllm_mask_stats(
        _ptr(logits), _ptr(prev_idx), rows, cols, tau, kappa, _rng(rng), _ptr(idx_out), _ptr(l1),
        _ptr(mp), _stream(stream)))
    return idx_out, l1, mp


# ---------------------------------------------------------------------------
# channel permutation before pruning
# ---------------------------------------------------------------------------

def _perm(perm, cols):
    return _need(perm, "perm", torch.int32, (cols,))


def maskllm_perm_shift(W, stream=None):
    """int32 [1] device tensor: the fixed-point shift of W (INT32_MIN if W is
    not finite)."""
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    out = torch.empty((4,), dtype=torch.int32, device=W.device)   # 16-byte slot
    _check("maskllm_perm_shift", lib().maskllm_perm_shift(_ptr(W), rows, cols, _ptr(out),
                                                          _stream(stream)))
    return out[:1]


def maskllm_perm_metric(W, perm, shift, stream=None):
    """int64 [1] device tensor: the fixed-point kept magnitude of perm."""
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _perm(perm, cols)
    out = torch.empty((2,), dtype=torch.int64, device=W.device)
    _check("maskllm_perm_metric", lib().maskllm_perm_metric(
        _ptr(W), rows, cols, _ptr(perm), _ptr(shift), _ptr(out), _stream(stream)))
    return out[:1]


def maskllm_permute_columns(W, perm, W_out=None, stream=None):
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _perm(perm, cols)
    W_out = _out(W_out, "W_out", torch.bfloat16, (rows, cols), W)
    _check("maskllm_permute_columns", lib().maskllm_permute_columns(
        _ptr(W), rows, cols, _ptr(perm), _ptr(W_out), _stream(stream)))
    return W_out


def maskllm_perm_workspace_bytes(rows: int, cols: int) -> int:
    return int(lib().maskllm_perm_workspace_bytes(rows, cols))


def _workspace(workspace, rows, cols, like):
    need = maskllm_perm_workspace_bytes(rows, cols)
    if need <= 0:
        raise MaskLLMError("maskllm_perm_workspace_bytes", 2)
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=like.device)
    return workspace


def maskllm_perm_swap_gains(W, perm, workspace=None, stream=None):
    """Returns (gains int64 [cols, cols], info int32 [1], shift int32 [1])."""
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _perm(perm, cols)
    workspace = _workspace(workspace, rows, cols, W)
    gains = torch.empty((cols, cols), dtype=torch.int64, device=W.device)
    small = torch.zeros((8,), dtype=torch.int32, device=W.device)   # info, shift in 16-byte slots
    _check("maskllm_perm_swap_gains", lib().maskllm_perm_swap_gains(
        _ptr(W), rows, cols, _ptr(perm), _ptr(workspace), workspace.numel(), _ptr(gains),
        _ptr(small), small.data_ptr() + 16, _stream(stream)))
    return gains, small[0:1], small[4:5]


def maskllm_perm_search(W, perm, max_swaps, workspace=None, log=True, stream=None):
    """Steepest-ascent channel-swap search; perm (int32 [cols], device) is
    updated in place.  Returns (n_swaps int32 [1], swaps int32 [max_swaps, 2]
    | None, gains int64 [max_swaps] | None, shift int32 [1])."""
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _perm(perm, cols)
    workspace = _workspace(workspace, rows, cols, W)
    m = max(int(max_swaps), 1)
    swaps = torch.zeros((m, 2), dtype=torch.int32, device=W.device) if log else None
    gains = torch.zeros((m,), dtype=torch.int64, device=W.device) if log else None
    small = torch.zeros((8,), dtype=torch.int32, device=W.device)   # n_swaps, shift
    _check("maskllm_perm_search", lib().maskllm_perm_search(
        _ptr(W), rows, cols, _ptr(perm), int(max_swaps), _ptr(workspace), workspace.numel(),
        _ptr(swaps), _ptr(gains), _ptr(small), small.data_ptr() + 16, _stream(stream)))
    return small[0:1], swaps, gains, small[4:5]


def maskllm_perm_search_static(W, perm, max_swaps, log=True, stream=None):
    """maskllm_perm_search with its scratch in the library's own device array
    (no allocation by the caller or the library); same results.  Returns
    (n_swaps int32 [1], swaps | None, gains | None, shift int32 [1]).  The
    result tensors here are allocated by torch for convenience; a caller that
    cannot allocate passes its own buffers to the C function."""
    rows, cols = W.shape
    _need(W, "W", torch.bfloat16, (rows, cols))
    _perm(perm, cols)
    m = max(int(max_swaps), 1)
    swaps = torch.zeros((m, 2), dtype=torch.int32, device=W.device) if log else None
    gains = torch.zeros((m,), dtype=torch.int64, device=W.device) if log else None
    small = torch.zeros((8,), dtype=torch.int32, device=W.device)
    _check("maskllm_perm_search_static", lib().maskllm_perm_search_static(
        _ptr(W), rows, cols, _ptr(perm), int(max_swaps), _ptr(swaps), _ptr(gains), _ptr(small),
        small.data_ptr() + 16, _stream(stream)))
    return small[0:1], swaps, gains, small[4:5]


# ---------------------------------------------------------------------------
# 2:4 sparse x dense product
# ---------------------------------------------------------------------------

def maskllm_spmm(values, meta, B, C=None, stream=None):
    """C [M, N] fp32 = A B^T with A given as maskllm_hard_compress output
    (values bf16 [M, K/2], meta int32 [M, K/32]) and B bf16 [N, K]."""
    M, half = values.shape
    K = 2 * half
    N = B.shape[0]
    _need(values, "values", torch.bfloat16, (M, half))
    _need(meta, "meta", torch.int32, (M, K // 32))
    _need(B, "B", torch.bfloat16, (N, K))
    C = _out(C, "C", torch.float32, (M, N), values)
    _check("maskllm_spmm", lib().maskllm_spmm(_ptr(values), _ptr(meta), M, K, _ptr(B), N, _ptr(C),
                                              _stream(stream)))
    return C


def maskllm_forward_stats(W, logits, tau, kappa, rng, prev_idx=None, W_out=None, want_row_sq=True,
                          want_idx=True, want_l1=None, want_maxprob=True, stream=None):
    """The forward and the step's diagnostics in one pass.  Returns (W_out,
    row_sq | None, idx | None, l1 int32 | None, maxprob | None); l1 holds
    uint32 values in an int32 tensor."""
    rows, cols = W.shape
    g = cols // 4
    _need(W, "W", torch.bfloat16, (rows, cols))
    _need(logits, "logits", torch.float32, (rows, g, 6))
    if prev_idx is not None:
        _need(prev_idx, "prev_idx", torch.uint8, (rows, g))
    W_out = _out(W_out, "W_out", torch.bfloat16, (rows, cols), W)
    dev = W.device
    row_sq = torch.empty((rows,), dtype=torch.float32, device=dev) if want_row_sq else None
    idx = torch.empty((rows, g), dtype=torch.uint8, device=dev) if want_idx else None
    if want_l1 is None:
        want_l1 = prev_idx is not None
    l1 = torch.empty((rows,), dtype=torch.int32, device=dev) if want_l1 else None
    mp = torch.empty((rows,), dtype=torch.float32, device=dev) if want_maxprob else None
    _check("maskllm_forward_stats", lib().maskllm_forward_stats(
        _ptr(W), _ptr(logits), _ptr(prev_idx), rows, cols, tau, kappa, _rng(rng), _ptr(W_out),
        _ptr(row_sq), _ptr(idx), _ptr(l1), _ptr(mp), _stream(stream)))
    return W_out, row_sq, idx, l1, mp


def maskllm_backward_stats(W, logits, grad_W_out, tau, kappa, rng, reg_coeff=0.0, prev_idx=None,
                           dlogits_out=None, want_idx=True, want_l1=None, want_maxprob=True,
                           stream=None):
    """The backward and the step's diagnostics in one pass.  Returns
    (dlogits, idx | None, l1 int32 | None, maxprob | None); l1 holds uint32
    values in an int32 tensor."""
    rows, cols = W.shape
    g = cols // 4
    _need(W, "W", torch.bfloat16, (rows, cols))
    _need(logits, "logits", torch.float32, (rows, g, 6))
    _need(grad_W_out, "grad_W_out", torch.bfloat16, (rows, cols))
    if prev_idx is not None:
        _need(prev_idx, "prev_idx", torch.uint8, (rows, g))
    dlogits_out = _out(dlogits_out, "dlogits_out", torch.float32, (rows, g, 6), W)
    dev = W.device
    idx = torch.empty((rows, g), dtype=torch.uint8, device=dev) if want_idx else None
    if want_l1 is None:
        want_l1 = prev_idx is not None
    l1 = torch.empty((rows,), dtype=torch.int32, device=dev) if want_l1 else None
    mp = torch.empty((rows,), dtype=torch.float32, device=dev) if want_maxprob else None
    _check("maskllm_backward_stats", lib().maskllm_backward_stats(
        _ptr(W), _ptr(logits), _ptr(grad_W_out), _ptr(prev_idx), rows, cols, tau, kappa,
        _rng(rng), reg_coeff, _ptr(dlogits_out), _ptr(idx), _ptr(l1), _ptr(mp), _stream(stream)))
    return dlogits_out, idx, l1, mp
