"""The C-ABI library builds, loads, exports every entry point of
include/maskllm.h, and rejects bad arguments on the host (no GPU needed: every
case here fails validation before any CUDA call)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "maskllm.h")

OK, INVALID, SHAPE, ALIGN, ALIAS = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    from semi_structured_sparsity_gb300 import _build, binding
    _build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(maskllm_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    from semi_structured_sparsity_gb300 import binding
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(binding.EXPORTS)


def test_status_strings(L):
    from semi_structured_sparsity_gb300 import binding
    for code, name in binding.STATUS.items():
        assert L.maskllm_status_string(code).decode() == name
    assert L.maskllm_last_cuda_error().decode() == ""


def _rng():
    from semi_structured_sparsity_gb300 import binding
    return binding.maskllm_rng(0, 0, 0)


# Fake, never-dereferenced device addresses: validation looks only at values.
A, B, Cc, D, E = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000


def test_forward_validation(L):
    r = _rng()
    f = L.maskllm_forward
    assert f(None, B, 4, 64, 1.0, 1.0, r, Cc, None, None, None) == INVALID
    assert f(A, B, 4, 64, 1.0, 1.0, r, None, None, None, None) == INVALID
    assert f(A + 8, B, 4, 64, 1.0, 1.0, r, Cc, None, None, None) == ALIGN
    assert f(A, B, 4, 64, 1.0, 1.0, r, Cc, D + 4, None, None) == ALIGN
    assert f(A, B, 0, 64, 1.0, 1.0, r, Cc, None, None, None) == SHAPE
    assert f(A, B, 4, 48, 1.0, 1.0, r, Cc, None, None, None) == SHAPE
    assert f(A, B, 4, 0, 1.0, 1.0, r, Cc, None, None, None) == SHAPE
    assert f(A, B, -1, 64, 1.0, 1.0, r, Cc, None, None, None) == SHAPE
    assert f(A, B, 1 << 40, 1 << 10, 1.0, 1.0, r, Cc, None, None, None) == SHAPE
    for tau in (0.0, -1.0, float("inf"), float("nan"), 1e-45):
        assert f(A, B, 4, 64, tau, 1.0, r, Cc, None, None, None) == INVALID, tau
    assert f(A, B, 4, 64, 1.0, float("nan"), r, Cc, None, None, None) == INVALID
    # W_out overlapping W; row_sq overlapping logits; probs overlapping W_out
    assert f(A, B, 4, 64, 1.0, 1.0, r, A + 256, None, None, None) == ALIAS
    assert f(A, B, 4, 64, 1.0, 1.0, r, Cc, B + 16, None, None) == ALIAS
    assert f(A, B, 4, 64, 1.0, 1.0, r, Cc, None, Cc + 64, None) == ALIAS


def test_backward_validation(L):
    r = _rng()
    f = L.maskllm_backward
    assert f(A, B, None, 4, 64, 1.0, 1.0, r, 0.0, D, None) == INVALID
    assert f(A, B, Cc, 4, 64, 1.0, 1.0, r, float("inf"), D, None) == INVALID
    assert f(A, B, Cc, 4, 33, 1.0, 1.0, r, 0.0, D, None) == SHAPE
    assert f(A, B, Cc, 4, 64, 1.0, 1.0, r, 0.0, D + 2, None) == ALIGN
    # dlogits (4*64*6 bytes) starting inside G
    assert f(A, B, Cc, 4, 64, 1.0, 1.0, r, 0.0, Cc + 64, None) == ALIAS
    # adjacent but not overlapping is fine up to the CUDA call; use a distinct
    # region to confirm the alias check itself accepts it: the next failure
    # would be a CUDA error, which needs a device -- so stop at validation.


def test_compress_and_other_validation(L):
    r = _rng()
    assert L.maskllm_hard_compress(A, B, 4, 64, Cc, None, None, None) == INVALID
    assert L.maskllm_hard_compress(A, B, 4, 64, Cc, D, E + 1, None) == ALIGN
    assert L.maskllm_hard_compress(A, B, 4, 64, Cc, Cc + 16, None, None) == ALIAS
    assert L.maskllm_hard_compress(A, B, 4, 64, Cc, D, A, None) == ALIAS
    assert L.maskllm_decompress(A, B, 4, 64, A, None) == ALIAS
    assert L.maskllm_decompress(A, B, 4, 16, Cc, None) == SHAPE
    assert L.maskllm_prior_init(A, 4, 64, float("nan"), B, None) == INVALID
    assert L.maskllm_prior_init(A, 4, 64, 1.0, A + 32, None) == ALIAS
    assert L.maskllm_noise_words(r, -1, 4, A, None) == INVALID
    assert L.maskllm_noise_words(r, 0, 0, A, None) == INVALID
    assert L.maskllm_noise_words(r, 0, 4, A + 4, None) == ALIGN


def test_binding_refuses_host_tensors(L):
    torch = pytest.importorskip("torch")
    from semi_structured_sparsity_gb300 import binding
    W = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.maskllm_prior_init(W, 1.0)


def _mat(**kw):
    from semi_structured_sparsity_gb300 import binding
    m = binding.maskllm_matrix()
    m.rows, m.cols = kw.pop("rows", 4), kw.pop("cols", 64)
    for k, v in kw.items():
        setattr(m, k, v)
    return m


def test_batched_validation(L):
    from semi_structured_sparsity_gb300 import binding
    arr = (binding.maskllm_matrix * 3)()
    assert L.maskllm_forward_batched(arr, 0, 1.0, 1.0, 0, 0, None) == INVALID
    assert L.maskllm_forward_batched(None, 1, 1.0, 1.0, 0, 0, None) == INVALID
    # matrix 1 is missing its output
    arr[0] = _mat(W=A, logits=B, W_out=Cc)
    arr[1] = _mat(W=D, logits=E)
    assert L.maskllm_forward_batched(arr, 2, 1.0, 1.0, 0, 0, None) == INVALID
    # matrix 1 writes over matrix 0's logits
    arr[1] = _mat(W=D, logits=E, W_out=B + 64)
    assert L.maskllm_forward_batched(arr, 2, 1.0, 1.0, 0, 0, None) == ALIAS
    arr[1] = _mat(W=D, logits=E, W_out=0x600000, rows=4, cols=40)
    assert L.maskllm_forward_batched(arr, 2, 1.0, 1.0, 0, 0, None) == SHAPE
    assert L.maskllm_backward_batched(arr, 1, 1.0, 1.0, 0, 0, 0.0, None) == INVALID
    assert L.maskllm_forward_batched(arr, 1, -1.0, 1.0, 0, 0, None) == INVALID


def test_batched_alias_across_launches(L):
    from semi_structured_sparsity_gb300 import binding
    n = 20   # more than one launch's worth
    arr = (binding.maskllm_matrix * n)()
    base = 0x10000000
    for i in range(n):
        off = base + i * 0x100000
        arr[i] = _mat(W=off, logits_out=off + 0x10000)
    arr[19].logits_out = base + 0x10        # writes over matrix 0's W, in another launch
    assert L.maskllm_prior_init_batched(arr, n, 1.0, None) == ALIAS


def test_prior_from_mask_batched_validation(L):
    from semi_structured_sparsity_gb300 import binding
    arr = (binding.maskllm_matrix * 2)()
    arr[0] = _mat(logits_out=B)
    arr[0].meta = A
    arr[1] = _mat(logits_out=D)               # no codes
    assert L.maskllm_prior_from_mask_batched(arr, 2, 1.0, 0.0, None) == INVALID
    arr[1].meta = E
    assert L.maskllm_prior_from_mask_batched(arr, 2, float("nan"), 0.0, None) == INVALID
    arr[1].logits_out = A + 16                # writes over matrix 0's codes
    assert L.maskllm_prior_from_mask_batched(arr, 2, 1.0, 0.0, None) == ALIAS
    arr[1].logits_out = D + 4                 # misaligned output
    assert L.maskllm_prior_from_mask_batched(arr, 2, 1.0, 0.0, None) == ALIGN
    arr[1] = _mat(logits_out=D, rows=4, cols=40)
    arr[1].meta = E
    assert L.maskllm_prior_from_mask_batched(arr, 2, 1.0, 0.0, None) == SHAPE


def test_diagnostics_batched_validation(L):
    from semi_structured_sparsity_gb300 import binding
    arr = (binding.maskllm_matrix * 2)()
    arr[0] = _mat(logits=A, idx_out=B)
    arr[1] = _mat(logits=D, maxprob_row_out=E)
    for fn in (L.maskllm_mask_stats_batched, L.maskllm_forward_stats_batched):
        assert fn(arr, 0, 1.0, 1.0, 0, 0, None) == INVALID
        assert fn(None, 1, 1.0, 1.0, 0, 0, None) == INVALID
        assert fn(arr, 2, 0.0, 1.0, 0, 0, None) == INVALID              # tau <= 0
        assert fn(arr, 2, 1.0, float("inf"), 0, 0, None) == INVALID     # kappa not finite
    # the L1 distance needs the previous draws
    arr[1] = _mat(logits=D, l1_row_out=E)
    assert L.maskllm_mask_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == INVALID
    arr[1].prev_idx = Cc
    arr[1].l1_row_out = Cc + 4                # misaligned output
    assert L.maskllm_mask_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == ALIGN
    arr[1].l1_row_out = A + 32                # writes over matrix 0's logits
    assert L.maskllm_mask_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == ALIAS
    arr[1] = _mat(logits=D, maxprob_row_out=E, rows=1, cols=(1 << 24) + 32)
    assert L.maskllm_mask_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == SHAPE
    # the fused pass also needs W and W_out
    arr[1] = _mat(logits=D, maxprob_row_out=E)
    assert L.maskllm_forward_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == INVALID
    arr[0] = _mat(W=0x700000, logits=A, W_out=0x710000, idx_out=B)
    arr[1] = _mat(W=0x720000, logits=D, W_out=0x730000, row_sq_out=0x730000 + 16)
    assert L.maskllm_forward_stats_batched(arr, 2, 1.0, 1.0, 0, 0, None) == ALIAS


def test_full_batch_of_fused_diagnostics_validates_every_span(L):
    # 16 matrices x (3 inputs + 5 outputs): validation records every span
    # and finds the alias between the last matrix and the first
    from semi_structured_sparsity_gb300 import binding
    n = binding.MAX_BATCH
    arr = (binding.maskllm_matrix * n)()
    base = 0x10000000
    for i in range(n):
        o = base + i * 0x100000
        arr[i] = _mat(W=o, logits=o + 0x1000, prev_idx=o + 0x2000, W_out=o + 0x3000,
                      row_sq_out=o + 0x4000, idx_out=o + 0x5000, l1_row_out=o + 0x6000,
                      maxprob_row_out=o + 0x7000)
    arr[n - 1].maxprob_row_out = base + 0x3000   # over matrix 0's W_out
    assert L.maskllm_forward_stats_batched(arr, n, 1.0, 1.0, 0, 0, None) == ALIAS


def test_backward_stats_validation(L):
    from semi_structured_sparsity_gb300 import binding
    r = _rng()
    bs = L.maskllm_backward_stats
    # W, logits, grad_W_out, prev_idx, rows, cols, tau, kappa, rng, reg, dlogits, idx, l1, maxprob
    assert bs(A, B, None, None, 4, 64, 1.0, 1.0, r, 0.0, Cc, None, None, None, None) == INVALID
    assert bs(A, B, D, None, 4, 64, 1.0, 1.0, r, 0.0, None, None, None, None, None) == INVALID
    assert bs(A, B, D, None, 4, 64, 1.0, 1.0, r, 0.0, Cc, None, E, None, None) == INVALID  # L1, no prev
    assert bs(A, B, D, None, 4, 64, 0.0, 1.0, r, 0.0, Cc, None, None, None, None) == INVALID
    assert bs(A, B, D, None, 4, 64, 1.0, 1.0, r, float("nan"), Cc, None, None, None, None) == INVALID
    assert bs(A, B, D, None, 1, (1 << 24) + 32, 1.0, 1.0, r, 0.0, Cc, None, None, None, E) == SHAPE
    assert bs(A, B, D, E + 8, 4, 64, 1.0, 1.0, r, 0.0, Cc, None, None, None, None) == ALIGN
    assert bs(A, B, D, E, 4, 64, 1.0, 1.0, r, 0.0, Cc, A + 32, None, None, None) == ALIAS
    arr = (binding.maskllm_matrix * 2)()
    arr[0] = _mat(W=A, logits=B, grad_W_out=D, dlogits_out=Cc)
    arr[1] = _mat(W=A + 0x1000, logits=B + 0x1000, grad_W_out=D + 0x1000, dlogits_out=Cc + 0x1000,
                  l1_row_out=E)
    bb = L.maskllm_backward_stats_batched
    assert bb(arr, 2, 1.0, 1.0, 0, 0, 0.0, None) == INVALID            # L1 without prev
    arr[1].prev_idx = E + 0x100
    arr[1].maxprob_row_out = Cc + 16                                    # over matrix 0's dlogits
    assert bb(arr, 2, 1.0, 1.0, 0, 0, 0.0, None) == ALIAS


def test_next_entry_points_validation(L):
    r = _rng()
    assert L.maskllm_prior_from_mask(A, 4, 64, float("inf"), 0.0, B, None) == INVALID
    assert L.maskllm_prior_from_mask(A, 4, 48, 1.0, 0.0, B, None) == SHAPE
    assert L.maskllm_prior_from_mask(A, 4, 64, 1.0, 0.0, A + 16, None) == ALIAS
    # the L1 distance needs the previous draws; cols above 2^24; tau <= 0
    assert L.maskllm_mask_stats(A, None, 4, 64, 1.0, 1.0, r, None, B, None, None) == INVALID
    assert L.maskllm_mask_stats(A, None, 1, (1 << 24) + 32, 1.0, 1.0, r, None, None, Cc, None) == SHAPE
    assert L.maskllm_mask_stats(A, None, 4, 64, 0.0, 1.0, r, None, None, Cc, None) == INVALID
    assert L.maskllm_mask_stats(A, None, 4, 64, 1.0, 1.0, r, A + 64, None, None, None) == ALIAS


def test_permutation_entry_points_validation(L):
    ws = L.maskllm_perm_workspace_bytes(64, 128)
    assert ws == 128 * 128 * 4 + 2 * 64 * 128 * 4 + 256 + 256 + 128 // 8   # 10 tiles: 80 B
    assert L.maskllm_perm_workspace_bytes(64, 48) == 0            # cols % 32
    assert L.maskllm_perm_workspace_bytes(64, 32768 + 32) == 0    # cols above 32768
    assert L.maskllm_perm_workspace_bytes((1 << 24) + 1, 32) == 0
    big = 0x40000000
    # shift / metric / permute: null, alignment, shape, alias
    assert L.maskllm_perm_shift(A, 4, 64, None, None) == INVALID
    assert L.maskllm_perm_shift(A, 4, 64, B + 4, None) == ALIGN
    assert L.maskllm_perm_shift(A, 4, 64, A + 16, None) == ALIAS
    assert L.maskllm_perm_metric(A, 4, 64, B, Cc, None, None) == INVALID
    assert L.maskllm_perm_metric(A, 4, 64, B, Cc, B + 16, None) == ALIAS
    assert L.maskllm_permute_columns(A, 4, 64, B, A, None) == ALIAS
    assert L.maskllm_permute_columns(A, 4, 65536, B, Cc, None) == SHAPE
    # gains: workspace too small, info missing, gains over the workspace
    assert L.maskllm_perm_swap_gains(A, 64, 128, B, big, ws - 1, Cc, D, None, None) == INVALID
    assert L.maskllm_perm_swap_gains(A, 64, 128, B, big, ws, Cc, None, None, None) == INVALID
    assert L.maskllm_perm_swap_gains(A, 64, 128, B, big, ws, big + 64, D, None, None) == ALIAS
    # search: negative max_swaps, perm inside W, logs over each other
    assert L.maskllm_perm_search(A, 64, 128, B, -1, big, ws, None, None, D, None, None) == INVALID
    assert L.maskllm_perm_search(A, 64, 128, A + 16, 5, big, ws, None, None, D, None, None) == ALIAS
    assert L.maskllm_perm_search(A, 64, 128, B, 5, big, ws, Cc, Cc + 16, D, None, None) == ALIAS
    assert L.maskllm_perm_search(A, 64, 128, B, 5, big, ws, Cc + 8, None, D, None, None) == ALIGN


def test_no_alloc_search_validation(L):
    # the library-held scratch holds cols = 1024 up to 3583 rows
    assert L.maskllm_perm_search_static(A, 3584, 1024, B, 5, None, None, D, None, None) == SHAPE
    assert L.maskllm_perm_search_static(A, 64, 4096, B, 5, None, None, D, None, None) == SHAPE
    assert L.maskllm_perm_search_static(A, 64, 128, B, -1, None, None, D, None, None) == INVALID
    assert L.maskllm_perm_search_static(A, 64, 128, None, 5, None, None, D, None, None) == INVALID
    assert L.maskllm_perm_search_static(A, 64, 128, A + 16, 5, None, None, D, None, None) == ALIAS
    assert L.maskllm_perm_search_static(A, 64, 128, B, 5, Cc + 8, None, D, None, None) == ALIGN


def test_spmm_validation(L):
    assert L.maskllm_spmm(A, B, 128, 64, Cc, 256, None, None) == INVALID
    assert L.maskllm_spmm(A, B, 128, 48, Cc, 256, D, None) == SHAPE       # K % 32
    assert L.maskllm_spmm(A, B, 0, 64, Cc, 256, D, None) == SHAPE
    assert L.maskllm_spmm(A, B, 128, 64, Cc, 0, D, None) == SHAPE
    assert L.maskllm_spmm(A, B, 128, 64, Cc, 65535 * 256 + 1, D, None) == SHAPE   # grid y
    assert L.maskllm_spmm(A + 8, B, 128, 64, Cc, 256, D, None) == ALIGN
    assert L.maskllm_spmm(A, B, 128, 64, Cc, 256, Cc + 64, None) == ALIAS  # C over B


def test_spmm_tile_hook_validation(L):
    for n in (100, 129, 288, -32, 96):
        assert L.maskllm_test_spmm_tile_n(n) == INVALID
    for n in (128, 160, 192, 224, 256, 0):
        assert L.maskllm_test_spmm_tile_n(n) == 0


def test_forward_stats_validation(L):
    r = _rng()
    f = L.maskllm_forward_stats
    assert f(A, B, None, 4, 64, 1.0, 1.0, r, None, None, None, None, None, None) == INVALID
    assert f(A, B, None, 4, 64, 1.0, 1.0, r, Cc, None, None, D, None, None) == INVALID   # L1 needs prev
    assert f(A, B, None, 1, (1 << 24) + 32, 1.0, 1.0, r, Cc, None, None, None, None, None) == SHAPE
    assert f(A, B, None, 4, 64, 0.0, 1.0, r, Cc, None, None, None, None, None) == INVALID
    assert f(A, B, None, 4, 64, 1.0, 1.0, r, A + 16, None, None, None, None, None) == ALIAS
    assert f(A, B, None, 4, 64, 1.0, 1.0, r, Cc, D + 4, None, None, None, None) == ALIGN
