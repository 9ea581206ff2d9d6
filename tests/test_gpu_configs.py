"""GPU parity on the five workloads at full size, in the launch configuration
the benchmark times (batched launches over each block's matrices).

Where the oracle cannot redo a whole workload in seconds, it recomputes
sampled rows (every 64th row plus the last row of each matrix; for the
32-layer workloads all sampled rows of the first and last layer and the first
and last row of every matrix of every other layer), and properties that hold
at any size are checked on every element.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as W
from tests._helpers import (assert_bf16_ulps, assert_bits_equal, assert_close, bits16, bits32,
                            sampled_rows, ROWSQ_RTOL)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# keep-mask of each candidate over the 4 positions (lexicographic kept pairs)
PAIRS = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


def _alloc_block(wl, layer, need=("fwd", "bwd"), keep_noise=True):
    """Inputs and outputs of one layer's matrices (logits built as the bench does)."""
    mats = []
    for m, (name, rows, cols) in enumerate(wl.matrices):
        x = W.matrix_inputs(wl, layer, m, device="cuda")
        if x.L is None:
            x.L = mk.maskllm_prior_init(x.W, wl.prior_scale) + x.L_noise
            if not keep_noise:
                x.L_noise = None
        d = {"x": x, "W": x.W, "logits": x.L, "grad_W_out": x.G, "tensor_id": x.tensor_id}
        if "fwd" in need:
            d["W_out"] = torch.empty_like(x.W)
            d["row_sq_out"] = torch.empty((rows,), device="cuda")
        if "bwd" in need:
            d["dlogits_out"] = torch.empty_like(x.L)
        if "cmp" in need:
            d["values_out"] = torch.empty((rows, cols // 2), dtype=torch.bfloat16, device="cuda")
            d["meta_out"] = torch.empty((rows, cols // 32), dtype=torch.int32, device="cuda")
            d["idx_out"] = torch.empty((rows, cols // 4), dtype=torch.uint8, device="cuda")
        mats.append(d)
    return mats


def _check_rows(wl, d, rows_to_check, step=0, check_prior=True, fwd=True, bwd=True):
    x = d["x"]
    idx = torch.tensor(rows_to_check, device="cuda")
    Wr = bits16(x.W[idx])
    Lr_gpu = x.L[idx].cpu().numpy()
    if x.L_noise is not None and check_prior:
        # the logits were built on the GPU from our prior kernel + noise; the
        # oracle builds its own from W and the same noise
        Lr = orc.prior_init(Wr, wl.prior_scale) + x.L_noise[idx].cpu().numpy()
        assert_bits_equal(Lr_gpu.view(np.uint32), Lr.astype(np.float32).view(np.uint32),
                          "prior + noise logits")
    for k, r in enumerate(rows_to_check):
        Wb, Lh = Wr[k:k + 1], Lr_gpu[k:k + 1]
        if fwd:
            wW, wsq, _, _ = orc.forward(Wb, Lh, wl.tau, wl.kappa, 0, step, x.tensor_id,
                                        row_begin=r)
            assert_bf16_ulps(bits16(d["W_out"][r:r + 1]), wW, what="W' row %d" % r)
            assert_close(d["row_sq_out"][r:r + 1].cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0,
                         what="row_sq row %d" % r)
        if bwd:
            Gb = bits16(x.G[r:r + 1])
            want = orc.backward(Wb, Lh, Gb, wl.tau, wl.kappa, 0, step, x.tensor_id,
                                row_begin=r)
            assert_close(d["dlogits_out"][r:r + 1].cpu().numpy(), want,
                         what="dlogits row %d" % r)


def _full_properties(d):
    """|W'| <= |W| with the sign kept (M in [0, 1]) on every element."""
    w = d["W"].float()
    wo = d["W_out"].float()
    assert bool((wo.abs() <= w.abs()).all())
    assert bool(((wo == 0) | (torch.sign(wo) == torch.sign(w))).all())


def test_single_layer_full():
    wl = W.WORKLOADS["single"]
    mats = _alloc_block(wl, 0, need=("fwd", "bwd", "cmp"))
    d = mats[0]
    d["probs_out"] = torch.empty_like(d["logits"])
    d["logits_out"] = torch.empty_like(d["logits"])
    mk.maskllm_prior_init_batched(mats, 300.0)
    mk.maskllm_forward_batched(mats, wl.tau, wl.kappa, 0, 0)
    mk.maskllm_backward_batched(mats, wl.tau, wl.kappa, 0, 0)
    mk.maskllm_hard_compress_batched(mats)
    torch.cuda.synchronize()
    Wb, Lh, Gb = bits16(d["W"]), d["logits"].cpu().numpy(), bits16(d["grad_W_out"])
    wW, wsq, wp, _ = orc.forward(Wb, Lh, wl.tau, wl.kappa, 0, 0, d["tensor_id"], want_probs=True)
    assert_bf16_ulps(bits16(d["W_out"]), wW)
    assert_close(d["probs_out"].cpu().numpy(), wp, what="p")
    assert_close(d["row_sq_out"].cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
    assert_close(d["dlogits_out"].cpu().numpy(),
                 orc.backward(Wb, Lh, Gb, wl.tau, wl.kappa, 0, 0, d["tensor_id"]),
                 what="dlogits")
    wv, wm, wi = orc.hard_compress(Wb, Lh)
    assert_bits_equal(bits16(d["values_out"]), wv, "values")
    assert_bits_equal(bits32(d["meta_out"]), wm, "meta")
    assert_bits_equal(d["idx_out"].cpu().numpy(), wi, "idx")
    assert_bits_equal(bits32(d["logits_out"]), orc.prior_init(Wb, 300.0).view(np.uint32),
                      "prior")


def test_llama2_7b_block_full_size():
    wl = W.WORKLOADS["llama2_7b_block"]
    mats = _alloc_block(wl, 0, need=("fwd", "bwd", "cmp"))
    mk.maskllm_forward_batched(mats, wl.tau, wl.kappa, 0, 3)
    mk.maskllm_backward_batched(mats, wl.tau, wl.kappa, 0, 3)
    mk.maskllm_hard_compress_batched(mats)
    torch.cuda.synchronize()
    assert mk.maskllm_device_status() == 0
    for d in mats:
        rows = d["W"].shape[0]
        _check_rows(wl, d, sampled_rows(rows), step=3)
        _full_properties(d)
        wv, wm, _ = orc.hard_compress(bits16(d["W"]), d["logits"].cpu().numpy())
        assert_bits_equal(bits16(d["values_out"]), wv, "values")
        assert_bits_equal(bits32(d["meta_out"]), wm, "meta")


def test_llama2_7b_all_layers_resident_logits():
    """32 layers x 7 matrices (6.5e9 weights), all logits and dlogits resident;
    one forward + backward mask step over every layer."""
    wl = W.WORKLOADS["llama2_7b_full"]
    ends = (0, wl.layers - 1)
    layers = [_alloc_block(wl, layer, keep_noise=layer in ends) for layer in range(wl.layers)]
    every = [d for blk in layers for d in blk]
    assert sum(d["W"].numel() for d in every) == 6_476_005_376
    mk.maskllm_forward_batched(every, wl.tau, wl.kappa, 0, 0)
    mk.maskllm_backward_batched(every, wl.tau, wl.kappa, 0, 0)
    torch.cuda.synchronize()
    assert mk.maskllm_device_status() == 0
    for layer, blk in enumerate(layers):
        for d in blk:
            rows = d["W"].shape[0]
            pick = sampled_rows(rows) if layer in ends else [0, rows - 1]
            _check_rows(wl, d, pick, check_prior=layer in ends)
    del layers, every
    torch.cuda.empty_cache()


def test_nemotron4_15b_layer_by_layer():
    wl = W.WORKLOADS["nemotron4_15b"]
    total = 0
    for layer in range(wl.layers):
        blk = _alloc_block(wl, layer)
        total += sum(d["W"].numel() for d in blk)
        mk.maskllm_forward_batched(blk, wl.tau, wl.kappa, 0, 0)
        mk.maskllm_backward_batched(blk, wl.tau, wl.kappa, 0, 0)
        torch.cuda.synchronize()
        for d in blk:
            rows = d["W"].shape[0]
            pick = sampled_rows(rows) if layer in (0, wl.layers - 1) else [0, rows - 1]
            _check_rows(wl, d, pick)
            if layer == 0:
                _full_properties(d)
        del blk
    assert total == 12_482_248_704
    assert mk.maskllm_device_status() == 0
    torch.cuda.empty_cache()


def test_compress_7b_near_one_hot_full_bit_exact():
    """Every value and code of the whole block against the oracle, including
    the 1% of groups whose two top logits are exactly equal (lowest index
    wins); and the tau -> 0 companion forward."""
    wl = W.WORKLOADS["compress_7b"]
    mats = _alloc_block(wl, 0, need=("fwd", "cmp"))
    mk.maskllm_hard_compress_batched(mats)
    mk.maskllm_forward_batched(mats, wl.tau, wl.kappa, 0, 0)
    torch.cuda.synchronize()
    n_ties = 0
    for d in mats:
        L = d["logits"]
        top2 = torch.topk(L, 2, dim=-1).values
        tie = top2[..., 0] == top2[..., 1]
        n_ties += int(tie.sum())
        wv, wm, wi = orc.hard_compress(bits16(d["W"]), L.cpu().numpy())
        assert_bits_equal(bits16(d["values_out"]), wv, "values")
        assert_bits_equal(bits32(d["meta_out"]), wm, "meta")
        assert_bits_equal(d["idx_out"].cpu().numpy(), wi, "idx")
        # tau = 0.05, kappa = 100.  Without a tie the +8 logit wins by
        # kappa*(8 - max other) >> the noise range, p is exactly one-hot and
        # W' keeps exactly the hard mask's two weights.  With a tie the noise
        # decides between the tied candidates and may leave a mixture, so W'
        # can only be nonzero on the union of their kept positions.
        rows, cols = d["W"].shape
        w = d["W"].view(rows, cols // 4, 4).float()
        wo = d["W_out"].view(rows, cols // 4, 4).float()
        S = torch.zeros((6, 4), device="cuda")
        for c, (i, j) in enumerate(PAIRS):
            S[c, i] = S[c, j] = 1.0
        kept = S[d["idx_out"].long()] > 0
        hard = torch.where(kept, w, torch.zeros_like(w))
        assert bool((wo == hard).all(dim=-1)[~tie].all())
        union = ((L == top2[..., :1]).float() @ S) > 0
        assert int(((wo != 0) & ~union).sum()) == 0
        _check_rows(wl, d, sampled_rows(rows, every=512), bwd=False, check_prior=False)
    assert n_ties > 0
