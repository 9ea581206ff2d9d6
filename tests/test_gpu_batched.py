"""GPU: batched calls (several matrices per launch) against the oracle and the
single-matrix calls, and the bounded-wait timeout path (a wait that runs out
sets the device error word, the context stays usable)."""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as wl
from tests._helpers import (assert_bf16_ulps, assert_bits_equal, assert_close, bits16, bits32,
                            ROWSQ_RTOL)

pytestmark = pytest.mark.gpu

# mixed shapes: long rows with ragged chunks, rows of exactly one chunk, short
# rows packed several per chunk, odd row counts
BATCH = [(37, 4128), (16, 4096), (5, 11008), (300, 64), (9, 1056), (64, 224), (3, 96)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


def _mats(shapes, seed=0):
    out = []
    for i, (r, c) in enumerate(shapes):
        W, L, G = wl.random_case(r, c, seed=seed + i, device="cuda")
        out.append({"W": W, "logits": L, "grad_W_out": G, "tensor_id": 100 + i,
                    "logits_out": torch.empty_like(L),
                    "W_out": torch.empty_like(W),
                    "row_sq_out": torch.empty((r,), device="cuda"),
                    "probs_out": torch.empty_like(L),
                    "dlogits_out": torch.empty_like(L),
                    "values_out": torch.empty((r, c // 2), dtype=torch.bfloat16, device="cuda"),
                    "meta_out": torch.empty((r, c // 32), dtype=torch.int32, device="cuda"),
                    "idx_out": torch.empty((r, c // 4), dtype=torch.uint8, device="cuda")})
    return out


@pytest.mark.parametrize("n", [len(BATCH), 20])
def test_batched_calls_match_oracle(n):
    shapes = (BATCH * 3)[:n]
    mats = _mats(shapes, seed=3)
    tau, kappa, seed, step, reg = 2.0, 50.0, 77, 5, 0.1
    mk.maskllm_prior_init_batched(mats, 300.0)
    mk.maskllm_forward_batched(mats, tau, kappa, seed, step)
    mk.maskllm_backward_batched(mats, tau, kappa, seed, step, reg_coeff=reg)
    mk.maskllm_hard_compress_batched(mats)
    torch.cuda.synchronize()
    assert mk.maskllm_device_status() == 0
    for m in mats:
        Wb, Lh, Gb = bits16(m["W"]), m["logits"].cpu().numpy(), bits16(m["grad_W_out"])
        rows, cols = m["W"].shape
        tid = m["tensor_id"]
        assert_bits_equal(bits32(m["logits_out"]), orc.prior_init(Wb, 300.0).view(np.uint32),
                          "prior")
        wW, wsq, wp, _ = orc.forward(Wb, Lh, tau, kappa, seed, step, tid, want_probs=True)
        assert_bf16_ulps(bits16(m["W_out"]), wW)
        assert_close(m["probs_out"].cpu().numpy(), wp, what="p")
        assert_close(m["row_sq_out"].cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
        assert_close(m["dlogits_out"].cpu().numpy(),
                     orc.backward(Wb, Lh, Gb, tau, kappa, seed, step, tid, reg), what="dlogits")
        wv, wm, wi = orc.hard_compress(Wb, Lh)
        assert_bits_equal(bits16(m["values_out"]), wv, "values")
        assert_bits_equal(bits32(m["meta_out"]), wm, "meta")
        assert_bits_equal(m["idx_out"].cpu().numpy(), wi, "idx")


def test_batched_equals_single_calls_bitwise():
    mats = _mats(BATCH, seed=11)
    tau, kappa, seed, step = 1.0, 300.0, 1, 2
    mk.maskllm_forward_batched(mats, tau, kappa, seed, step)
    mk.maskllm_backward_batched(mats, tau, kappa, seed, step)
    for m in mats:
        Wo, sq, _ = mk.maskllm_forward(m["W"], m["logits"], tau, kappa,
                                       (seed, step, m["tensor_id"]))
        dL = mk.maskllm_backward(m["W"], m["logits"], m["grad_W_out"], tau, kappa,
                                 (seed, step, m["tensor_id"]))
        torch.cuda.synchronize()
        assert_bits_equal(bits16(Wo), bits16(m["W_out"]), "W' batched vs single")
        assert_bits_equal(bits32(sq), bits32(m["row_sq_out"]), "row_sq batched vs single")
        assert_bits_equal(bits32(dL), bits32(m["dlogits_out"]), "dlogits batched vs single")


def test_batched_optional_outputs_may_be_null_per_matrix():
    mats = _mats(BATCH[:3], seed=21)
    mats[1]["probs_out"] = None
    mats[2]["row_sq_out"] = None
    mats[0]["idx_out"] = None
    mk.maskllm_forward_batched(mats, 4.0, 100.0, 0, 0)
    mk.maskllm_hard_compress_batched(mats)
    torch.cuda.synchronize()
    for m in mats:
        Wb, Lh = bits16(m["W"]), m["logits"].cpu().numpy()
        wW, wsq, wp, _ = orc.forward(Wb, Lh, 4.0, 100.0, 0, 0, m["tensor_id"], want_probs=True)
        assert_bf16_ulps(bits16(m["W_out"]), wW)
        if m["row_sq_out"] is not None:
            assert_close(m["row_sq_out"].cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0)
        wv, wm, _ = orc.hard_compress(Wb, Lh)
        assert_bits_equal(bits32(m["meta_out"]), wm, "meta")


def test_batched_rejects_cross_matrix_alias():
    mats = _mats(BATCH[:2], seed=31)
    mats[1]["dlogits_out"] = mats[0]["logits"]          # an output over another matrix's input
    with pytest.raises(mk.MaskLLMError) as e:
        mk.maskllm_backward_batched(mats, 1.0, 1.0, 0, 0)
    assert e.value.status == 4


def test_wait_timeout_sets_error_and_context_survives():
    """A wait that nothing will satisfy (the producer is told to issue no copies)
    gives up after the configured bound; the kernel returns, the error word
    reads MASKLLM_ERR_TIMEOUT, and the next launches work normally."""
    W, L, G = wl.random_case(8, 1024, seed=50, device="cuda")
    assert mk.maskllm_device_status() == 0
    try:
        mk.maskllm_set_wait_timeout(50_000_000)       # 50 ms
        mk.maskllm_test_withhold_loads(True)
        mk.maskllm_forward(W, L, 1.0, 10.0, (0, 0, 0))
        mk.maskllm_backward(W, L, G, 1.0, 10.0, (0, 0, 0))
        assert mk.maskllm_device_status() == 6      # MASKLLM_ERR_TIMEOUT
        assert mk.maskllm_device_status() == 0      # read clears it
        # every other pipelined kernel takes the same way out
        prev = torch.zeros((8, 256), dtype=torch.uint8, device="cuda")
        for run in (lambda: mk.maskllm_prior_init(W, 1.0),
                    lambda: mk.maskllm_hard_compress(W, L),
                    lambda: mk.maskllm_mask_stats(L, 1.0, 10.0, (0, 0, 0), prev_idx=prev),
                    lambda: mk.maskllm_forward_stats(W, L, 1.0, 10.0, (0, 0, 0), prev_idx=prev),
                    lambda: mk.maskllm_backward_stats(W, L, G, 1.0, 10.0, (0, 0, 0),
                                                      prev_idx=prev)):
            run()
            assert mk.maskllm_device_status() == 6
            assert mk.maskllm_device_status() == 0
    finally:
        mk.maskllm_test_withhold_loads(False)
        mk.maskllm_set_wait_timeout(2_000_000_000)
    Wo, sq, _ = mk.maskllm_forward(W, L, 1.0, 10.0, (0, 0, 0))
    dl, idx, _, _ = mk.maskllm_backward_stats(W, L, G, 1.0, 10.0, (0, 0, 0))
    torch.cuda.synchronize()
    assert mk.maskllm_device_status() == 0
    assert_bf16_ulps(bits16(Wo), orc.forward(bits16(W), L.cpu().numpy(), 1.0, 10.0, 0)[0])
    assert torch.equal(dl.view(torch.int32),
                       mk.maskllm_backward(W, L, G, 1.0, 10.0, (0, 0, 0)).view(torch.int32))


def _random_shapes(rng, n):
    """Row lengths that exercise every chunking case: short rows packed
    several to a chunk, rows of exactly one chunk, long rows with a ragged
    last chunk (also not a multiple of 64 groups), single rows."""
    cols = [32, 64, 96, 1056, 2048, 4096, 4128, 5504, 6144, 11008]
    return [(int(rng.integers(1, 70)), int(rng.choice(cols))) for _ in range(n)]


@pytest.mark.parametrize("trial", range(6))
def test_random_batches_equal_single_calls(trial):
    """Seeded random batches (1 to 20 matrices, so up to two launches) of
    random shapes: every batched stream operation -- prior, forward,
    backward, hard-compress, the diagnostics alone and fused into the
    forward and the backward -- writes exactly what its single-matrix call
    writes, matrix by matrix."""
    rng = np.random.default_rng(1000 + trial)
    n = int(rng.integers(1, 21))
    shapes = _random_shapes(rng, n)
    tau, kappa, seed, step = float(rng.choice([0.3, 1.0, 2.0])), float(rng.choice([3.0, 40.0])), 9, 5
    mats = _mats(shapes, seed=50 * trial)
    for i, (m, (r, c)) in enumerate(zip(mats, shapes)):
        g = c // 4
        m["prev_idx"] = mk.maskllm_mask_stats(m["logits"], tau, kappa, (seed, step - 1, 100 + i))[0]
        m["l1_row_out"] = torch.empty((r,), dtype=torch.int32, device="cuda")
        m["maxprob_row_out"] = torch.empty((r,), device="cuda")
        m["draws_out"] = torch.empty((r, g), dtype=torch.uint8, device="cuda")

    def equal(a, b):
        return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))

    # prior, forward, backward, hard-compress
    mk.maskllm_prior_init_batched(mats, 2.5)
    mk.maskllm_forward_batched(mats, tau, kappa, seed, step)
    mk.maskllm_backward_batched(mats, tau, kappa, seed, step, 0.0)
    mk.maskllm_hard_compress_batched(mats)
    torch.cuda.synchronize()
    for i, (m, (r, c)) in enumerate(zip(mats, shapes)):
        rng_i = (seed, step, 100 + i)
        assert equal(m["logits_out"], mk.maskllm_prior_init(m["W"], 2.5))
        Wo, sq, pr = mk.maskllm_forward(m["W"], m["logits"], tau, kappa, rng_i,
                                        probs_out=torch.empty_like(m["logits"]))
        assert equal(m["W_out"], Wo) and equal(m["row_sq_out"], sq) and equal(m["probs_out"], pr)
        assert equal(m["dlogits_out"], mk.maskllm_backward(m["W"], m["logits"], m["grad_W_out"],
                                                            tau, kappa, rng_i))
        v, meta, idx = mk.maskllm_hard_compress(m["W"], m["logits"], want_idx=True)
        assert equal(m["values_out"], v) and equal(m["meta_out"], meta) and equal(m["idx_out"], idx)

    # the diagnostics: alone, with the forward, with the backward
    diag = [dict(m, idx_out=m["draws_out"]) for m in mats]
    mk.maskllm_mask_stats_batched([dict(d, W=None) for d in diag], tau, kappa, seed, step)
    torch.cuda.synchronize()
    for i, d in enumerate(diag):
        idx, l1, mp = mk.maskllm_mask_stats(d["logits"], tau, kappa, (seed, step, 100 + i),
                                            prev_idx=d["prev_idx"])
        torch.cuda.synchronize()
        assert equal(d["draws_out"], idx) and equal(d["l1_row_out"], l1)
        assert equal(d["maxprob_row_out"], mp)
    mk.maskllm_forward_stats_batched(diag, tau, kappa, seed, step)
    torch.cuda.synchronize()
    for i, d in enumerate(diag):
        Wo, sq, idx, l1, mp = mk.maskllm_forward_stats(d["W"], d["logits"], tau, kappa,
                                                       (seed, step, 100 + i),
                                                       prev_idx=d["prev_idx"])
        torch.cuda.synchronize()
        assert equal(d["W_out"], Wo) and equal(d["row_sq_out"], sq)
        assert equal(d["draws_out"], idx) and equal(d["l1_row_out"], l1)
        assert equal(d["maxprob_row_out"], mp)
    mk.maskllm_backward_stats_batched(diag, tau, kappa, seed, step, 0.0)
    torch.cuda.synchronize()
    for i, d in enumerate(diag):
        dl, idx, l1, mp = mk.maskllm_backward_stats(d["W"], d["logits"], d["grad_W_out"], tau,
                                                    kappa, (seed, step, 100 + i),
                                                    prev_idx=d["prev_idx"])
        torch.cuda.synchronize()
        assert equal(d["dlogits_out"], dl)
        assert equal(d["draws_out"], idx) and equal(d["l1_row_out"], l1)
        assert equal(d["maxprob_row_out"], mp)
