"""GPU parity: every entry point of libmaskllm, called through the C ABI (via
the ctypes binding), against the CPU oracle, element by element, on seeded
inputs that span several tiles with ragged tails, plus the edge cases."""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as wl
from tests._helpers import (assert_bf16_ulps, assert_bits_equal, assert_close, bits16, bits32,
                            ROWSQ_RTOL)

pytestmark = pytest.mark.gpu

# (rows, cols): minimum width, widths whose rows take non-power-of-two thread
# segments, a row longer than one pass with a ragged second pass, the
# 11008-wide LLaMA down projection, and many short rows per pass.
SHAPES = [(1, 32), (3, 96), (7, 160), (64, 224), (300, 64), (5, 4128), (2, 8192), (33, 11008),
          (256, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()
    orc.lib()


def _case(rows, cols, seed, **kw):
    W, L, G = wl.random_case(rows, cols, seed, device="cuda", **kw)
    return W, L, G


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_forward_matches_oracle(rows, cols):
    W, L, _ = _case(rows, cols, seed=rows * 7 + cols)
    tau, kappa, rng = 4.0, 100.0, (0, 0, 0)
    probs = torch.empty((rows, cols // 4, 6), dtype=torch.float32, device="cuda")
    Wo, sq, _ = mk.maskllm_forward(W, L, tau, kappa, rng, probs_out=probs)
    Wo_nop, sq_nop, _ = mk.maskllm_forward(W, L, tau, kappa, rng)
    torch.cuda.synchronize()
    want_W, want_sq, want_p, _ = orc.forward(bits16(W), L.cpu().numpy(), tau, kappa, *rng,
                                             want_probs=True)
    assert_bf16_ulps(bits16(Wo), want_W)
    assert_close(probs.cpu().numpy(), want_p, what="p")
    assert_close(sq.cpu().numpy(), want_sq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
    # the debug output changes nothing else
    assert_bits_equal(bits16(Wo_nop), bits16(Wo), "W' with/without probs")
    assert_bits_equal(bits32(sq_nop), bits32(sq), "row_sq with/without probs")


@pytest.mark.parametrize("tau,kappa,seed,step,tid", [
    (1.0, 300.0, 0, 0, 0), (0.2, 500.0, 0xFFFFFFFF12345678, 7, 255), (0.5, 300.0, 1, 1, 3),
    (0.05, 100.0, 2, 0, 9), (3.0, -4.0, 5, 1 << 31, 1 << 30),
    # z spread of ~60 per unit logit puts many probabilities (and soft-mask
    # entries) below 2^-126: the fp32 subnormal range must be kept, not flushed
    (1.0, 60.0, 3, 0, 0), (1.0, 85.0, 4, 0, 0)])
def test_forward_backward_across_temperatures(tau, kappa, seed, step, tid):
    rows, cols = 40, 1056
    W, L, G = _case(rows, cols, seed=11)
    rng = (seed, step, tid)
    probs = torch.empty((rows, cols // 4, 6), dtype=torch.float32, device="cuda")
    Wo, sq, _ = mk.maskllm_forward(W, L, tau, kappa, rng, probs_out=probs)
    dL = mk.maskllm_backward(W, L, G, tau, kappa, rng)
    torch.cuda.synchronize()
    Wb, Lh, Gb = bits16(W), L.cpu().numpy(), bits16(G)
    want_W, want_sq, want_p, _ = orc.forward(Wb, Lh, tau, kappa, *rng, want_probs=True)
    assert_bf16_ulps(bits16(Wo), want_W)
    assert_close(probs.cpu().numpy(), want_p, what="p")
    assert_close(sq.cpu().numpy(), want_sq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
    want_d = orc.backward(Wb, Lh, Gb, tau, kappa, *rng)
    assert_close(dL.cpu().numpy(), want_d, what="dlogits")


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("reg", [0.0, 0.25])
def test_backward_matches_oracle(rows, cols, reg):
    W, L, G = _case(rows, cols, seed=rows * 5 + cols + 1)
    tau, kappa, rng = 4.0, 100.0, (3, 2, 1)
    dL = mk.maskllm_backward(W, L, G, tau, kappa, rng, reg_coeff=reg)
    torch.cuda.synchronize()
    want = orc.backward(bits16(W), L.cpu().numpy(), bits16(G), tau, kappa, *rng, reg_coeff=reg)
    assert_close(dL.cpu().numpy(), want, what="dlogits")


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_prior_bit_exact(rows, cols):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rows + cols)
    x = torch.randn((rows, cols), generator=gen, device="cuda") * 0.02
    # exercise exponent gaps, zeros of both signs, subnormals and large values
    x.view(-1)[::17] *= 1e-30
    x.view(-1)[::29] = 0.0
    x.view(-1)[::31] = -0.0
    x.view(-1)[::37] *= 1e30
    W = x.to(torch.bfloat16)
    for scale in (300.0, 1.0, -0.5, 1.0000001):
        L = mk.maskllm_prior_init(W, scale)
        torch.cuda.synchronize()
        assert_bits_equal(bits32(L), orc.prior_init(bits16(W), scale).view(np.uint32), "prior")


def test_prior_propagates_nan_positions():
    W = torch.zeros((2, 32), dtype=torch.bfloat16, device="cuda")
    W[0, 5] = float("nan")
    W[1, 0] = float("inf")
    L = mk.maskllm_prior_init(W, 2.0).cpu().numpy()
    want = orc.prior_init(bits16(W), 2.0)
    assert (np.isnan(L) == np.isnan(want)).all()
    ok = ~np.isnan(want)
    assert_bits_equal(L[ok].view(np.uint32), want[ok].view(np.uint32), "prior (non-NaN)")


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_hard_compress_bit_exact_and_round_trip(rows, cols):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rows * 3 + cols)
    W = torch.randint(-32768, 32768, (rows, cols), generator=gen, device="cuda",
                      dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    # integer-valued logits make many exact ties; add NaNs and infinities
    L = torch.randint(-2, 3, (rows, cols // 4, 6), generator=gen, device="cuda").float()
    flat = L.view(-1)
    flat[::13] = float("nan")
    flat[::41] = float("inf")
    flat[::43] = float("-inf")
    L[::3, ::5, :] = float("nan")       # some all-NaN groups
    vals, meta, idx = mk.maskllm_hard_compress(W, L, want_idx=True)
    vals2, meta2, _ = mk.maskllm_hard_compress(W, L)
    D = mk.maskllm_decompress(vals, meta, rows, cols)
    torch.cuda.synchronize()
    wv, wm, wi = orc.hard_compress(bits16(W), L.cpu().numpy())
    assert_bits_equal(bits16(vals), wv, "values")
    assert_bits_equal(bits32(meta), wm, "meta")
    assert_bits_equal(idx.cpu().numpy(), wi, "idx")
    assert_bits_equal(bits16(vals2), wv, "values (no idx)")
    assert_bits_equal(bits32(meta2), wm, "meta (no idx)")
    assert_bits_equal(bits16(D), orc.decompress(wv, wm, rows, cols), "decompressed")


def test_noise_words_bit_exact():
    for seed, step, tid, g0, n in [(0, 0, 0, 0, 4099), (0xFFFFFFFFFFFFFFFF, 1, 2, 123, 1),
                                   (0x0123456789ABCDEF, 77, 1 << 31, (5 << 32) - 3, 1000),
                                   (42, 0xFFFFFFFF, 0xFFFFFFFF, (1 << 40) + 17, 513)]:
        got = mk.maskllm_noise_words((seed, step, tid), g0, n)
        torch.cuda.synchronize()
        assert_bits_equal(bits32(got), orc.noise_words(seed, step, tid, g0, n), "noise words")


def test_forward_is_deterministic_and_stream_safe():
    W, L, _ = _case(64, 4096, seed=5)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = mk.maskllm_forward(W, L, 1.0, 300.0, (9, 1, 2))
    s.synchronize()
    b = mk.maskllm_forward(W, L, 1.0, 300.0, (9, 1, 2))
    torch.cuda.synchronize()
    assert_bits_equal(bits16(a[0]), bits16(b[0]), "W'")
    assert_bits_equal(bits32(a[1]), bits32(b[1]), "row_sq")


def test_outputs_are_overwritten_not_accumulated():
    W, L, G = _case(16, 256, seed=6)
    dL = torch.full((16, 64, 6), 123.0, device="cuda")
    Wo = torch.full((16, 256), 7.0, device="cuda", dtype=torch.bfloat16)
    mk.maskllm_backward(W, L, G, 1.0, 10.0, (0, 0, 0), dlogits_out=dL)
    mk.maskllm_forward(W, L, 1.0, 10.0, (0, 0, 0), W_out=Wo)
    torch.cuda.synchronize()
    assert_close(dL.cpu().numpy(), orc.backward(bits16(W), L.cpu().numpy(), bits16(G), 1.0,
                                                10.0, 0), what="dlogits")
    assert_bf16_ulps(bits16(Wo), orc.forward(bits16(W), L.cpu().numpy(), 1.0, 10.0, 0)[0])


def test_invalid_arguments_launch_nothing():
    W, L, G = _case(4, 64, seed=7)
    with pytest.raises(mk.MaskLLMError) as e:
        mk.maskllm_forward(W, L, 0.0, 1.0, (0, 0, 0))
    assert e.value.status == 1
    with pytest.raises(mk.MaskLLMError) as e:
        mk.maskllm_forward(W, L, 1.0, 1.0, (0, 0, 0), W_out=W)   # output aliases input
    assert e.value.status == 4
    assert mk.maskllm_device_status() == 0


def test_device_status_clean_after_work():
    W, L, G = _case(128, 2048, seed=8)
    mk.maskllm_forward(W, L, 1.0, 1.0, (0, 0, 0))
    mk.maskllm_backward(W, L, G, 1.0, 1.0, (0, 0, 0))
    mk.maskllm_hard_compress(W, L)
    assert mk.maskllm_device_status() == 0
