"""GPU parity of the entry points beyond the training step: logits from a
given mask (MaskLLM Table 2) and the convergence diagnostics (MaskLLM Fig. 5),
against the oracle."""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as wl
from tests._helpers import assert_bits_equal, assert_close, bits32

pytestmark = pytest.mark.gpu

SHAPES = [(1, 32), (3, 96), (7, 160), (300, 64), (5, 4128), (33, 11008), (256, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_prior_from_mask_bit_exact(rows, cols):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(rows * 11 + cols)
    meta = torch.randint(-2**31, 2**31 - 1, (rows, cols // 32), generator=gen, device="cuda",
                         dtype=torch.int64).to(torch.int32)   # every code, valid or not
    L = mk.maskllm_prior_from_mask(meta, rows, cols, 7.5, -0.25)
    torch.cuda.synchronize()
    want = orc.prior_from_mask(bits32(meta), rows, cols, 7.5, -0.25)
    assert_bits_equal(bits32(L), want.view(np.uint32), "logits from mask")


def _random_codes(rows, cols, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    return torch.randint(-2**31, 2**31 - 1, (rows, cols // 32), generator=gen, device="cuda",
                         dtype=torch.int64).to(torch.int32)   # every code, valid or not


@pytest.mark.parametrize("n", [len(SHAPES), 20])
def test_prior_from_mask_batched_matches_single_calls_and_oracle(n):
    """One batched launch over matrices whose last chunks are full (codes
    copied into the stage) and ragged (codes loaded per thread); 20 matrices
    take two launches."""
    shapes = [SHAPES[i % len(SHAPES)] for i in range(n)]
    mats = []
    for i, (rows, cols) in enumerate(shapes):
        meta = _random_codes(rows, cols, 900 + i)
        mats.append({"meta": meta, "logits_out": torch.full((rows, cols // 4, 6), float("nan"),
                                                            device="cuda")})
    mk.maskllm_prior_from_mask_batched(mats, 2.5, -1.0)
    torch.cuda.synchronize()
    for (rows, cols), m in zip(shapes, mats):
        single = mk.maskllm_prior_from_mask(m["meta"], rows, cols, 2.5, -1.0)
        torch.cuda.synchronize()
        assert torch.equal(single.view(torch.int32), m["logits_out"].view(torch.int32))
        want = orc.prior_from_mask(bits32(m["meta"]), rows, cols, 2.5, -1.0)
        assert_bits_equal(bits32(m["logits_out"]), want.view(np.uint32), "batched logits")


def test_prior_from_mask_round_trips_hard_compress():
    W, L, _ = wl.random_case(64, 4096, seed=77, device="cuda")
    vals, meta, idx = mk.maskllm_hard_compress(W, L, want_idx=True)
    P = mk.maskllm_prior_from_mask(meta, 64, 4096, 1.0, 0.0)
    vals2, meta2, idx2 = mk.maskllm_hard_compress(W, P, want_idx=True)
    torch.cuda.synchronize()
    assert torch.equal(meta, meta2) and torch.equal(idx, idx2) and torch.equal(vals, vals2)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("tau,kappa", [(1.0, 3.0), (0.2, 500.0), (4.0, 0.0), (0.5, 1e6)])
def test_mask_stats_match_oracle(rows, cols, tau, kappa):
    _, L, _ = wl.random_case(rows, cols, seed=rows + cols, device="cuda")
    rng_prev, rng = (5, 10, 3), (5, 11, 3)
    prev, _, _ = mk.maskllm_mask_stats(L, tau, kappa, rng_prev)
    idx, l1, mp = mk.maskllm_mask_stats(L, tau, kappa, rng, prev_idx=prev)
    none_idx, none_l1, none_mp = mk.maskllm_mask_stats(L, tau, kappa, rng, want_idx=False)
    torch.cuda.synchronize()
    Lh = L.cpu().numpy()
    wprev, _, _ = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng_prev)
    widx, wl1, wmp = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng, prev_idx=wprev)
    assert_bits_equal(prev.cpu().numpy(), wprev, "previous draws")
    assert_bits_equal(idx.cpu().numpy(), widx, "draws")
    assert_bits_equal(l1.cpu().numpy().view(np.uint32), wl1.astype(np.uint32), "L1 per row")
    assert_close(mp.cpu().numpy(), wmp, rtol=1e-5, atol=0, what="max-probability row sum")
    assert none_idx is None and none_l1 is None
    assert torch.equal(none_mp, mp)


def test_mask_stats_draw_is_the_forward_argmax():
    """The draw is the candidate the soft mask of the same step tends to: the
    first maximum of p as the forward reports it."""
    W, L, _ = wl.random_case(64, 2048, seed=91, device="cuda")
    probs = torch.empty_like(L)
    mk.maskllm_forward(W, L, 0.5, 30.0, (2, 4, 6), probs_out=probs)
    idx, _, _ = mk.maskllm_mask_stats(L, 0.5, 30.0, (2, 4, 6))
    torch.cuda.synchronize()
    p = probs.cpu().numpy()
    top = np.sort(p, axis=2)
    clear = (top[..., -1] - top[..., -2]) > 1e-6      # no near-tie in p
    assert clear.mean() > 0.99
    assert (idx.cpu().numpy()[clear] == p.argmax(2)[clear]).all()


def test_mask_stats_validation():
    _, L, _ = wl.random_case(4, 64, seed=1, device="cuda")
    l1 = torch.empty((4,), dtype=torch.int32, device="cuda")
    st = mk.lib().maskllm_mask_stats(L.data_ptr(), None, 4, 64, 1.0, 1.0, mk._rng((0, 0, 0)),
                                     None, l1.data_ptr(), None, None)
    assert st == 1   # the L1 distance needs the previous draws


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("tau,kappa", [(1.0, 3.0), (0.2, 500.0)])
def test_forward_stats_is_forward_plus_stats(rows, cols, tau, kappa):
    """The fused pass: W' and row_sq bit-identical to maskllm_forward (and
    within the forward's tolerance of the oracle), draws / L1 / max
    probability bit-identical to maskllm_mask_stats and as the oracle."""
    from tests._helpers import ROWSQ_RTOL, assert_bf16_ulps, bits16
    W, L, _ = wl.random_case(rows, cols, seed=3 * rows + cols, device="cuda")
    rng_prev, rng = (9, 20, 4), (9, 21, 4)
    prev, _, _ = mk.maskllm_mask_stats(L, tau, kappa, rng_prev)
    Wo, rsq, idx, l1, mp = mk.maskllm_forward_stats(W, L, tau, kappa, rng, prev_idx=prev)
    Wf = torch.empty_like(W)
    rf = torch.empty((rows,), device="cuda")
    mk.maskllm_forward(W, L, tau, kappa, rng, W_out=Wf, row_sq_out=rf)
    sidx, sl1, smp = mk.maskllm_mask_stats(L, tau, kappa, rng, prev_idx=prev)
    torch.cuda.synchronize()
    assert torch.equal(Wo.view(torch.int16), Wf.view(torch.int16))
    # the row sums are added in the forward's and the diagnostics' order
    assert torch.equal(rsq.view(torch.int32), rf.view(torch.int32))
    assert torch.equal(idx, sidx) and torch.equal(l1, sl1)
    assert torch.equal(mp.view(torch.int32), smp.view(torch.int32))
    Wb, Lh = bits16(W), L.cpu().numpy()
    wW, wsq, _, _ = orc.forward(Wb, Lh, tau, kappa, *rng)
    assert_bf16_ulps(bits16(Wo), wW)
    assert_close(rsq.cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
    wprev, _, _ = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng_prev)
    widx, wl1, wmp = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng, prev_idx=wprev)
    assert_bits_equal(idx.cpu().numpy(), widx, "draws")
    assert_bits_equal(l1.cpu().numpy().view(np.uint32), wl1.astype(np.uint32), "L1 per row")
    assert_close(mp.cpu().numpy(), wmp, rtol=1e-5, atol=0, what="max-probability row sum")


@pytest.mark.parametrize("n", [len(SHAPES), 20])
def test_diagnostics_batched_match_single_calls_and_oracle(n):
    """maskllm_mask_stats_batched and maskllm_forward_stats_batched over
    matrices of every test shape (long rows, rows shorter than a chunk,
    ragged last chunks), each with its own tensor id: every output
    bit-identical to the single-matrix call, draws and L1 to the oracle; 20
    matrices take two launches."""
    tau, kappa, seed, step = 0.5, 40.0, 9, 21
    shapes = [SHAPES[i % len(SHAPES)] for i in range(n)]
    mats, fmats = [], []
    for i, (rows, cols) in enumerate(shapes):
        W, L, _ = wl.random_case(rows, cols, seed=700 + i, device="cuda")
        tid = 3 + i
        prev, _, _ = mk.maskllm_mask_stats(L, tau, kappa, (seed, step - 1, tid))
        g = cols // 4
        mats.append({"W": None, "logits": L, "tensor_id": tid, "prev_idx": prev,
                     "idx_out": torch.empty((rows, g), dtype=torch.uint8, device="cuda"),
                     "l1_row_out": torch.empty((rows,), dtype=torch.int32, device="cuda"),
                     "maxprob_row_out": torch.empty((rows,), device="cuda")})
        fmats.append({"W": W, "logits": L, "tensor_id": tid, "prev_idx": prev,
                      "W_out": torch.empty_like(W),
                      "row_sq_out": torch.empty((rows,), device="cuda"),
                      "idx_out": torch.empty((rows, g), dtype=torch.uint8, device="cuda"),
                      "l1_row_out": torch.empty((rows,), dtype=torch.int32, device="cuda"),
                      "maxprob_row_out": torch.empty((rows,), device="cuda")})
    mk.maskllm_mask_stats_batched(mats, tau, kappa, seed, step)
    mk.maskllm_forward_stats_batched(fmats, tau, kappa, seed, step)
    torch.cuda.synchronize()
    for (rows, cols), m, f in zip(shapes, mats, fmats):
        rng = (seed, step, m["tensor_id"])
        idx, l1, mp = mk.maskllm_mask_stats(m["logits"], tau, kappa, rng, prev_idx=m["prev_idx"])
        Wo, rsq, fidx, fl1, fmp = mk.maskllm_forward_stats(f["W"], f["logits"], tau, kappa, rng,
                                                           prev_idx=f["prev_idx"])
        torch.cuda.synchronize()
        assert torch.equal(m["idx_out"], idx) and torch.equal(m["l1_row_out"], l1)
        assert torch.equal(m["maxprob_row_out"].view(torch.int32), mp.view(torch.int32))
        assert torch.equal(f["W_out"].view(torch.int16), Wo.view(torch.int16))
        assert torch.equal(f["row_sq_out"].view(torch.int32), rsq.view(torch.int32))
        assert torch.equal(f["idx_out"], fidx) and torch.equal(f["l1_row_out"], fl1)
        assert torch.equal(f["maxprob_row_out"].view(torch.int32), fmp.view(torch.int32))
        Lh = m["logits"].cpu().numpy()
        wprev, _, _ = orc.mask_stats(Lh, rows, cols, tau, kappa, seed, step - 1, m["tensor_id"])
        widx, wl1, wmp = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng, prev_idx=wprev)
        assert_bits_equal(m["idx_out"].cpu().numpy(), widx, "batched draws")
        assert_bits_equal(m["l1_row_out"].cpu().numpy().view(np.uint32), wl1.astype(np.uint32),
                          "batched L1 per row")
        assert_close(m["maxprob_row_out"].cpu().numpy(), wmp, rtol=1e-5, atol=0,
                     what="batched max-probability row sum")


def test_diagnostics_batched_optional_outputs_per_matrix():
    """A batch whose matrices leave out different optional outputs (no
    previous draws and no L1, no draws, no max probability, no row sums):
    what each writes equals the single call's bit for bit."""
    tau, kappa, seed, step = 1.0, 3.0, 4, 9
    shapes = [(7, 160), (300, 64), (5, 4128), (33, 11008)]
    mats, fmats, want = [], [], []
    for i, (rows, cols) in enumerate(shapes):
        W, L, _ = wl.random_case(rows, cols, seed=800 + i, device="cuda")
        g = cols // 4
        prev = None if i == 0 else mk.maskllm_mask_stats(L, tau, kappa, (seed, step - 1, i))[0]
        m = {"W": None, "logits": L, "tensor_id": i, "prev_idx": prev,
             "idx_out": None if i == 1 else torch.full((rows, g), 255, dtype=torch.uint8,
                                                       device="cuda"),
             "l1_row_out": None if prev is None else torch.full((rows,), -1, dtype=torch.int32,
                                                                device="cuda"),
             "maxprob_row_out": None if i == 2 else torch.full((rows,), -1.0, device="cuda")}
        f = dict(m, W=W, W_out=torch.empty_like(W),
                 row_sq_out=None if i == 3 else torch.empty((rows,), device="cuda"),
                 idx_out=None if m["idx_out"] is None else torch.empty_like(m["idx_out"]),
                 l1_row_out=None if m["l1_row_out"] is None else torch.empty_like(m["l1_row_out"]),
                 maxprob_row_out=(None if m["maxprob_row_out"] is None
                                  else torch.empty_like(m["maxprob_row_out"])))
        mats.append(m)
        fmats.append(f)
        want.append((L, W, prev))
    mk.maskllm_mask_stats_batched(mats, tau, kappa, seed, step)
    mk.maskllm_forward_stats_batched(fmats, tau, kappa, seed, step)
    torch.cuda.synchronize()
    for i, (m, f, (L, W, prev)) in enumerate(zip(mats, fmats, want)):
        rng = (seed, step, i)
        idx, l1, mp = mk.maskllm_mask_stats(L, tau, kappa, rng, prev_idx=prev)
        Wo, rsq, _, _, _ = mk.maskllm_forward_stats(W, L, tau, kappa, rng, prev_idx=prev)
        torch.cuda.synchronize()
        for out, ref in ((m["idx_out"], idx), (f["idx_out"], idx)):
            if out is not None:
                assert torch.equal(out, ref)
        for out, ref in ((m["l1_row_out"], l1), (f["l1_row_out"], l1)):
            if out is not None:
                assert torch.equal(out, ref)
        for out, ref in ((m["maxprob_row_out"], mp), (f["maxprob_row_out"], mp)):
            if out is not None:
                assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
        assert torch.equal(f["W_out"].view(torch.int16), Wo.view(torch.int16))
        if f["row_sq_out"] is not None:
            assert torch.equal(f["row_sq_out"].view(torch.int32), rsq.view(torch.int32))


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("tau,kappa,reg", [(1.0, 3.0, 0.0), (0.2, 500.0, 0.25)])
def test_backward_stats_is_backward_plus_stats(rows, cols, tau, kappa, reg):
    """The backward with the diagnostics: dlogits bit-identical to
    maskllm_backward (and within its tolerance of the oracle), draws / L1 /
    max probability bit-identical to maskllm_mask_stats and as the oracle."""
    W, L, G = wl.random_case(rows, cols, seed=5 * rows + cols, device="cuda")
    rng_prev, rng = (7, 30, 2), (7, 31, 2)
    prev, _, _ = mk.maskllm_mask_stats(L, tau, kappa, rng_prev)
    dl, idx, l1, mp = mk.maskllm_backward_stats(W, L, G, tau, kappa, rng, reg_coeff=reg,
                                                prev_idx=prev)
    dref = mk.maskllm_backward(W, L, G, tau, kappa, rng, reg_coeff=reg)
    sidx, sl1, smp = mk.maskllm_mask_stats(L, tau, kappa, rng, prev_idx=prev)
    torch.cuda.synchronize()
    assert torch.equal(dl.view(torch.int32), dref.view(torch.int32))
    assert torch.equal(idx, sidx) and torch.equal(l1, sl1)
    assert torch.equal(mp.view(torch.int32), smp.view(torch.int32))
    from tests._helpers import bits16
    Lh = L.cpu().numpy()
    want = orc.backward(bits16(W), Lh, bits16(G), tau, kappa, *rng, reg_coeff=reg)
    assert_close(dl.cpu().numpy(), want, what="dlogits")
    wprev, _, _ = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng_prev)
    widx, wl1, wmp = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng, prev_idx=wprev)
    assert_bits_equal(idx.cpu().numpy(), widx, "draws")
    assert_bits_equal(l1.cpu().numpy().view(np.uint32), wl1.astype(np.uint32), "L1 per row")
    assert_close(mp.cpu().numpy(), wmp, rtol=1e-5, atol=0, what="max-probability row sum")


@pytest.mark.parametrize("n", [len(SHAPES), 20])
def test_backward_stats_batched_match_single_calls(n):
    """One batched launch (two for 20 matrices) over every test shape, each
    matrix with its own tensor id; matrix 0 without previous draws (no L1),
    matrix 1 without draws out: every output bit-identical to the single
    call's."""
    tau, kappa, seed, step, reg = 0.5, 40.0, 3, 12, 0.1
    shapes = [SHAPES[i % len(SHAPES)] for i in range(n)]
    mats = []
    for i, (rows, cols) in enumerate(shapes):
        W, L, G = wl.random_case(rows, cols, seed=600 + i, device="cuda")
        g = cols // 4
        prev = None if i == 0 else mk.maskllm_mask_stats(L, tau, kappa, (seed, step - 1, i))[0]
        mats.append({"W": W, "logits": L, "grad_W_out": G, "tensor_id": i, "prev_idx": prev,
                     "dlogits_out": torch.empty_like(L),
                     "idx_out": None if i == 1 else torch.empty((rows, g), dtype=torch.uint8,
                                                                device="cuda"),
                     "l1_row_out": None if prev is None else torch.empty((rows,), dtype=torch.int32,
                                                                         device="cuda"),
                     "maxprob_row_out": torch.empty((rows,), device="cuda")})
    mk.maskllm_backward_stats_batched(mats, tau, kappa, seed, step, reg)
    torch.cuda.synchronize()
    for i, m in enumerate(mats):
        dl, idx, l1, mp = mk.maskllm_backward_stats(m["W"], m["logits"], m["grad_W_out"], tau,
                                                    kappa, (seed, step, i), reg_coeff=reg,
                                                    prev_idx=m["prev_idx"])
        torch.cuda.synchronize()
        assert torch.equal(m["dlogits_out"].view(torch.int32), dl.view(torch.int32))
        if m["idx_out"] is not None:
            assert torch.equal(m["idx_out"], idx)
        if m["l1_row_out"] is not None:
            assert torch.equal(m["l1_row_out"], l1)
        assert torch.equal(m["maxprob_row_out"].view(torch.int32), mp.view(torch.int32))


def test_forward_stats_optional_outputs():
    W, L, _ = wl.random_case(40, 256, seed=5, device="cuda")
    Wo, rsq, idx, l1, mp = mk.maskllm_forward_stats(W, L, 1.0, 3.0, (1, 2, 3), want_row_sq=False,
                                                    want_idx=False, want_maxprob=False)
    Wf = mk.maskllm_forward(W, L, 1.0, 3.0, (1, 2, 3))[0]
    torch.cuda.synchronize()
    assert rsq is None and idx is None and l1 is None and mp is None
    assert torch.equal(Wo.view(torch.int16), Wf.view(torch.int16))


def test_diagnostics_on_the_longest_rows():
    """Rows of 2^24 weights, the longest the diagnostics accept (4096
    chunks a row, each row finished by one CTA; an L1 row sum is exact in
    fp32 up to 2^24): the diagnostics pass and both fused passes against the
    oracle, and the fused passes' forward and backward outputs against the
    plain calls."""
    from tests._helpers import ROWSQ_RTOL, assert_bf16_ulps, bits16
    rows, cols = 2, 1 << 24
    tau, kappa = 0.5, 20.0
    W, L, G = wl.random_case(rows, cols, seed=4242, device="cuda")
    rng_prev, rng = (3, 1, 9), (3, 2, 9)
    prev, _, _ = mk.maskllm_mask_stats(L, tau, kappa, rng_prev)
    idx, l1, mp = mk.maskllm_mask_stats(L, tau, kappa, rng, prev_idx=prev)
    Wo, rsq, fidx, fl1, fmp = mk.maskllm_forward_stats(W, L, tau, kappa, rng, prev_idx=prev)
    dl, bidx, bl1, bmp = mk.maskllm_backward_stats(W, L, G, tau, kappa, rng, prev_idx=prev)
    dref = mk.maskllm_backward(W, L, G, tau, kappa, rng)
    torch.cuda.synchronize()
    for a, b in ((idx, fidx), (idx, bidx), (l1, fl1), (l1, bl1)):
        assert torch.equal(a, b)
    for a in (fmp, bmp):
        assert torch.equal(a.view(torch.int32), mp.view(torch.int32))
    assert torch.equal(dl.view(torch.int32), dref.view(torch.int32))
    Lh = L.cpu().numpy()
    wprev, _, _ = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng_prev)
    widx, wl1, wmp = orc.mask_stats(Lh, rows, cols, tau, kappa, *rng, prev_idx=wprev)
    assert_bits_equal(prev.cpu().numpy(), wprev, "previous draws")
    assert_bits_equal(idx.cpu().numpy(), widx, "draws")
    assert_bits_equal(l1.cpu().numpy().view(np.uint32), wl1.astype(np.uint32), "L1 per row")
    assert_close(mp.cpu().numpy(), wmp, rtol=1e-5, atol=0, what="max-probability row sum")
    wW, wsq, _, _ = orc.forward(bits16(W), Lh, tau, kappa, *rng)
    assert_bf16_ulps(bits16(Wo), wW)
    assert_close(rsq.cpu().numpy(), wsq, rtol=ROWSQ_RTOL, atol=0, what="row_sq")
