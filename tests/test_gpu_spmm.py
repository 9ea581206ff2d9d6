"""GPU parity of the 2:4 sparse x dense product ("Accelerating Sparse Deep
Neural Networks", Sec. 3.2) against the oracle: C = A B^T with A in the
compressed layout of the hard mask.

The compressed operands come from the oracle's own hard_compress of seeded
weights and logits (nothing the oracle reads comes from the GPU).  With
small-integer data every partial sum is an integer below 2^24, so fp32
accumulation in any order is exact and the comparison is bit-exact.  With
real-valued data the bound is |C - C_exact| <= 1e-5 * S, S = sum_k
|A[m,k] B[n,k]|: products are exact in fp32, and K/2 <= 2048 fp32 additions
in any order stay far below it (a single misplaced term is of order S/K and
fails it)."""
import numpy as np
import pytest
import torch

import oracle as orc
from semi_structured_sparsity_gb300 import binding as mk
from semi_structured_sparsity_gb300 import workloads as W
from tests._helpers import bits16

pytestmark = pytest.mark.gpu

RTOL_S = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mk.lib()


def operands(M, K, N, seed, integers=False):
    """Seeded W, logits and B on the host; A compressed by the oracle."""
    g = torch.Generator().manual_seed(seed)
    if integers:
        Wf = torch.randint(-8, 9, (M, K), generator=g).float()
        Bf = torch.randint(-8, 9, (N, K), generator=g).float()
    else:
        Wf = torch.randn((M, K), generator=g) * 0.02
        Bf = torch.randn((N, K), generator=g)
    Wb = bits16(Wf.to(torch.bfloat16))
    Bb = bits16(Bf.to(torch.bfloat16))
    L = torch.randn((M, K // 4, 6), generator=g).numpy()
    vals, meta, _ = orc.hard_compress(Wb, L)
    return vals, meta, Bb


def to_gpu(vals, meta, Bb):
    v = torch.from_numpy(vals.view(np.int16)).view(torch.bfloat16).cuda()
    m = torch.from_numpy(meta.view(np.int32)).cuda()
    b = torch.from_numpy(Bb.view(np.int16)).view(torch.bfloat16).cuda()
    return v, m, b


@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (200, 96, 300), (1, 32, 1), (257, 128, 5),
                                   (384, 1024, 520), (130, 32, 257),
                                   # last 128-deep stage with one 64-deep half
                                   # (K = 160) or three K = 32 blocks (K = 224);
                                   # the second CTA of a pair holding one row
                                   (129, 160, 256), (512, 224, 136), (385, 4096, 64)])
def test_small_integers_bit_exact(M, K, N):
    vals, meta, Bb = operands(M, K, N, M + K + N, integers=True)
    C = mk.maskllm_spmm(*to_gpu(vals, meta, Bb))
    want, _ = orc.spmm(vals, meta, M, K, Bb)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), want)
    assert mk.maskllm_device_status() == 0


@pytest.mark.parametrize("M,K,N", [(256, 512, 256), (333, 2048, 700), (128, 4096, 64)])
def test_real_values_within_bound(M, K, N):
    vals, meta, Bb = operands(M, K, N, 7 * M + N)
    C = mk.maskllm_spmm(*to_gpu(vals, meta, Bb)).cpu().numpy().astype(np.float64)
    want, S = orc.spmm(vals, meta, M, K, Bb)
    err = np.abs(C - want)
    assert (err <= RTOL_S * S + 1e-30).all(), float((err / (S + 1e-30)).max())


def test_output_not_16_byte_aligned_is_rejected():
    """Every pointer of the library starts on a 16-byte boundary; a C four
    bytes off is refused before anything runs and left untouched."""
    M, K, N = 300, 256, 256
    vals, meta, Bb = operands(M, K, N, 11, integers=True)
    v, m, b = to_gpu(vals, meta, Bb)
    buf = torch.full((M * N + 1,), float("nan"), device="cuda")
    C = buf[1:].view(M, N)
    assert C.data_ptr() % 16 != 0
    with pytest.raises(mk.MaskLLMError, match="ALIGNMENT"):
        mk.maskllm_spmm(v, m, b, C=C)
    assert torch.isnan(buf).all()
    assert mk.maskllm_device_status() == 0


@pytest.mark.parametrize("width", [128, 160, 192, 224, 256])
def test_every_tile_width_bit_exact(width):
    """The tile width (columns of C per CTA pair) is chosen per call; each
    width, forced, gives the exact product on ragged shapes: 700 columns
    leave a partial last tile for every width, 300 rows a partial pair."""
    M, K, N = 300, 192, 700
    vals, meta, Bb = operands(M, K, N, width, integers=True)
    try:
        mk.maskllm_test_spmm_tile_n(width)
        C = mk.maskllm_spmm(*to_gpu(vals, meta, Bb))
        torch.cuda.synchronize()
    finally:
        mk.maskllm_test_spmm_tile_n(0)
    want, _ = orc.spmm(vals, meta, M, K, Bb)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), want)
    assert mk.maskllm_device_status() == 0


def test_two_calls_in_a_row_and_output_overwritten():
    vals, meta, Bb = operands(256, 256, 512, 3, integers=True)
    v, m, b = to_gpu(vals, meta, Bb)
    C = torch.full((256, 512), float("nan"), device="cuda")
    mk.maskllm_spmm(v, m, b, C=C)
    mk.maskllm_spmm(v, m, b, C=C)
    want, _ = orc.spmm(vals, meta, 256, 256, Bb)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), want)


@pytest.mark.slow
def test_q_projection_full_size_sampled_rows():
    """The LLaMA-2-7B q projection (4096 x 4096), pruned by the hard mask of
    its magnitude prior, times 2048 activation rows: 64 sampled rows of C
    against the oracle."""
    wl = W.WORKLOADS["llama2_7b_block"]
    x = W.matrix_inputs(wl, 0, 0, device="cpu", with_grad=False)
    Wb = bits16(x.W)
    L = orc.prior_init(Wb, 1.0)
    vals, meta, _ = orc.hard_compress(Wb, L)
    M, K = Wb.shape
    N = 2048
    Bb = bits16(W.normal_bf16(N, K, 1.0, 99))
    C = mk.maskllm_spmm(*to_gpu(vals, meta, Bb))
    rows = np.random.default_rng(0).choice(M, 64, replace=False)
    want, S = orc.spmm(vals[rows], meta[rows], len(rows), K, Bb)
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    assert (np.abs(got - want) <= RTOL_S * S + 1e-30).all()
