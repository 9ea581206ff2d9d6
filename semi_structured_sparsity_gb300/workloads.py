"""Seeded synthetic inputs for the mask layer: shapes, distributions and seeds.

This module holds no arithmetic of the method itself.  It only draws the
frozen weights W, the logits (or the noise that is added to a prior), the
upstream gradients G, and it names the workload shapes.  Both the CUDA path
and the CPU oracle receive the tensors it makes.

Workloads (the weight shapes of the models the MaskLLM project page evaluates,
abstract: LLaMA-2, Nemotron-4):

* ``single``       one layer, W [256, 1024] ~ N(0, 0.02), logits ~ N(0, 1),
                   G ~ N(0, 1e-3); tau 4, kappa 100.
* ``llama2_7b_block``  the seven linears of one LLaMA-2-7B block (W is
                   [out, in]): q, k, v, o 4096x4096; gate, up 11008x4096;
                   down 4096x11008.  W ~ N(0, 0.02); logits = magnitude prior
                   with scale 300 plus N(0, 0.1); G ~ N(0, 1e-3); tau 1,
                   kappa 300.
* ``llama2_7b_full``   32 such blocks (6,476,005,376 weights), tau 0.5,
                   kappa 300, all logits resident.
* ``nemotron4_15b``    32 layers of q, o 6144x6144; k, v 1024x6144;
                   up 24576x6144; down 6144x24576.  W ~ N(0, 0.015),
                   logits ~ N(0, 1), G ~ N(0, 1e-3); tau 0.2, kappa 500;
                   processed layer by layer.
* ``compress_7b``  the llama2_7b_block shapes with near-one-hot logits: one
                   candidate per group at exactly +8, the rest N(0, 1), and in
                   1% of groups a second candidate also at exactly +8 (a tie).

The per-tensor seed is a pure function of (workload, layer, matrix, role), so
every tensor can be regenerated on its own; the layer's own noise stream uses
seed 0, step 0 and tensor id = layer * 8 + matrix index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

ROLE_W, ROLE_L, ROLE_G = 1, 2, 3

LLAMA2_7B_BLOCK = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096),
                   ("o", 4096, 4096), ("gate", 11008, 4096), ("up", 11008, 4096),
                   ("down", 4096, 11008)]
NEMOTRON4_15B_LAYER = [("q", 6144, 6144), ("k", 1024, 6144), ("v", 1024, 6144),
                       ("o", 6144, 6144), ("up", 24576, 6144), ("down", 6144, 24576)]


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                      # 1..5, used in the seed
    matrices: list = field(default_factory=list)   # [(name, rows, cols)]
    layers: int = 1
    w_sigma: float = 0.02
    logits: str = "normal"          # "normal" | "prior" | "onehot"
    l_sigma: float = 1.0
    prior_scale: float = 300.0
    g_sigma: float = 1e-3
    tau: float = 1.0
    kappa: float = 300.0

    @property
    def weights_per_layer(self) -> int:
        return sum(r * c for _, r, c in self.matrices)

    @property
    def weights(self) -> int:
        return self.weights_per_layer * self.layers


WORKLOADS = {
    "single": Workload("single", 1, [("w", 256, 1024)], 1, 0.02, "normal", 1.0, 0.0,
                       1e-3, 4.0, 100.0),
    "llama2_7b_block": Workload("llama2_7b_block", 2, LLAMA2_7B_BLOCK, 1, 0.02, "prior",
                                0.1, 300.0, 1e-3, 1.0, 300.0),
    "llama2_7b_full": Workload("llama2_7b_full", 3, LLAMA2_7B_BLOCK, 32, 0.02, "prior",
                               0.1, 300.0, 1e-3, 0.5, 300.0),
    "nemotron4_15b": Workload("nemotron4_15b", 4, NEMOTRON4_15B_LAYER, 32, 0.015, "normal",
                              1.0, 0.0, 1e-3, 0.2, 500.0),
    "compress_7b": Workload("compress_7b", 5, LLAMA2_7B_BLOCK, 1, 0.02, "onehot", 1.0, 0.0,
                            1e-3, 0.05, 100.0),
}

ONEHOT_WIN = 8.0
ONEHOT_TIE_FRACTION = 0.01


def tensor_seed(workload_index: int, layer: int, matrix: int, role: int) -> int:
    return ((workload_index * 64 + layer) * 16 + matrix) * 4 + role


def noise_tensor_id(layer: int, matrix: int) -> int:
    return layer * 8 + matrix


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(rows: int, cols: int, sigma: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, sigma^2) drawn in fp32, rounded to bf16 (nearest, ties to even)."""
    x = torch.randn((rows, cols), generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    return (x * sigma).to(torch.bfloat16)


def normal_f32(shape, sigma: float, seed: int, device="cpu") -> torch.Tensor:
    x = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return x * sigma if sigma != 1.0 else x


def onehot_logits(rows: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
    """Near-one-hot logits [rows, cols/4, 6]: one winner at exactly +8, the rest
    N(0, 1); in a seeded 1% of groups a second, different candidate is also at
    exactly +8."""
    groups = rows * cols // 4
    g = _gen(seed, device)
    L = torch.randn((groups, 6), generator=g, device=device, dtype=torch.float32)
    win = torch.randint(0, 6, (groups,), generator=g, device=device)
    tie = torch.rand((groups,), generator=g, device=device) < ONEHOT_TIE_FRACTION
    other = (win + torch.randint(1, 6, (groups,), generator=g, device=device)) % 6
    ar = torch.arange(groups, device=device)
    L[ar, win] = ONEHOT_WIN
    L[ar[tie], other[tie]] = ONEHOT_WIN
    return L.view(rows, cols // 4, 6)


@dataclass
class MatrixInputs:
    """Inputs of one matrix.  For ``logits == "prior"`` workloads ``L`` is None
    and ``L_noise`` holds the N(0, l_sigma) term that each side adds to its own
    magnitude prior of W."""
    name: str
    rows: int
    cols: int
    W: torch.Tensor
    G: torch.Tensor
    L: torch.Tensor | None
    L_noise: torch.Tensor | None
    tensor_id: int


def matrix_inputs(wl: Workload, layer: int, m: int, device="cpu", with_grad=True
                  ) -> MatrixInputs:
    name, rows, cols = wl.matrices[m]
    W = normal_bf16(rows, cols, wl.w_sigma, tensor_seed(wl.index, layer, m, ROLE_W), device)
    G = (normal_bf16(rows, cols, wl.g_sigma, tensor_seed(wl.index, layer, m, ROLE_G), device)
         if with_grad else None)
    lseed = tensor_seed(wl.index, layer, m, ROLE_L)
    L = L_noise = None
    if wl.logits == "normal":
        L = normal_f32((rows, cols // 4, 6), wl.l_sigma, lseed, device)
    elif wl.logits == "prior":
        L_noise = normal_f32((rows, cols // 4, 6), wl.l_sigma, lseed, device)
    elif wl.logits == "onehot":
        L = onehot_logits(rows, cols, lseed, device)
    else:
        raise ValueError(wl.logits)
    return MatrixInputs(name, rows, cols, W, G, L, L_noise, noise_tensor_id(layer, m))


def random_case(rows: int, cols: int, seed: int, w_sigma=0.02, l_sigma=1.0, g_sigma=1e-3,
                device="cpu"):
    """A generic seeded case (W bf16, L f32 [rows, cols/4, 6], G bf16)."""
    W = normal_bf16(rows, cols, w_sigma, seed * 4 + 1, device)
    L = normal_f32((rows, cols // 4, 6), l_sigma, seed * 4 + 2, device)
    G = normal_bf16(rows, cols, g_sigma, seed * 4 + 3, device)
    return W, L, G


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")
