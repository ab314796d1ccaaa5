"""Seeded synthetic inputs for the MoE layer (shared by tests and the bench).

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic.  The same bytes it returns feed both the GPU library and
the CPU oracle.

Workload recipe (what the Ling-3.0-flash batch-1 decode post's layer looks
like, with random values in place of trained weights):
  * weights  W_r [E, H], W_gu [E, 2I, H], W_d [E, H, I]   ~ N(0, 0.02) in bf16
  * tokens   x [M, H]                                     ~ N(0, 1)    in bf16
  * skewed routing: a per-expert router bias b[e] = ln p_{pi(e)} with
    p_r proportional to r^-s (Zipf, s = 1.1) over ranks r = 1..E and pi a
    seeded permutation, so tokens of a block share experts.
Values are drawn in fp32 and rounded to bf16 (round to nearest even, which is
what ``Tensor.to(torch.bfloat16)`` does).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_experts: int
    topk: int
    inter: int


TINY = LayerShape(hidden=256, n_experts=16, topk=2, inter=128)
LING = LayerShape(hidden=2560, n_experts=512, topk=8, inter=512)
# The per-GPU slice of the post's 4-way tensor-parallel split: every GPU holds
# inter/4 = 128 rows of every expert's gate/up and the matching 128 columns
# of its down projection, routes redundantly and streams a quarter of each
# activated expert (the partial outputs are summed across GPUs afterwards).
LING_TP4 = LayerShape(hidden=2560, n_experts=512, topk=8, inter=128)
SHAPES = {"ling": LING, "ling_tp4": LING_TP4}
# The model's vocabulary projection: hidden 2560 and "about 157k" tokens (the
# pages give no exact count; 157,184 is the multiple of 128 nearest 157k).
LM_HEAD_VOCAB = 157184


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, std, g, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def layer_weights(shape: LayerShape, seed: int, device="cpu", std: float = WEIGHT_STD):
    """(w_router [E,H], w_gate_up [E,2I,H], w_down [E,H,I]) bf16 from one generator,
    drawn in the order W_r, W_gu, W_d."""
    g = _gen(seed, device)
    E, H, I = shape.n_experts, shape.hidden, shape.inter
    w_r = _randn_bf16((E, H), std, g, device)
    if str(device).startswith("cuda"):
        # draw the big tensors expert by expert: bounded fp32 temporaries
        w_gu = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
        for e in range(E):
            w_gu[e] = _randn_bf16((2 * I, H), std, g, device)
        w_d = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
        for e in range(E):
            w_d[e] = _randn_bf16((H, I), std, g, device)
    else:
        w_gu = _randn_bf16((E, 2 * I, H), std, g, device)
        w_d = _randn_bf16((E, H, I), std, g, device)
    return w_r, w_gu, w_d


def lm_head_weight(vocab: int, hidden: int, seed: int, device="cpu", std: float = WEIGHT_STD) -> torch.Tensor:
    """W [vocab, hidden] bf16 ~ N(0, std) from one generator (on CUDA in blocks
    of 8192 rows to bound temporaries)."""
    g = _gen(seed, device)
    if not str(device).startswith("cuda"):
        return _randn_bf16((vocab, hidden), std, g, device)
    w = torch.empty((vocab, hidden), dtype=torch.bfloat16, device=device)
    for r in range(0, vocab, 8192):
        n = min(8192, vocab - r)
        w[r:r + n] = _randn_bf16((n, hidden), std, g, device)
    return w


def fp8_rows(w: torch.Tensor):
    """Per-row fp8 (E4M3) codes and fp32 scales of a weight [..., rows, cols]:
    scale = max|row| / 448 (1 for an all-zero row), code = E4M3(w / scale)
    rounded to nearest even by torch's conversion.  Returns (uint8 codes,
    float32 scales [..., rows])."""
    w = w.float()
    amax = w.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (w / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return q, scale.to(torch.float32)


def fp8_expert_weights(shape: LayerShape, seed: int, device="cpu", std: float = WEIGHT_STD):
    """(w_router bf16 [E,H], q_gate_up u8 [E,2I,H], s_gate_up f32 [E,2I],
    q_down u8 [E,H,I], s_down f32 [E,H]): the router as layer_weights draws
    it, the experts drawn in fp32 ~ N(0, std) and quantized per output row
    (expert by expert on CUDA to bound temporaries)."""
    g = _gen(seed, device)
    E, H, I = shape.n_experts, shape.hidden, shape.inter
    w_r = _randn_bf16((E, H), std, g, device)
    q_gu = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=device)
    s_gu = torch.empty((E, 2 * I), dtype=torch.float32, device=device)
    q_d = torch.empty((E, H, I), dtype=torch.uint8, device=device)
    s_d = torch.empty((E, H), dtype=torch.float32, device=device)
    for e in range(E):
        q_gu[e], s_gu[e] = fp8_rows(torch.randn(2 * I, H, generator=g, device=device) * std)
    for e in range(E):
        q_d[e], s_d[e] = fp8_rows(torch.randn(H, I, generator=g, device=device) * std)
    return w_r, q_gu, s_gu, q_d, s_d


def tokens(M: int, hidden: int, seed: int, device="cpu") -> torch.Tensor:
    """x [M, hidden] bf16 ~ N(0,1)."""
    return _randn_bf16((M, hidden), 1.0, _gen(seed, device), device)


def tiny_case(M: int = 1, seed: int = 0, shape: LayerShape = TINY):
    """The small oracle-check layer: all tensors from ONE generator, order
    W_r, W_gu, W_d, x."""
    g = _gen(seed, "cpu")
    E, H, I = shape.n_experts, shape.hidden, shape.inter
    w_r = _randn_bf16((E, H), WEIGHT_STD, g, "cpu")
    w_gu = _randn_bf16((E, 2 * I, H), WEIGHT_STD, g, "cpu")
    w_d = _randn_bf16((E, H, I), WEIGHT_STD, g, "cpu")
    x = _randn_bf16((M, H), 1.0, g, "cpu")
    return w_r, w_gu, w_d, x


def zipf_router_bias(n_experts: int, s: float = 1.1, seed: int = 7) -> torch.Tensor:
    """fp32 [E]: b[e] = ln p_{pi(e)},  p_r = r^-s / sum_r' r'^-s,  pi ~ seeded permutation."""
    ranks = np.arange(1, n_experts + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    perm = torch.randperm(n_experts, generator=_gen(seed, "cpu")).numpy()
    return torch.from_numpy(np.log(p[perm]).astype(np.float32))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """A bf16 tensor's bit patterns as a numpy uint16 array (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)
