"""Python face of the expert contraction on either engine (include/gemv.h):
y[m][r] = sum_k W[r][k] x[m][k], bf16 in, fp32 out, M <= 16 tokens, on the
CUDA cores or the tensor cores over the layer kernel's packed tile layout.
Argument marshalling only: the work runs in the library's kernels."""
from __future__ import annotations

import torch

from . import native as N
from .layer import _ptr, _stream_ptr

CUDA_CORES = N.MOE_GEMV_CUDA_CORES
TENSOR_CORES = N.MOE_GEMV_TENSOR_CORES


def pack(w: torch.Tensor, stream=None) -> torch.Tensor:
    """Packed copy (8-row tiles, fragment order) of a bf16 [rows][k] weight."""
    if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_contiguous() or not w.is_cuda:
        raise ValueError("w must be a contiguous bf16 [rows][k] CUDA tensor")
    packed = torch.empty_like(w)
    N.check("moe_gemv_pack", N.lib().moe_gemv_pack(_ptr(w), _ptr(packed), w.shape[0], w.shape[1],
                                                   _stream_ptr(stream)))
    return packed


def gemv(packed: torch.Tensor, x: torch.Tensor, engine: int, y: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """y = W x (fp32 [M][rows]) on `engine` (CUDA_CORES or TENSOR_CORES)."""
    rows, k = packed.shape
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 2 or x.shape[1] != k:
        raise ValueError("x must be contiguous bf16 [M][k]")
    if y is None:
        y = torch.empty((x.shape[0], rows), dtype=torch.float32, device=x.device)
    N.check("moe_gemv", N.lib().moe_gemv(_ptr(packed), _ptr(x), _ptr(y), rows, k, x.shape[0], engine,
                                         _stream_ptr(stream)))
    return y


def status() -> int:
    """Sticky device status of the GEMV kernels (synchronises; clears it)."""
    return N.lib().moe_gemv_get_status()
