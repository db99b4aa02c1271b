"""Frozen-base NF4 linear layer for PyTorch autograd.

The forward is the fused NF4-dequant matmul; the backward returns dL/dX through
the fused input-gradient kernel and no gradient for the quantized weight, which
is frozen ("Zenbit", zenbit.pallas_nf4 bullet: the backward computes dL/dX
only, without materialising the dequantized weight; "bitsandbytes", the layer
paragraph: a 4-bit linear layer over a quantized weight).

This module only marshals arguments: it flattens leading dimensions, casts the
incoming gradient to bf16 (the kernels' input type) and the returned gradient
to the input's dtype. Every product runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import NF4Weight, nf4_matmul_bwd_dx, nf4_matmul_fwd, nf4_quantize


class NF4LinearFunction(torch.autograd.Function):
    """y = x · dequant(W)ᵀ for bf16 x [..., cols] -> fp32 y [..., rows]."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: NF4Weight) -> torch.Tensor:
        if x.dtype != torch.bfloat16:
            raise ValueError(f"x must be bfloat16, got {x.dtype}")
        if x.shape[-1] != weight.cols:
            raise ValueError(f"x must end in {weight.cols} features, got {tuple(x.shape)}")
        lead = x.shape[:-1]
        y = nf4_matmul_fwd(x.reshape(-1, weight.cols).contiguous(), weight)
        ctx.weight = weight
        ctx.lead = lead
        return y.reshape(*lead, weight.rows)

    @staticmethod
    def backward(ctx, gy: torch.Tensor):
        if not ctx.needs_input_grad[0]:
            return None, None
        w = ctx.weight
        gy2 = gy.reshape(-1, w.rows).to(torch.bfloat16).contiguous()
        gx = nf4_matmul_bwd_dx(gy2, w)
        return gx.reshape(*ctx.lead, w.cols).to(torch.bfloat16), None


def nf4_linear(x: torch.Tensor, weight: NF4Weight) -> torch.Tensor:
    """Differentiable in x; the quantized weight gets no gradient."""
    return NF4LinearFunction.apply(x, weight)


class NF4Linear(torch.nn.Module):
    """A frozen linear layer (no bias) holding its weight NF4-quantized.

    The packed codes, absmax codes and second-level scales are buffers: they
    move with the module and are saved in its state dict, and no optimizer
    sees them."""

    def __init__(self, weight: torch.Tensor):
        super().__init__()
        if weight.dim() != 2:
            raise ValueError("weight must be 2-D [out_features, in_features]")
        q = nf4_quantize(weight.detach().to(torch.float32).contiguous())
        self.register_buffer("codes", q.codes)
        self.register_buffer("absmax_q", q.absmax_q)
        self.register_buffer("absmax_scale", q.absmax_scale)
        self.out_features, self.in_features = q.rows, q.cols

    def quantized_weight(self) -> NF4Weight:
        return NF4Weight(self.codes, self.absmax_q, self.absmax_scale, self.out_features,
                         self.in_features)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return nf4_linear(x, self.quantized_weight())

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, nf4"
