"""Frozen-base NF4 linear layer for PyTorch autograd.

The forward is the fused NF4-dequant matmul; the backward returns dL/dX through
the fused input-gradient kernel and no gradient for the quantized weight, which
is frozen ("Zenbit", zenbit.pallas_nf4 bullet: the backward computes dL/dX
only, without materialising the dequantized weight; "bitsandbytes", the layer
paragraph: a 4-bit linear layer over a quantized weight).

This module only marshals arguments: it flattens leading dimensions, casts the
incoming gradient to the input's type (bf16 or fp16, the kernels' activation
types) and the returned gradient to the input's dtype. Every product runs in
the library's kernels. Weights may be NF4, FP4 or int8 ("bitsandbytes", the
4-bit paragraph: Linear4bit / LinearNF4 / LinearFP4 layers; "Zenbit",
zenbit.int8 bullet).
"""
from __future__ import annotations

import torch

from . import NF4Weight, nf4_matmul_bwd_dx, nf4_matmul_fwd, nf4_quantize


class NF4LinearFunction(torch.autograd.Function):
    """y = x · dequant(W)ᵀ for bf16 or fp16 x [..., cols] -> y [..., rows] of
    `out_dtype` (fp32 or bf16)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: NF4Weight,
                out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
        if x.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError(f"x must be bfloat16 or float16, got {x.dtype}")
        if x.shape[-1] != weight.cols:
            raise ValueError(f"x must end in {weight.cols} features, got {tuple(x.shape)}")
        lead = x.shape[:-1]
        y = nf4_matmul_fwd(x.reshape(-1, weight.cols).contiguous(), weight, out_dtype=out_dtype)
        ctx.weight = weight
        ctx.lead = lead
        ctx.x_dtype = x.dtype
        return y.reshape(*lead, weight.rows)

    @staticmethod
    def backward(ctx, gy: torch.Tensor):
        if not ctx.needs_input_grad[0]:
            return None, None, None
        w = ctx.weight
        gy2 = gy.reshape(-1, w.rows).to(ctx.x_dtype).contiguous()
        # a bf16 input gets its gradient straight from the kernel's bf16 output
        out = torch.bfloat16 if ctx.x_dtype == torch.bfloat16 else torch.float32
        gx = nf4_matmul_bwd_dx(gy2, w, out_dtype=out)
        return gx.reshape(*ctx.lead, w.cols).to(ctx.x_dtype), None, None


def nf4_linear(x: torch.Tensor, weight: NF4Weight,
               out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """Differentiable in x; the quantized weight gets no gradient."""
    return NF4LinearFunction.apply(x, weight, out_dtype)


class NF4Linear(torch.nn.Module):
    """A frozen linear layer (no bias) holding its weight quantized (NF4 by
    default; "fp4" or "int8" on request).

    The codes and scales are buffers: they move with the module and are saved
    in its state dict, and no optimizer sees them."""

    def __init__(self, weight: torch.Tensor, dtype: str = "nf4",
                 out_dtype: torch.dtype = torch.float32):
        super().__init__()
        if weight.dim() != 2:
            raise ValueError("weight must be 2-D [out_features, in_features]")
        w = weight.detach()
        if w.dtype not in (torch.float32, torch.bfloat16):
            w = w.to(torch.float32)
        q = nf4_quantize(w.contiguous(), dtype=dtype)
        self.register_buffer("codes", q.codes)
        if q.absmax_q is not None:
            self.register_buffer("absmax_q", q.absmax_q)
        else:
            self.absmax_q = None
        self.register_buffer("absmax_scale", q.absmax_scale)
        self.out_features, self.in_features = q.rows, q.cols
        self.qdtype = dtype
        self.out_dtype = out_dtype

    def quantized_weight(self) -> NF4Weight:
        return NF4Weight(self.codes, self.absmax_q, self.absmax_scale, self.out_features,
                         self.in_features, self.qdtype)

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return nf4_linear(x, self.quantized_weight(), self.out_dtype)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"{self.qdtype}")
