"""Seeded synthetic inputs for the NF4 quantize / fused-matmul workloads.

This module only draws random numbers and names shapes. It holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can be fed from
it without sharing any of the computation. All tensors are created on the CPU
with ``torch.Generator`` seeded explicitly; callers move them where they need
them.

Value distributions follow the workloads the method is exercised on: weights
~ N(0, 0.02^2) (a 7B-class transformer's linear layers), optionally with a
small fraction of entries replaced by N(0, 0.5^2) outliers; activations
~ N(0, 1) and output gradients ~ N(0, 0.01^2), rounded to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# Seed plan: W = 0, X / dY = 1, outlier mask = 2, outlier values = 3;
# projection p of the decoder layer draws its weight from seed 10 + p.
SEED_W, SEED_X, SEED_MASK, SEED_OUTLIER = 0, 1, 2, 3


def normal(shape, std: float, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def weight(rows: int, cols: int, std: float = 0.02, seed: int = SEED_W,
           outlier_frac: float = 0.0, outlier_std: float = 0.5,
           mask_seed: int = SEED_MASK, value_seed: int = SEED_OUTLIER) -> torch.Tensor:
    """fp32 [rows, cols] ~ N(0, std^2); each entry independently (probability
    ``outlier_frac``) replaced by an N(0, outlier_std^2) draw."""
    w = normal((rows, cols), std, seed)
    if outlier_frac > 0:
        g = torch.Generator(device="cpu").manual_seed(int(mask_seed))
        mask = torch.rand(rows, cols, generator=g) < outlier_frac
        w = torch.where(mask, normal((rows, cols), outlier_std, value_seed), w)
    return w.contiguous()


def activations(m: int, k: int, std: float = 1.0, seed: int = SEED_X,
                dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """bf16 (or fp16) [m, k] ~ N(0, std^2), rounded to nearest-even from fp32."""
    return normal((m, k), std, seed).to(dtype).contiguous()


@dataclass(frozen=True)
class Projection:
    name: str
    rows: int          # N, output features
    cols: int          # K, input features
    seed: int
    std: float = 0.02
    outlier_frac: float = 0.0

    def make_weight(self) -> torch.Tensor:
        return weight(self.rows, self.cols, self.std, self.seed, self.outlier_frac)


@dataclass(frozen=True)
class Workload:
    """One named workload: weights, forward token counts, dX token counts."""
    name: str
    projections: tuple
    fwd_m: tuple = ()
    dx_m: tuple = ()
    x_std: float = 1.0
    dy_std: float = 0.01
    notes: str = ""
    extra: dict = field(default_factory=dict)
    # Projections that read the same input and can be issued together, in
    # layer order; projections not named run alone.
    concurrent: tuple = ()
    # Weight format ("nf4", "fp4", "int8"), element type of the weights fed to
    # quantize ("f32", "bf16"), of the activations ("bf16", "f16") and of the
    # matmul outputs ("f32", "bf16").
    wdtype: str = "nf4"
    w_in: str = "f32"
    act: str = "bf16"
    out: str = "f32"

    def issue_groups(self):
        """Projection indices grouped for issue, in order: each group's
        matmuls are independent of one another."""
        named = {i for g in self.concurrent for i in g}
        out, seen = [], set()
        for i in range(len(self.projections)):
            if i in seen:
                continue
            g = next((tuple(g) for g in self.concurrent if i in g), (i,)) if i in named else (i,)
            out.append(g)
            seen.update(g)
        return out


QWEN_LAYER = tuple(
    Projection(n, r, c, 10 + p) for p, (n, r, c) in enumerate([
        ("q_proj", 3584, 3584), ("k_proj", 512, 3584), ("v_proj", 512, 3584),
        ("o_proj", 3584, 3584), ("gate_proj", 18944, 3584), ("up_proj", 18944, 3584),
        ("down_proj", 3584, 18944)]))

WORKLOADS = {
    # NF4 round trip plus fused forward at a size the oracle finishes instantly
    "tiny_256": Workload("tiny_256", (Projection("w", 256, 256, SEED_W),), fwd_m=(8,), dx_m=(8,)),
    # decode-shaped forward: 4096x4096 projection with 0.1% outliers
    "decode_4096": Workload("decode_4096",
                            (Projection("w", 4096, 4096, SEED_W, outlier_frac=0.001),),
                            fwd_m=(1, 4, 16)),
    # prefill-shaped forward: MLP up projection 11008x4096, 4096 tokens
    "prefill_up_11008x4096": Workload("prefill_up_11008x4096",
                                      (Projection("up", 11008, 4096, SEED_W),), fwd_m=(4096,)),
    # frozen-base backward: MLP down projection 4096x11008, 2048 tokens
    "bwd_down_4096x11008": Workload("bwd_down_4096x11008",
                                    (Projection("down", 4096, 11008, SEED_W),), dx_m=(2048,),
                                    dy_std=0.01),
    # Qwen2.5-7B-shaped decoder layer, all seven linear weights
    # (q, k, v share the layer input; gate and up share the MLP input)
    "qwen2.5_7b_layer": Workload("qwen2.5_7b_layer", QWEN_LAYER, fwd_m=(1, 64, 2048), dx_m=(2048,),
                                 concurrent=((0, 1, 2), (4, 5))),
    # the prefill weight from a bf16 checkpoint, bf16 outputs
    "prefill_up_11008x4096_bf16": Workload("prefill_up_11008x4096_bf16",
                                           (Projection("up", 11008, 4096, SEED_W),), fwd_m=(4096,),
                                           w_in="bf16", out="bf16"),
    # the other weight formats on the decode and prefill shapes
    "decode_4096_fp4": Workload("decode_4096_fp4",
                                (Projection("w", 4096, 4096, SEED_W, outlier_frac=0.001),),
                                fwd_m=(1, 4, 16), wdtype="fp4"),
    "decode_4096_int8": Workload("decode_4096_int8",
                                 (Projection("w", 4096, 4096, SEED_W, outlier_frac=0.001),),
                                 fwd_m=(1, 4, 16), wdtype="int8"),
    "prefill_up_11008x4096_fp4": Workload("prefill_up_11008x4096_fp4",
                                          (Projection("up", 11008, 4096, SEED_W),), fwd_m=(4096,),
                                          wdtype="fp4"),
    "prefill_up_11008x4096_int8": Workload("prefill_up_11008x4096_int8",
                                           (Projection("up", 11008, 4096, SEED_W),),
                                           fwd_m=(4096,), wdtype="int8"),
    # fp16 activations and output gradients on the backward weight
    "bwd_down_4096x11008_f16": Workload("bwd_down_4096x11008_f16",
                                        (Projection("down", 4096, 11008, SEED_W),), dx_m=(2048,),
                                        dy_std=0.01, act="f16"),
}
