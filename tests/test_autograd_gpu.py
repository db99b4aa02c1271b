"""The autograd wrapper over the fused kernels: forward equals the fused
forward, the input gradient is the fused input-gradient kernel applied to the
bf16-cast incoming gradient (then cast to the input's dtype), the quantized
weight gets no gradient, and both match the oracle within the stated
tolerance."""
import numpy as np
import pytest
import torch

import dequant_gemm_gb300 as nf4
from dequant_gemm_gb300 import workloads as wl
from dequant_gemm_gb300.autograd import NF4Linear, nf4_linear
from oracle import nf4_oracle as o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REL_FRO, MAX_REL = 2e-3, 5e-3


def assert_tol(Y, Y_ref, what=""):
    rf, mr = o.rel_frobenius(Y, Y_ref), o.max_rel_to_max(Y, Y_ref)
    assert rf <= REL_FRO and mr <= MAX_REL, f"{what}: rel_fro={rf:.3e} max_rel={mr:.3e}"


@pytest.mark.parametrize("lead", [(1,), (3, 7), (2, 64)])
def test_linear_forward_backward(lead):
    rows, cols = 384, 512
    W = wl.weight(rows, cols, seed=21)
    q = nf4.nf4_quantize(W.to(DEV))
    n = int(np.prod(lead))
    X = wl.activations(n, cols, seed=22).reshape(*lead, cols).to(DEV).requires_grad_(True)
    G = wl.normal((n, rows), 0.01, seed=23).reshape(*lead, rows).to(DEV)

    Y = nf4_linear(X, q)
    assert Y.shape == (*lead, rows) and Y.dtype == torch.float32
    (Y * G).sum().backward()
    assert X.grad is not None and X.grad.dtype == torch.bfloat16 and X.grad.shape == X.shape

    # the wrapper adds only reshapes and casts around the fused kernels
    Y_k = nf4.nf4_matmul_fwd(X.detach().reshape(n, cols), q)
    dX_k = nf4.nf4_matmul_bwd_dx(G.reshape(n, rows).to(torch.bfloat16), q)
    assert torch.equal(Y.detach().reshape(n, rows), Y_k)
    assert torch.equal(X.grad.reshape(n, cols), dX_k.to(torch.bfloat16))

    # and the fused results meet the oracle
    Wh = o.dequantize(*o.quantize(W.numpy()), rows, cols)
    Xn = X.detach().reshape(n, cols).float().cpu().numpy()
    Gn = G.reshape(n, rows).to(torch.bfloat16).float().cpu().numpy()
    assert_tol(Y_k.cpu().numpy(), o.matmul_fwd(Xn, Wh), f"linear fwd {lead}")
    assert_tol(dX_k.cpu().numpy(), o.matmul_bwd_dx(Gn, Wh), f"linear dX {lead}")


def test_module_is_frozen_and_matches():
    rows, cols = 256, 320
    W = wl.weight(rows, cols, seed=31).to(DEV)
    layer = NF4Linear(W)
    assert list(layer.parameters()) == []
    assert {k for k, _ in layer.named_buffers()} == {"codes", "absmax_q", "absmax_scale"}
    X = wl.activations(5, cols, seed=32).to(DEV).requires_grad_(True)
    Y = layer(X)
    Y.sum().backward()
    q = nf4.nf4_quantize(W)
    assert torch.equal(Y.detach(), nf4.nf4_matmul_fwd(X.detach(), q))
    ones = torch.ones(5, rows, dtype=torch.bfloat16, device=DEV)
    assert torch.equal(X.grad, nf4.nf4_matmul_bwd_dx(ones, q, out_dtype=torch.bfloat16))
    assert nf4.nf4_poll_device_status() == 0


@pytest.mark.parametrize("dtype", ["fp4", "int8"])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16])
def test_module_formats_and_input_types(dtype, xdt):
    """Linear layers over FP4 and int8 weights, with bf16 and fp16 inputs and
    a bf16 output: forward and input gradient meet the oracle."""
    rows, cols = 256, 384
    W = wl.weight(rows, cols, seed=41)
    layer = NF4Linear(W.to(DEV), dtype=dtype, out_dtype=torch.bfloat16)
    assert list(layer.parameters()) == []
    X = wl.normal((6, cols), 1.0, seed=42).to(xdt).to(DEV).requires_grad_(True)
    Y = layer(X)
    assert Y.dtype == torch.bfloat16
    G = wl.normal((6, rows), 0.01, seed=43).to(DEV)
    (Y.float() * G).sum().backward()
    assert X.grad.dtype == xdt
    if dtype == "int8":
        What = o.int8_dequantize_flat(*o.int8_quantize_flat(W.numpy().reshape(-1))).reshape(rows, cols)
    else:
        lv = o.levels_of(dtype)
        What = o.dequantize(*o.quantize(W.numpy(), lv), rows, cols, lv)
    Xn = X.detach().float().cpu().numpy()
    Gn = G.to(torch.bfloat16).to(xdt).float().cpu().numpy()
    u = 2.0 ** -8     # one bf16 rounding of the output
    rf = o.rel_frobenius(Y.float().detach().cpu().numpy(), o.matmul_fwd(Xn, What))
    assert rf <= REL_FRO + u
    ref = o.matmul_bwd_dx(Gn, What)
    rfd = o.rel_frobenius(X.grad.float().cpu().numpy(), ref)
    assert rfd <= REL_FRO + 2 * u
    assert nf4.nf4_poll_device_status() == 0
