"""The tensor-core kernels feed the MMA exactly the dequantized weight rounded
to the operand type, and the small-M kernel scales exactly the fp16 level it
multiplies.

With one-hot activations every output element is one weight times 1.0 plus
exact zeros, so the fused forward returns the transpose of the operand matrix
and the input gradient the matrix itself, whatever the reduction order or the
split of the reduction. The operand matrix is the oracle's fp32 dequantized
weight rounded to nearest even in bf16 (fp16 with fp16 activations). This
pins, element by element, the forward's level pair tables, the input
gradient's byte-plane permutes and the int8 conversion, which the fp64
tolerance tests can only bound. Weights stay in the normal range of both
operand types (the smallest nonzero dequantized weight here is ~1e-3).
"""
import numpy as np
import pytest
import torch

import dequant_gemm_gb300 as nf4
from dequant_gemm_gb300 import workloads as wl
from oracle import nf4_oracle as o

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FORMATS = ("nf4", "fp4", "int8")
ACTS = (torch.bfloat16, torch.float16)


def oracle_operands(W, dtype, act):
    """fp32 dequantized weight rounded to the operand type, as fp32. 4-bit:
    the oracle's dequantized weight. int8: the fused kernels scale a block
    by its step fl32(a / 127), computed once, so the operand is
    fl32(q * fl32(a / 127)) from the oracle's codes and absmax (the
    stand-alone dequantize rounds fl32(q * a) / 127 instead; the two differ
    by at most an fp32 ulp)."""
    rows, cols = W.shape
    if dtype == "int8":
        qv, a = o.int8_quantize_flat(W.reshape(-1))
        step = (np.asarray(a, dtype=np.float32) / np.float32(127.0)).astype(np.float32)
        What = (qv.reshape(-1, 64).astype(np.float32) * step[:, None]).astype(np.float32)
        What = What.reshape(rows, cols)
    else:
        lv = o.levels_of(dtype)
        What = o.dequantize(*o.quantize(W, lv), rows, cols, lv)
    return torch.from_numpy(np.ascontiguousarray(What, dtype=np.float32)).to(act).float()


def one_hot(m, k, act):
    X = torch.zeros(m, k, dtype=act)
    X[torch.arange(m), torch.arange(m)] = 1.0
    return X


@pytest.mark.parametrize("act", ACTS, ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("N,K", [(384, 256), (256, 640)])
def test_forward_operands_are_the_rounded_dequantized_weight(dtype, act, N, K):
    W = wl.weight(N, K, seed=29).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    X = one_hot(K, K, act).to(DEV)          # K tokens: above the small-M path
    Y = nf4.nf4_matmul_fwd(X, q).cpu()
    ref = oracle_operands(W, dtype, act).t()
    bad = (Y != ref).sum().item()
    assert bad == 0, f"{bad} of {Y.numel()} operands differ"


@pytest.mark.parametrize("act", ACTS, ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("N,K", [(384, 256), (640, 512)])
def test_input_gradient_operands_are_the_rounded_dequantized_weight(dtype, act, N, K):
    W = wl.weight(N, K, seed=31).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    dY = one_hot(N, N, act).to(DEV)         # N tokens, one per weight row
    dX = nf4.nf4_matmul_bwd_dx(dY, q).cpu()
    ref = oracle_operands(W, dtype, act)
    bad = (dX != ref).sum().item()
    assert bad == 0, f"{bad} of {dX.numel()} operands differ"


def small_m_products(W, dtype):
    """What the small-M kernel computes for one weight and an activation of
    1: the code's level rounded to fp16 (the operand its MMAs take; int8: the
    integer, exact) times the block scale after the MMA, in fp32: â from the
    oracle for 4-bit codes, fl32(a / 127) for int8."""
    rows, cols = W.shape
    if dtype == "int8":
        qv, a = o.int8_quantize_flat(W.reshape(-1))
        step = (np.asarray(a, dtype=np.float32) / np.float32(127.0)).astype(np.float32)
        v = qv.reshape(-1, 64).astype(np.float32) * step[:, None]
    else:
        lv = o.levels_of(dtype)
        packed, a8, s2 = o.quantize(W, lv)
        q = o.unpack_nibbles(packed).reshape(-1, 64)
        lv16 = lv.astype(np.float16).astype(np.float32)
        v = lv16[q] * o.dequant_absmax(a8, s2).astype(np.float32)[:, None]
    return np.ascontiguousarray(v.astype(np.float32).reshape(rows, cols))


@pytest.mark.parametrize("act", ACTS, ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("N,K,M", [(512, 4096, 1), (4096, 4096, 16), (1040, 18944, 4),
                                   (136, 45056, 12), (8200, 1024, 1)])
def test_small_m_forward_is_exact_on_one_hot_tokens(dtype, act, N, K, M):
    """Token m carries a single 1 at column k_m (spread over the row), so
    Y[m, n] is that one weight's product: fp32(level16 * scale), bit for bit
    (the activation's power-of-two rescale into fp16 and back is exact for
    1; every other block adds exact zeros)."""
    W = wl.weight(N, K, seed=37).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    ks = [(m * (K // M) + 37 * m + 5) % K for m in range(M)]
    X = torch.zeros(M, K, dtype=act)
    X[torch.arange(M), torch.tensor(ks)] = 1.0
    Y = nf4.nf4_matmul_fwd(X.to(DEV), q).cpu()
    ref = torch.from_numpy(small_m_products(W, dtype)[:, ks].T.copy())
    bad = (Y != ref).sum().item()
    assert bad == 0, f"{bad} of {Y.numel()} outputs differ"


@pytest.mark.parametrize("act", ACTS, ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("M", [17, 64, 100, 200])
def test_tensor_core_forward_tiles_pick_exact_operands(dtype, act, M):
    """Every token tile width (64, 128, 256) and split: token m's single 1 at
    column k_m returns column k_m of the operand matrix."""
    N, K = 640, 1024
    W = wl.weight(N, K, seed=41).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    ks = [(13 * m + 7) % K for m in range(M)]
    X = torch.zeros(M, K, dtype=act)
    X[torch.arange(M), torch.tensor(ks)] = 1.0
    Y = nf4.nf4_matmul_fwd(X.to(DEV), q).cpu()
    ref = oracle_operands(W, dtype, act)[:, ks].t()
    bad = (Y != ref).sum().item()
    assert bad == 0, f"{bad} of {Y.numel()} outputs differ"


@pytest.mark.parametrize("act", ACTS, ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("M", [1, 5, 64, 100, 200])
def test_tensor_core_input_gradient_tiles_pick_exact_operands(dtype, act, M):
    """The input gradient at every token tile width: token m's single 1 at
    weight row n_m returns row n_m of the operand matrix."""
    N, K = 640, 1024
    W = wl.weight(N, K, seed=43).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    ns = [(29 * m + 3) % N for m in range(M)]
    dY = torch.zeros(M, N, dtype=act)
    dY[torch.arange(M), torch.tensor(ns)] = 1.0
    dX = nf4.nf4_matmul_bwd_dx(dY.to(DEV), q).cpu()
    ref = oracle_operands(W, dtype, act)[ns, :]
    bad = (dX != ref).sum().item()
    assert bad == 0, f"{bad} of {dX.numel()} outputs differ"


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=("f32", "bf16"))
@pytest.mark.parametrize("M", [1, 16, 64, 200])
def test_accumulate_adds_the_exact_product(M, out_dtype):
    """NF4_ACCUMULATE on one-hot tokens: each output becomes its previous
    contents plus one product, added once in fp32 (and for a bf16 output
    rounded to nearest even), on both the small-M and the tensor-core paths."""
    N, K = 384, 1024
    W = wl.weight(N, K, seed=47).numpy()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    ks = [(11 * m + 3) % K for m in range(M)]
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    X[torch.arange(M), torch.tensor(ks)] = 1.0
    prod = (torch.from_numpy(small_m_products(W, "nf4")) if M <= 16
            else oracle_operands(W, "nf4", torch.bfloat16))[:, ks].t()
    Y0 = (torch.randn(M, N, generator=torch.Generator().manual_seed(M)) * 0.05).to(out_dtype)
    Y = Y0.to(DEV)
    nf4.nf4_matmul_fwd(X.to(DEV), q, out=Y, accumulate=True)
    ref = (Y0.float() + prod).to(out_dtype)
    bad = (Y.cpu() != ref).sum().item()
    assert bad == 0, f"{bad} of {Y.numel()} outputs differ"


@pytest.mark.parametrize("dtype", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 16])
def test_grouped_forward_is_exact_on_one_hot_tokens(dtype, M):
    """nf4_matmul_fwd_group: every weight of the group (different row counts,
    so the row tiles of one launch switch weights mid-grid) gets its own
    exact products."""
    K = 2048
    Ws = [wl.weight(n, K, seed=50 + n % 7).numpy() for n in (1040, 96, 528, 16)]
    qs = [nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype) for W in Ws]
    ks = [(97 * m + 11) % K for m in range(M)]
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    X[torch.arange(M), torch.tensor(ks)] = 1.0
    Ys = nf4.nf4_matmul_fwd_group(X.to(DEV), qs)
    for W, Y in zip(Ws, Ys):
        ref = torch.from_numpy(small_m_products(W, dtype)[:, ks].T.copy())
        bad = (Y.cpu() != ref).sum().item()
        assert bad == 0, f"{bad} of {Y.numel()} outputs differ (rows {W.shape[0]})"
