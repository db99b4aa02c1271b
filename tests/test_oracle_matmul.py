"""Pins for the oracle's fp64 matmuls: one-hot activations reproduce weight
columns exactly, an integer case is checked against an exact triple loop, the
input-gradient is the transpose identity of the forward, and a bf16 operand
simulation shows the stated tolerance is reachable with bf16 tensor-core
operands."""
import numpy as np
import torch

from oracle import nf4_oracle as o
from dequant_gemm_gb300 import workloads


def test_one_hot_rows_reproduce_weight():
    W = workloads.weight(48, 192, seed=4).numpy()
    packed, a8, s2 = o.quantize(W)
    What = o.dequantize(packed, a8, s2, 48, 192)
    X = np.zeros((5, 192))
    ks = [0, 7, 64, 100, 191]
    for m, k in enumerate(ks):
        X[m, k] = 1.0
    Y = o.matmul_fwd(X, What)
    assert Y.shape == (5, 48)
    for m, k in enumerate(ks):
        assert np.array_equal(Y[m], What[:, k].astype(np.float64))
    dY = np.zeros((3, 48))
    ns = [0, 17, 47]
    for m, n in enumerate(ns):
        dY[m, n] = 1.0
    dX = o.matmul_bwd_dx(dY, What)
    assert dX.shape == (3, 192)
    for m, n in enumerate(ns):
        assert np.array_equal(dX[m], What[n].astype(np.float64))


def test_integer_case_against_exact_loop():
    rng = np.random.default_rng(1)
    X = rng.integers(-3, 4, (3, 8)).astype(np.float64)
    Wn = rng.integers(-3, 4, (5, 8)).astype(np.float64)
    Y = o.matmul_fwd(X, Wn)
    for m in range(3):
        for n in range(5):
            assert Y[m, n] == sum(X[m, k] * Wn[n, k] for k in range(8))
    dY = rng.integers(-3, 4, (3, 5)).astype(np.float64)
    dX = o.matmul_bwd_dx(dY, Wn)
    for m in range(3):
        for k in range(8):
            assert dX[m, k] == sum(dY[m, n] * Wn[n, k] for n in range(5))


def test_error_measures():
    Y = np.array([[1.0, -2.0], [0.5, 4.0]])
    assert o.rel_frobenius(Y, Y) == 0 and o.max_rel_to_max(Y, Y) == 0
    Z = Y.copy()
    Z[1, 1] += 0.04
    assert abs(o.max_rel_to_max(Z, Y) - 0.01) < 1e-15
    assert abs(o.rel_frobenius(Z, Y) - 0.04 / np.sqrt(1 + 4 + 0.25 + 16)) < 1e-15


def test_bf16_operands_fit_the_tolerance():
    """With what rounded to bf16 and fp32 accumulation, the tiny workload's
    forward stays inside rel-Frobenius 2e-3 and max 5e-3 of max|Y|: the margin a
    bf16 tensor-core path has to work with."""
    W = workloads.weight(256, 256).numpy()
    X = workloads.activations(8, 256).float().numpy()
    packed, a8, s2 = o.quantize(W)
    What = o.dequantize(packed, a8, s2, 256, 256)
    Y_ref = o.matmul_fwd(X, What)
    Wb = torch.from_numpy(What).bfloat16().float().numpy()
    Y = (X.astype(np.float32) @ Wb.T.astype(np.float32)).astype(np.float64)
    assert o.rel_frobenius(Y, Y_ref) < 2e-3
    assert o.max_rel_to_max(Y, Y_ref) < 5e-3
