"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Quantize and dequantize are bit-exact (codes, absmax codes, scales, fp32
dequantized weights). The fused matmuls meet the stated tolerance against the
oracle's fp64 dequantize-then-multiply: relative Frobenius error <= 2e-3 and
max error <= 5e-3 * max|Y_ref|. Small cases are compared in full; full-size
workloads on sampled rows / columns the oracle computes one by one, and in
full against an fp32 PyTorch product of the (bit-exact) dequantized weight.
"""
import functools

import numpy as np
import pytest
import torch

import dequant_gemm_gb300 as nf4
from dequant_gemm_gb300 import workloads as wl
from oracle import nf4_oracle as o
from tests.oracle_views import OracleWeight, sample_indices

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
torch.backends.cuda.matmul.allow_tf32 = False   # the fp32 cross-check must be fp32
REL_FRO, MAX_REL = 2e-3, 5e-3


def assert_tol(Y, Y_ref, what=""):
    rf, mr = o.rel_frobenius(Y, Y_ref), o.max_rel_to_max(Y, Y_ref)
    assert rf <= REL_FRO and mr <= MAX_REL, f"{what}: rel_fro={rf:.3e} max_rel={mr:.3e}"


def assert_quant_groups(W_np, q, groups):
    codes = q.codes.cpu().numpy()
    a8 = q.absmax_q.cpu().numpy()
    s2 = q.absmax_scale.cpu().numpy()
    flat = W_np.reshape(-1)
    for g in groups:
        lo, hi = g * 16384, min((g + 1) * 16384, flat.size)
        pc, pa, ps = o.quantize_flat(flat[lo:hi])
        assert np.array_equal(codes[lo // 2:hi // 2], pc), f"codes differ in group {g}"
        assert np.array_equal(a8[lo // 64:hi // 64], pa), f"absmax codes differ in group {g}"
        assert s2[g].view(np.uint32) == ps[0].view(np.uint32), f"s2 differs in group {g}"


def assert_quant_full(W_np, q):
    pc, pa, ps = o.quantize(W_np)
    assert np.array_equal(q.codes.cpu().numpy(), pc)
    assert np.array_equal(q.absmax_q.cpu().numpy(), pa)
    assert np.array_equal(q.absmax_scale.cpu().numpy().view(np.uint32), ps.view(np.uint32))
    return pc, pa, ps


@functools.lru_cache(maxsize=None)
def weight_np(rows, cols, seed, outlier_frac=0.0):
    return wl.weight(rows, cols, seed=seed, outlier_frac=outlier_frac).numpy()


# ---------------------------------------------------------------- quantize --
def test_quantize_tiny_full_and_dequant():
    W = weight_np(256, 256, 0)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    pc, pa, ps = assert_quant_full(W, q)
    Wd = nf4.nf4_dequantize(q).cpu().numpy()
    ref = o.dequantize(pc, pa, ps, 256, 256)
    assert np.array_equal(Wd.view(np.uint32), ref.view(np.uint32))


def test_quantize_decode_full_with_outliers():
    W = weight_np(4096, 4096, 0, 0.001)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    pc, pa, ps = assert_quant_full(W, q)
    Wd = nf4.nf4_dequantize(q).cpu().numpy()
    ref = o.dequantize(pc, pa, ps, 4096, 4096)
    assert np.array_equal(Wd.view(np.uint32), ref.view(np.uint32))


@functools.lru_cache(maxsize=4)
def oracle_quant(rows, cols, seed, outlier_frac=0.0):
    return o.quantize(weight_np(rows, cols, seed, outlier_frac))


FULL_SIZE = [(11008, 4096, 0), (4096, 11008, 0)] + [(p.rows, p.cols, p.seed) for p in wl.QWEN_LAYER]


@pytest.mark.parametrize("rows,cols,seed", FULL_SIZE,
                         ids=[f"{r}x{c}s{s}" for r, c, s in FULL_SIZE])
def test_quantize_full_size_bit_exact(rows, cols, seed):
    """Every code, absmax code and scale of the full-size weights (the
    prefill and backward weights and all seven projections of the decoder
    layer) against the oracle."""
    W = weight_np(rows, cols, seed)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    pc, pa, ps = oracle_quant(rows, cols, seed)
    assert np.array_equal(q.codes.cpu().numpy(), pc)
    assert np.array_equal(q.absmax_q.cpu().numpy(), pa)
    assert np.array_equal(q.absmax_scale.cpu().numpy().view(np.uint32), ps.view(np.uint32))


def test_dequantize_full_size_bit_exact():
    """nf4_dequantize of the 11008 x 4096 weight, every element."""
    W = weight_np(11008, 4096, 0)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    Wd = nf4.nf4_dequantize(q).cpu().numpy()
    ref = o.dequantize(*oracle_quant(11008, 4096, 0), 11008, 4096)
    assert np.array_equal(Wd.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("rows,cols", [(1, 64), (3, 192), (100, 192), (257, 128), (5, 16384 + 64)])
def test_quantize_ragged_shapes(rows, cols):
    W = weight_np(rows, cols, 3)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    assert_quant_full(W, q)


def test_quantize_special_cases():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    flat = W.reshape(-1)
    flat[0:64] = 0.0                                  # all-zero block
    flat[64:128] = 0.0
    flat[64 + 7] = -0.0                               # -0 in an all-zero block
    flat[64 + 9] = 3.0                                # single nonzero
    flat[192:256] = np.linspace(-1, 1, 64)            # exact +-absmax
    flat[256:320] = 1e-30 * rng.standard_normal(64)   # tiny block
    flat[320:384] = 1e30 * rng.standard_normal(64)    # huge block
    flat[384:448] = 2.0 ** -140                       # subnormal, all equal
    flat[16384:32768] = 0.0                           # an all-zero group
    c = o.nf4_levels().astype(np.float64)
    mids = ((c[:-1] + c[1:]) / 2).astype(np.float32)  # values on the decision edges
    flat[448:463] = mids
    flat[463] = 1.0
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    pc, pa, ps = assert_quant_full(W, q)
    Wd = nf4.nf4_dequantize(q).cpu().numpy()
    ref = o.dequantize(pc, pa, ps, 64, 1024)
    assert np.array_equal(Wd.view(np.uint32), ref.view(np.uint32))


def test_quantize_writes_only_its_outputs():
    W = torch.from_numpy(weight_np(96, 320, 7)).to(DEV)
    pad = 64
    n = 96 * 320
    codes = torch.full((n // 2 + 2 * pad,), 0xA5, dtype=torch.uint8, device=DEV)
    a8 = torch.full((n // 64 + 2 * pad,), 0x5A, dtype=torch.uint8, device=DEV)
    s2 = torch.full((2 + 2 * 16,), 7.0, dtype=torch.float32, device=DEV)
    q = nf4.NF4Weight(codes[pad:pad + n // 2], a8[pad:pad + n // 64], s2[16:18], 96, 320)
    nf4.nf4_quantize(W, out=q)
    torch.cuda.synchronize()
    assert torch.all(codes[:pad] == 0xA5) and torch.all(codes[pad + n // 2:] == 0xA5)
    assert torch.all(a8[:pad] == 0x5A) and torch.all(a8[pad + n // 64:] == 0x5A)
    assert torch.all(s2[:16] == 7.0) and torch.all(s2[18:] == 7.0)
    assert_quant_full(W.cpu().numpy(), q)


# ----------------------------------------------------------------- forward --
def run_fwd(W_np, X_bf16):
    q = nf4.nf4_quantize(torch.from_numpy(W_np).to(DEV))
    Y = nf4.nf4_matmul_fwd(X_bf16.to(DEV), q)
    return q, Y.cpu().numpy()


def test_fwd_tiny_full():
    W = weight_np(256, 256, 0)
    X = wl.activations(8, 256)
    _, Y = run_fwd(W, X)
    Wh = o.dequantize(*o.quantize(W), 256, 256)
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), "tiny fwd")


@pytest.mark.parametrize("M", [1, 4, 16])
def test_fwd_decode_full(M):
    W = weight_np(4096, 4096, 0, 0.001)
    X = wl.activations(M, 4096)
    _, Y = run_fwd(W, X)
    Wh = OracleWeight(W).rows(np.arange(4096))
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), f"decode fwd M={M}")


@pytest.mark.parametrize("M", [2, 3, 7, 9, 15, 17, 33, 100, 130, 300])
def test_fwd_ragged_tokens(M):
    W = weight_np(520, 1024, 8)
    X = wl.activations(M, 1024, seed=M)
    _, Y = run_fwd(W, X)
    Wh = o.dequantize(*o.quantize(W), 520, 1024)
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), f"ragged fwd M={M}")


def check_fwd_large(W, M, seed):
    X = wl.activations(M, W.shape[1], seed=seed)
    q, Y = run_fwd(W, X)
    ow = OracleWeight(W)
    rows = sample_indices(W.shape[0], 96, seed=seed)
    Y_ref = o.matmul_fwd(X.float().numpy(), ow.rows(rows))
    assert_tol(Y[:, rows], Y_ref, f"fwd {W.shape} M={M} sampled rows")
    # full output against fp32 torch on the bit-exact dequantized weight
    Wd = nf4.nf4_dequantize(q)
    Yt = (X.to(DEV).float() @ Wd.T).double().cpu().numpy()
    assert_tol(Y, Yt, f"fwd {W.shape} M={M} full vs fp32")
    assert np.isfinite(Y).all()


@pytest.mark.parametrize("M", [64, 2048])
def test_fwd_outlier_weight_on_tensor_cores(M):
    """The 4096 x 4096 weight with 0.1% N(0, 0.5^2) outliers, whose bf16
    operand rounding uses most of the error budget, through the tensor-core
    kernels (M = 64: single CTAs; M = 2048: CTA pairs)."""
    W = weight_np(4096, 4096, 0, 0.001)
    X = wl.activations(M, 4096, seed=M + 5)
    _, Y = run_fwd(W, X)
    ow = OracleWeight(W)
    rows = np.arange(4096) if M == 64 else sample_indices(4096, 256, seed=M)
    assert_tol(Y[:, rows], o.matmul_fwd(X.float().numpy(), ow.rows(rows)),
               f"outlier fwd M={M}")


@pytest.mark.parametrize("M", [1, 16])
def test_fwd_small_m_long_rows(M):
    """Rows longer than the small-M kernel's 49152-weight reduction limit go
    to the tensor-core kernel and still meet the tolerance."""
    W = weight_np(128, 53248, 31)
    X = wl.activations(M, 53248, seed=M + 31)
    _, Y = run_fwd(W, X)
    Wh = o.dequantize(*o.quantize(W), 128, 53248)
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), f"long-row fwd M={M}")


def test_fwd_prefill_up():
    check_fwd_large(weight_np(11008, 4096, 0), 4096, 1)


@pytest.mark.parametrize("proj", [p for p in wl.QWEN_LAYER])
@pytest.mark.parametrize("M", [1, 64, 2048])
def test_fwd_qwen_layer(proj, M):
    check_fwd_large(weight_np(proj.rows, proj.cols, proj.seed), M, 100 + M)


# ---------------------------------------------------------------- backward --
def run_dx(W_np, dY_bf16):
    q = nf4.nf4_quantize(torch.from_numpy(W_np).to(DEV))
    dX = nf4.nf4_matmul_bwd_dx(dY_bf16.to(DEV), q)
    return q, dX.cpu().numpy()


def test_dx_tiny_full():
    W = weight_np(256, 256, 0)
    dY = wl.activations(8, 256, std=0.01)
    _, dX = run_dx(W, dY)
    Wh = o.dequantize(*o.quantize(W), 256, 256)
    assert_tol(dX, o.matmul_bwd_dx(dY.float().numpy(), Wh), "tiny dX")


@pytest.mark.parametrize("M", [1, 5, 16, 40, 129])
def test_dx_ragged_tokens(M):
    W = weight_np(264, 1088, 9)
    dY = wl.activations(M, 264, std=0.01, seed=M)
    _, dX = run_dx(W, dY)
    Wh = o.dequantize(*o.quantize(W), 264, 1088)
    assert_tol(dX, o.matmul_bwd_dx(dY.float().numpy(), Wh), f"ragged dX M={M}")


def check_dx_large(W, M, seed):
    dY = wl.activations(M, W.shape[0], std=0.01, seed=seed)
    q, dX = run_dx(W, dY)
    ow = OracleWeight(W)
    kbs = sample_indices(W.shape[1] // 64, 32, seed=seed)   # first and last included
    cols = OracleWeight.columns_of(kbs)
    dX_ref = o.matmul_bwd_dx(dY.float().numpy(), ow.col_blocks(kbs))
    assert_tol(dX[:, cols], dX_ref, f"dX {W.shape} M={M} sampled columns")
    Wd = nf4.nf4_dequantize(q)
    dXt = (dY.to(DEV).float() @ Wd).double().cpu().numpy()
    assert_tol(dX, dXt, f"dX {W.shape} M={M} full vs fp32")


def test_dx_bwd_down():
    check_dx_large(weight_np(4096, 11008, 0), 2048, 1)


@pytest.mark.parametrize("proj", [p for p in wl.QWEN_LAYER])
def test_dx_qwen_layer(proj):
    check_dx_large(weight_np(proj.rows, proj.cols, proj.seed), 2048, 7)


# ------------------------------------------------------------------- misc --
def test_empty_and_zero_extents():
    q = nf4.nf4_quantize(torch.from_numpy(weight_np(64, 128, 1)).to(DEV))
    X = torch.empty(0, 128, dtype=torch.bfloat16, device=DEV)
    assert nf4.nf4_matmul_fwd(X, q).shape == (0, 64)
    dY = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    assert nf4.nf4_matmul_bwd_dx(dY, q).shape == (0, 128)
    e = nf4.nf4_quantize(torch.empty(0, 64, dtype=torch.float32, device=DEV))
    assert e.codes.numel() == 0
    assert nf4.nf4_poll_device_status() == 0


def test_fwd_output_guard_bytes():
    W = weight_np(136, 256, 2)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    for M in (3, 40):
        X = wl.activations(M, 256, seed=M).to(DEV)
        n = M * 136
        buf = torch.full((n + 64,), 123.0, dtype=torch.float32, device=DEV)
        Y = buf[32:32 + n].view(M, 136)
        nf4.nf4_matmul_fwd(X, q, out=Y)
        dbuf = torch.full((M * 256 + 64,), 321.0, dtype=torch.float32, device=DEV)
        dX = dbuf[32:32 + M * 256].view(M, 256)
        dY = wl.activations(M, 136, std=0.01, seed=M + 1).to(DEV)
        nf4.nf4_matmul_bwd_dx(dY, q, out=dX)
        torch.cuda.synchronize()
        assert torch.all(buf[:32] == 123.0) and torch.all(buf[32 + n:] == 123.0)
        assert torch.all(dbuf[:32] == 321.0) and torch.all(dbuf[32 + M * 256:] == 321.0)
    assert nf4.nf4_poll_device_status_site() == (0, 0)


def test_non_default_stream():
    W = weight_np(512, 512, 4)
    X = wl.activations(16, 512).to(DEV)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    Y0 = nf4.nf4_matmul_fwd(X, q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q2 = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
        Y1 = nf4.nf4_matmul_fwd(X, q2)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(q.codes, q2.codes)
    assert torch.allclose(Y0, Y1, rtol=0, atol=1e-5 * Y0.abs().max().item())


def test_quantize_quotients_on_decision_edges():
    """Weights w = fl32(m * a) +- a few ulps for every decision midpoint m and
    many absmax values a (tiny, subnormal and huge included): the quotients
    w / a land on or next to the thresholds, where only the correctly rounded
    IEEE quotient gives the oracle's codes."""
    rng = np.random.default_rng(17)
    c = o.nf4_levels().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2
    nblocks = 4096
    absmax = np.concatenate([
        rng.uniform(1e-3, 1.0, nblocks - 64),
        10.0 ** rng.uniform(-38, -30, 16), 10.0 ** rng.uniform(-44, -39, 16),
        10.0 ** rng.uniform(20, 35, 16), rng.uniform(0.5, 2.0, 16)]).astype(np.float32)
    W = np.empty((nblocks, 64), dtype=np.float32)
    W[:, 0] = absmax * np.where(rng.random(nblocks) < 0.5, 1, -1).astype(np.float32)
    for j in range(1, 64):
        m = mids[rng.integers(0, 15, nblocks)] * np.where(rng.random(nblocks) < 0.5, 1, -1)
        m = np.clip(m, -0.999, 0.999)
        base = np.abs(m * absmax.astype(np.float64)).astype(np.float32)
        k = rng.integers(-3, 4, nblocks).astype(np.int32)
        mag = np.maximum(base.view(np.int32) + k, 0).view(np.float32)   # step |w| by k ulps
        W[:, j] = np.where(m < 0, -mag, mag)
    W = np.where(np.abs(W) > np.abs(W[:, :1]), W[:, :1], W).astype(np.float32)
    assert np.isfinite(W).all()
    W = W.reshape(256, 1024)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    assert_quant_full(W, q)


@pytest.mark.parametrize("rows,cols", [(8, 64), (24, 128), (136, 64), (8, 4096)])
@pytest.mark.parametrize("M", [1, 16, 40, 300])
def test_fwd_small_shapes(rows, cols, M):
    """Shortest reductions and fewest rows the format allows, on the decode
    and tensor-memory paths (the code tile is wider than the weight; at
    M = 300 one CTA pair whose second CTA holds no weight row)."""
    W = weight_np(rows, cols, 21)
    X = wl.activations(M, cols, seed=rows + M)
    _, Y = run_fwd(W, X)
    Wh = o.dequantize(*o.quantize(W), rows, cols)
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), f"fwd {rows}x{cols} M={M}")


@pytest.mark.parametrize("rows,cols", [(8, 64), (24, 128), (136, 64)])
@pytest.mark.parametrize("M", [3, 40, 200])
def test_dx_small_shapes(rows, cols, M):
    W = weight_np(rows, cols, 22)
    dY = wl.activations(M, rows, std=0.01, seed=rows + M)
    _, dX = run_dx(W, dY)
    Wh = o.dequantize(*o.quantize(W), rows, cols)
    assert_tol(dX, o.matmul_bwd_dx(dY.float().numpy(), Wh), f"dX {rows}x{cols} M={M}")


@pytest.mark.parametrize("M", [50, 100, 300])
def test_persistent_units_with_ragged_tails(M):
    """Many more tile units than SMs (each CTA or pair walks several, its
    copy ring and accumulator buffers running on across them), with a ragged
    last row tile and a ragged last token tile, through the 64-, 128- and
    256-token tiles; compared in full with the oracle, both directions and
    both output types."""
    rows, cols = 38920, 192            # 304 row tiles of 128, the last one ragged
    W = weight_np(rows, cols, 41)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    Wh = o.dequantize(*o.quantize(W), rows, cols)
    X = wl.activations(M, cols, seed=M + 42)
    Y = nf4.nf4_matmul_fwd(X.to(DEV), q)
    Y_ref = o.matmul_fwd(X.float().numpy(), Wh)
    assert_tol(Y.cpu().numpy(), Y_ref, f"persistent fwd M={M}")
    Yb = nf4.nf4_matmul_fwd(X.to(DEV), q, out_dtype=torch.bfloat16)
    assert torch.equal(Yb, Y.to(torch.bfloat16))     # no split: the same sums, rounded
    Wd = weight_np(192, 38912, 43)    # 304 column tiles, a short reduction
    qd = nf4.nf4_quantize(torch.from_numpy(Wd).to(DEV))
    dY = wl.activations(M, 192, std=0.01, seed=M + 44)
    dX = nf4.nf4_matmul_bwd_dx(dY.to(DEV), qd).cpu().numpy()
    dX_ref = o.matmul_bwd_dx(dY.float().numpy(), o.dequantize(*o.quantize(Wd), 192, 38912))
    assert_tol(dX, dX_ref, f"persistent dX M={M}")
    assert nf4.nf4_poll_device_status() == 0


@pytest.mark.parametrize("rows,cols,M", [
    (40, 24576, 1), (40, 24576, 16), (520, 7168, 3), (520, 7168, 12), (2056, 1024, 8),
    (2056, 7168, 1), (264, 49152, 8), (1544, 3584, 16), (4104, 4096, 5), (1032, 8192, 1),
    (8200, 1024, 1), (264, 49152, 16), (136, 45056, 12), (4104, 4096, 16), (520, 4096, 9)])
def test_fwd_small_m_launch_shapes(rows, cols, M):
    """The small-M forward over its launch shapes: with and without a
    cluster of K-slices (1 to 8), one or two n-tiles, one or two token
    tiles, the wide and the narrow level table, rows that end inside a
    row group and short or long slices; compared in full."""
    W = weight_np(rows, cols, 51)
    X = wl.activations(M, cols, seed=rows + cols + M)
    _, Y = run_fwd(W, X)
    Wh = o.dequantize(*o.quantize(W), rows, cols)
    assert_tol(Y, o.matmul_fwd(X.float().numpy(), Wh), f"fwd {rows}x{cols} M={M}")
