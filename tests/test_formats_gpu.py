"""Parity of the other weight formats, activation and output types, and the
accumulating epilogue with the CPU oracle, through the C ABI.

* FP4 (E2M1) and int8 quantize / dequantize are bit-exact against the oracle,
  from fp32 and from bf16 weights (a bf16 weight is quantized as its exact
  fp32 value), as are NF4 codes from bf16 weights.
* Fused matmuls of every format, with bf16 or fp16 activations, meet the
  stated tolerance (relative Frobenius <= 2e-3, max <= 5e-3 max|ref|) against
  the oracle's fp64 dequantize-then-multiply.
* A bf16 output is the fp32 result rounded to nearest even: it equals the
  fp32 output rounded to bf16 wherever the fp32 path does not split its
  reduction, and its error against fp64 stays within the fp32 bounds plus one
  bf16 rounding (2^-8 relative).
* NF4_ACCUMULATE adds the product to the output's contents.
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
REL_FRO, MAX_REL = 2e-3, 5e-3
BF16_U = 2.0 ** -8      # unit roundoff of bf16


def assert_tol(Y, Y_ref, what="", rel=REL_FRO, mx=MAX_REL):
    rf, mr = o.rel_frobenius(Y, Y_ref), o.max_rel_to_max(Y, Y_ref)
    assert rf <= rel and mr <= mx, f"{what}: rel_fro={rf:.3e} max_rel={mr:.3e}"


@functools.lru_cache(maxsize=None)
def weight_np(rows, cols, seed, outlier_frac=0.0):
    return wl.weight(rows, cols, seed=seed, outlier_frac=outlier_frac).numpy()


def oracle_quantize(W, dtype):
    if dtype == "int8":
        return o.int8_quantize_flat(W.reshape(-1))
    return o.quantize(W, o.levels_of(dtype))


def oracle_dequant(W, dtype):
    rows, cols = W.shape
    if dtype == "int8":
        return o.int8_dequantize_flat(*o.int8_quantize_flat(W.reshape(-1))).reshape(rows, cols)
    lv = o.levels_of(dtype)
    return o.dequantize(*o.quantize(W, lv), rows, cols, lv)


def assert_quant_equal(q, ref, dtype):
    if dtype == "int8":
        qv, a = ref
        assert np.array_equal(q.codes.cpu().numpy(), qv)
        assert np.array_equal(q.absmax_scale.cpu().numpy().view(np.uint32), a.view(np.uint32))
        return
    pc, pa, ps = ref
    assert np.array_equal(q.codes.cpu().numpy(), pc)
    assert np.array_equal(q.absmax_q.cpu().numpy(), pa)
    assert np.array_equal(q.absmax_scale.cpu().numpy().view(np.uint32), ps.view(np.uint32))


def special_weight(rng, rows=64, cols=1024):
    """Zero blocks and groups, single nonzeros, +-absmax, -0, tiny, huge and
    subnormal blocks, values on and next to every decision midpoint of the
    format's table (or int8 half-way points)."""
    W = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    f = W.reshape(-1)
    f[0:64] = 0.0
    f[64:128] = 0.0
    f[64 + 7] = -0.0
    f[64 + 9] = 3.0
    f[192:256] = np.linspace(-1, 1, 64)
    f[256:320] = 1e-30 * rng.standard_normal(64)
    f[320:384] = 1e30 * rng.standard_normal(64)
    f[384:448] = 2.0 ** -140
    f[16384:32768] = 0.0
    return W


def edge_weight(rng, dtype, nblocks=2048):
    """Blocks whose absmax is a (element 0) and whose other elements sit
    within 3 ulps of m * a for the format's decision points m."""
    if dtype == "int8":
        mids = (np.arange(-127, 127) + 0.5) / 127.0
    else:
        lv = np.sort(np.unique(np.abs(o.levels_of(dtype).astype(np.float64))))
        mids = (lv[:-1] + lv[1:]) / 2
    absmax = np.concatenate([rng.uniform(1e-3, 1.0, nblocks - 64), 10.0 ** rng.uniform(-38, -30, 16),
                             10.0 ** rng.uniform(-44, -39, 16), 10.0 ** rng.uniform(20, 35, 16),
                             rng.uniform(0.5, 2.0, 16)]).astype(np.float32)
    W = np.empty((nblocks, 64), dtype=np.float32)
    W[:, 0] = absmax * np.where(rng.random(nblocks) < 0.5, 1, -1).astype(np.float32)
    for j in range(1, 64):
        m = mids[rng.integers(0, mids.size, nblocks)] * np.where(rng.random(nblocks) < 0.5, 1, -1)
        base = np.abs(m * absmax.astype(np.float64)).astype(np.float32)
        k = rng.integers(-3, 4, nblocks).astype(np.int32)
        mag = np.maximum(base.view(np.int32) + k, 0).view(np.float32)
        W[:, j] = np.where(m < 0, -mag, mag)
    W = np.where(np.abs(W) > np.abs(W[:, :1]), W[:, :1], W).astype(np.float32)
    return W.reshape(nblocks // 16, 1024)


# ---------------------------------------------------------------- quantize --
@pytest.mark.parametrize("dtype", ["fp4", "int8"])
def test_quantize_formats_bit_exact(dtype):
    rng = np.random.default_rng(1)
    for W in (weight_np(4096, 4096, 0, 0.001), special_weight(rng), weight_np(3, 192, 3)):
        q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
        assert_quant_equal(q, oracle_quantize(W, dtype), dtype)
        Wd = nf4.nf4_dequantize(q).cpu().numpy()
        assert np.array_equal(Wd.view(np.uint32), oracle_dequant(W, dtype).view(np.uint32))
    assert nf4.nf4_poll_device_status() == 0


@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
def test_quantize_formats_on_decision_edges(dtype):
    W = edge_weight(np.random.default_rng(7), dtype)
    assert np.isfinite(W).all()
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    assert_quant_equal(q, oracle_quantize(W, dtype), dtype)


@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
def test_quantize_from_bf16_weights(dtype):
    """A bf16 weight quantizes to the codes of its exact fp32 value."""
    Wb = wl.weight(1024, 1536, seed=5, outlier_frac=0.001).to(torch.bfloat16)
    bits = Wb.view(torch.int16).numpy().view(np.uint16)
    W32 = o.bf16_to_fp32(bits).reshape(1024, 1536)
    q = nf4.nf4_quantize(Wb.to(DEV), dtype=dtype)
    assert_quant_equal(q, oracle_quantize(W32, dtype), dtype)


def test_quantize_bf16_full_size():
    Wb = torch.from_numpy(weight_np(11008, 4096, 0)).to(torch.bfloat16)
    W32 = o.bf16_to_fp32(Wb.view(torch.int16).numpy().view(np.uint16)).reshape(11008, 4096)
    q = nf4.nf4_quantize(Wb.to(DEV))
    assert_quant_equal(q, o.quantize(W32), "nf4")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16], ids=("bf16", "f16"))
@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
def test_dequantize_to_16_bits_is_the_rounded_fp32_weight(dtype, out_dtype):
    """nf4_dequantize_ex: the oracle's fp32 dequantized weight rounded to
    nearest even, bit for bit (special blocks included: fp16 takes 1e30 to
    infinity and tiny weights to subnormals or zero, like the rounding on
    the host)."""
    rng = np.random.default_rng(9)
    for W in (special_weight(rng), weight_np(3, 192, 4), weight_np(520, 1024, 8, 0.001)):
        q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
        Wd = nf4.nf4_dequantize(q, out_dtype=out_dtype).cpu()
        ref = torch.from_numpy(oracle_dequant(W, dtype)).to(out_dtype)
        assert Wd.dtype == out_dtype and Wd.shape == ref.shape
        assert torch.equal(Wd.view(torch.int16), ref.view(torch.int16))
    assert nf4.nf4_poll_device_status() == 0


def test_dequantize_bf16_full_size_matches_fp32_rounded():
    q = nf4.nf4_quantize(torch.from_numpy(weight_np(11008, 4096, 0)).to(DEV))
    out = torch.empty(11008, 4096, dtype=torch.bfloat16, device=DEV)
    Wb = nf4.nf4_dequantize(q, out=out)
    assert Wb.data_ptr() == out.data_ptr()
    assert torch.equal(Wb.view(torch.int16), nf4.nf4_dequantize(q).to(torch.bfloat16).view(torch.int16))


# ----------------------------------------------------------------- matmuls --
def run(W, dtype, A, dx, **kw):
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype)
    fn = nf4.nf4_matmul_bwd_dx if dx else nf4.nf4_matmul_fwd
    return q, fn(A.to(DEV), q, **kw)


@pytest.mark.parametrize("dtype", ["fp4", "int8"])
@pytest.mark.parametrize("M", [1, 5, 16, 40, 130, 300])
def test_fwd_formats(dtype, M):
    W = weight_np(520, 1024, 8)
    X = wl.activations(M, 1024, seed=M)
    _, Y = run(W, dtype, X, False)
    assert_tol(Y.cpu().numpy(), o.matmul_fwd(X.float().numpy(), oracle_dequant(W, dtype)),
               f"{dtype} fwd M={M}")


@pytest.mark.parametrize("dtype", ["fp4", "int8"])
@pytest.mark.parametrize("M", [1, 16, 40, 129, 300])
def test_dx_formats(dtype, M):
    W = weight_np(264, 1088, 9)
    dY = wl.activations(M, 264, std=0.01, seed=M)
    _, dX = run(W, dtype, dY, True)
    assert_tol(dX.cpu().numpy(), o.matmul_bwd_dx(dY.float().numpy(), oracle_dequant(W, dtype)),
               f"{dtype} dX M={M}")


@pytest.mark.parametrize("dtype", ["fp4", "int8"])
@pytest.mark.parametrize("M", [1, 2048])
def test_formats_full_size(dtype, M):
    """The 11008 x 4096 prefill weight: forward on sampled rows, input
    gradient (4096 x 11008 weight) on sampled column blocks, first and last
    included."""
    W = weight_np(11008, 4096, 0)
    X = wl.activations(M, 4096, seed=M + 2)
    _, Y = run(W, dtype, X, False)
    ow = OracleWeight(W, dtype)
    rows = sample_indices(11008, 96, seed=M)
    assert_tol(Y.cpu().numpy()[:, rows], o.matmul_fwd(X.float().numpy(), ow.rows(rows)),
               f"{dtype} fwd 11008x4096 M={M}")
    Wd = weight_np(4096, 11008, 0)
    dY = wl.activations(M, 4096, std=0.01, seed=M + 3)
    _, dX = run(Wd, dtype, dY, True)
    owd = OracleWeight(Wd, dtype)
    kbs = sample_indices(11008 // 64, 32, seed=M)
    assert_tol(dX.cpu().numpy()[:, OracleWeight.columns_of(kbs)],
               o.matmul_bwd_dx(dY.float().numpy(), owd.col_blocks(kbs)),
               f"{dtype} dX 4096x11008 M={M}")


@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
@pytest.mark.parametrize("M", [1, 16, 40, 300])
def test_fp16_activations(dtype, M):
    """fp16 X and dY: the dequantized weight enters the tensor cores as fp16."""
    W = weight_np(520, 1024, 12)
    X = wl.normal((M, 1024), 1.0, seed=M + 40).to(torch.float16)
    _, Y = run(W, dtype, X, False)
    What = oracle_dequant(W, dtype)
    assert_tol(Y.cpu().numpy(), o.matmul_fwd(X.float().numpy(), What), f"{dtype} fp16 fwd M={M}")
    dY = wl.normal((M, 520), 0.01, seed=M + 41).to(torch.float16)
    _, dX = run(W, dtype, dY, True)
    assert_tol(dX.cpu().numpy(), o.matmul_bwd_dx(dY.float().numpy(), What),
               f"{dtype} fp16 dX M={M}")


def bf16_round(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16)


@pytest.mark.parametrize("M", [1, 16, 300])
def test_bf16_output_small_shapes(M):
    """Error bound of a bf16 output: the fp32 bounds plus one rounding of at
    most 2^-8 of the value (triangle inequality)."""
    W = weight_np(520, 1024, 13)
    X = wl.activations(M, 1024, seed=M + 50)
    q, Y = run(W, "nf4", X, False, out_dtype=torch.bfloat16)
    assert Y.dtype == torch.bfloat16
    Y_ref = o.matmul_fwd(X.float().numpy(), oracle_dequant(W, "nf4"))
    assert_tol(Y.float().cpu().numpy(), Y_ref, f"bf16 fwd M={M}",
               rel=REL_FRO + BF16_U * (1 + REL_FRO), mx=MAX_REL + BF16_U * (1 + MAX_REL))
    if M <= 16:   # the small-M kernel reduces in a fixed order: same bits as fp32, rounded
        Y32 = nf4.nf4_matmul_fwd(X.to(DEV), q)
        assert torch.equal(bf16_round(Y32), Y)
    dY = wl.activations(M, 520, std=0.01, seed=M + 51)
    _, dX = run(W, "nf4", dY, True, out_dtype=torch.bfloat16)
    dX_ref = o.matmul_bwd_dx(dY.float().numpy(), oracle_dequant(W, "nf4"))
    assert_tol(dX.float().cpu().numpy(), dX_ref, f"bf16 dX M={M}",
               rel=REL_FRO + BF16_U * (1 + REL_FRO), mx=MAX_REL + BF16_U * (1 + MAX_REL))


def test_bf16_output_is_the_rounded_fp32_output_at_prefill_size():
    """4096 tokens x 11008 x 4096: enough tiles that neither path splits its
    reduction, so the bf16 output is exactly the fp32 output rounded."""
    W = weight_np(11008, 4096, 0)
    X = wl.activations(4096, 4096, seed=1).to(DEV)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    Y32 = nf4.nf4_matmul_fwd(X, q)
    Y16 = nf4.nf4_matmul_fwd(X, q, out_dtype=torch.bfloat16)
    assert torch.equal(bf16_round(Y32), Y16)
    dY = wl.activations(2048, 11008, std=0.01, seed=3).to(DEV)
    dX32 = nf4.nf4_matmul_bwd_dx(dY, q)
    dX16 = nf4.nf4_matmul_bwd_dx(dY, q, out_dtype=torch.bfloat16)
    assert torch.equal(bf16_round(dX32), dX16)


@pytest.mark.parametrize("M", [3, 64, 300, 2048])
def test_accumulate_adds_to_the_output(M):
    """fp32 with splits (small grids add their partial sums into the caller's
    output), fp32 without, and bf16."""
    W = weight_np(512, 3584, 14)
    X = wl.activations(M, 3584, seed=M + 60).to(DEV)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    P = nf4.nf4_matmul_fwd(X, q).double()
    Y0 = torch.from_numpy(wl.normal((M, 512), 1.0, seed=M + 61).numpy()).to(DEV)
    Y = Y0.clone()
    nf4.nf4_matmul_fwd(X, q, out=Y, accumulate=True)
    ref = o.matmul_fwd(X.float().cpu().numpy(), oracle_dequant(W, "nf4"))
    assert_tol((Y.double() - Y0.double()).cpu().numpy(), ref, f"accumulate fwd M={M}")
    assert_tol(P.cpu().numpy(), ref, f"plain fwd M={M}")
    Yb = Y0.to(torch.bfloat16)
    base = Yb.double()
    nf4.nf4_matmul_fwd(X, q, out=Yb, accumulate=True)
    total = ref + base.cpu().numpy()
    assert_tol(Yb.double().cpu().numpy(), total, f"accumulate bf16 M={M}",
               rel=REL_FRO + BF16_U * (1 + REL_FRO), mx=MAX_REL + BF16_U * (1 + MAX_REL))
    dY = wl.activations(M, 512, std=0.01, seed=M + 62).to(DEV)
    dX0 = torch.from_numpy(wl.normal((M, 3584), 0.05, seed=M + 63).numpy()).to(DEV)
    dX = dX0.clone()
    nf4.nf4_matmul_bwd_dx(dY, q, out=dX, accumulate=True)
    dref = o.matmul_bwd_dx(dY.float().cpu().numpy(), oracle_dequant(W, "nf4"))
    assert_tol((dX.double() - dX0.double()).cpu().numpy(), dref, f"accumulate dX M={M}")
    assert nf4.nf4_poll_device_status() == 0


@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
@pytest.mark.parametrize("M", [1, 6, 16, 40])
def test_fwd_group_matches_the_oracle(dtype, M):
    """Weights that share X (rows 520, 136 and 1032 over K = 3584, like a
    q/k/v group) in one small-M launch (M <= 16) or one tensor-core launch
    each (M = 40); every output against the oracle."""
    shapes = [(520, 3584), (136, 3584), (1032, 3584)]
    Ws = [weight_np(r, c, 60 + i) for i, (r, c) in enumerate(shapes)]
    qs = [nf4.nf4_quantize(torch.from_numpy(W).to(DEV), dtype=dtype) for W in Ws]
    X = wl.activations(M, 3584, seed=M + 61)
    Ys = nf4.nf4_matmul_fwd_group(X.to(DEV), qs)
    for W, Y, (r, c) in zip(Ws, Ys, shapes):
        ref = o.matmul_fwd(X.float().numpy(), oracle_dequant(W, dtype))
        assert_tol(Y.cpu().numpy(), ref, f"group {dtype} {r}x{c} M={M}")


@pytest.mark.parametrize("M", [3, 16])
def test_fwd_group_bf16_accumulate_fp16_activations(M):
    """A gate/up-like pair with fp16 activations, adding into bf16 outputs:
    each output is its starting value plus the product, rounded once."""
    shapes = [(264, 2048), (72, 2048)]
    Ws = [weight_np(r, c, 70 + i) for i, (r, c) in enumerate(shapes)]
    qs = [nf4.nf4_quantize(torch.from_numpy(W).to(DEV)) for W in Ws]
    X = wl.activations(M, 2048, seed=M + 71, dtype=torch.float16)
    start = [wl.activations(M, r, seed=M + 72 + i).float() for i, (r, _) in enumerate(shapes)]
    outs = [s.to(torch.bfloat16).to(DEV) for s in start]
    nf4.nf4_matmul_fwd_group(X.to(DEV), qs, outs=outs, accumulate=True)
    for W, Y, s0 in zip(Ws, outs, start):
        ref = o.matmul_fwd(X.float().numpy(), oracle_dequant(W, "nf4")) + \
            s0.to(torch.bfloat16).float().numpy()
        assert_tol(Y.float().cpu().numpy(), ref, f"group accumulate M={M}",
                   rel=REL_FRO + BF16_U * (1 + REL_FRO), mx=MAX_REL + BF16_U * (1 + MAX_REL))


def test_fwd_group_of_one_equals_the_single_call():
    """A group of one weight runs the same launch as nf4_matmul_fwd: the
    outputs are bitwise equal."""
    W = weight_np(4096, 4096, 80)
    q = nf4.nf4_quantize(torch.from_numpy(W).to(DEV))
    X = wl.activations(4, 4096, seed=81).to(DEV)
    (Yg,) = nf4.nf4_matmul_fwd_group(X, [q])
    assert torch.equal(Yg, nf4.nf4_matmul_fwd(X, q))
