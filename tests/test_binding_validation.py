"""Host-side argument checks of the Python binding, run on CPU tensors: every
malformed call raises ValueError before anything reaches the library (an
undersized output or a weight on another device would otherwise be written
or read out of bounds by the kernels)."""
import pytest
import torch

import dequant_gemm_gb300 as nf4


def weight(rows=16, cols=128, device="cpu"):
    return nf4.alloc_weight(rows, cols, device)


def test_fwd_rejects_bad_out():
    X = torch.zeros(4, 128, dtype=torch.bfloat16)
    w = weight()
    with pytest.raises(ValueError, match="shape"):
        nf4.nf4_matmul_fwd(X, w, out=torch.empty(4, 15))
    with pytest.raises(ValueError, match="shape"):
        nf4.nf4_matmul_fwd(X, w, out=torch.empty(64))
    with pytest.raises(ValueError, match="float32"):
        nf4.nf4_matmul_fwd(X, w, out=torch.empty(4, 16, dtype=torch.float16))
    with pytest.raises(ValueError, match="contiguous"):
        nf4.nf4_matmul_fwd(X, w, out=torch.empty(16, 4).t())


def test_dx_rejects_bad_out():
    dY = torch.zeros(4, 16, dtype=torch.bfloat16)
    w = weight()
    with pytest.raises(ValueError, match="shape"):
        nf4.nf4_matmul_bwd_dx(dY, w, out=torch.empty(4, 16))
    with pytest.raises(ValueError, match="contiguous"):
        nf4.nf4_matmul_bwd_dx(dY, w, out=torch.empty(128, 4).t())


def test_rejects_weight_arrays_of_the_wrong_size_or_type():
    X = torch.zeros(2, 128, dtype=torch.bfloat16)
    w = weight()
    short = nf4.NF4Weight(w.codes[:-1], w.absmax_q, w.absmax_scale, 16, 128)
    with pytest.raises(ValueError, match="codes"):
        nf4.nf4_matmul_fwd(X, short)
    bad_a8 = nf4.NF4Weight(w.codes, w.absmax_q[:16], w.absmax_scale, 16, 128)
    with pytest.raises(ValueError, match="absmax_q"):
        nf4.nf4_matmul_fwd(X, bad_a8)
    bad_s2 = nf4.NF4Weight(w.codes, w.absmax_q, w.absmax_scale.double(), 16, 128)
    with pytest.raises(ValueError, match="absmax_scale"):
        nf4.nf4_dequantize(bad_s2)
    odd = nf4.NF4Weight(w.codes, w.absmax_q, w.absmax_scale, 32, 64 + 32)
    with pytest.raises(ValueError, match="multiple"):
        nf4.nf4_matmul_fwd(torch.zeros(2, 96, dtype=torch.bfloat16), odd)


def test_rejects_tensors_on_another_device():
    X = torch.zeros(2, 128, dtype=torch.bfloat16)
    w_meta = weight(device="meta")
    with pytest.raises(ValueError, match="expected cpu"):
        nf4.nf4_matmul_fwd(X, w_meta)
    w = weight()
    with pytest.raises(ValueError, match="expected cpu"):
        nf4.nf4_matmul_fwd(X, w, out=torch.empty(2, 16, device="meta"))
    with pytest.raises(ValueError, match="expected cpu"):
        nf4.nf4_matmul_bwd_dx(torch.zeros(2, 16, dtype=torch.bfloat16), w_meta)
    with pytest.raises(ValueError, match="expected meta"):
        nf4.nf4_dequantize(w_meta, out=torch.empty(16, 128))


def test_quantize_rejects_bad_out_weight():
    W = torch.zeros(16, 128)
    with pytest.raises(ValueError, match="16x64"):
        nf4.nf4_quantize(W, out=weight(16, 64))
    with pytest.raises(ValueError, match="multiple"):
        nf4.nf4_quantize(torch.zeros(4, 96))
    with pytest.raises(ValueError, match="float32"):
        nf4.nf4_quantize(W.double())
    with pytest.raises(ValueError, match="expected cpu"):
        nf4.nf4_quantize(W, out=weight(device="meta"))


def test_well_formed_cpu_call_is_refused_for_the_device_alone():
    X = torch.zeros(2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA device"):
        nf4.nf4_matmul_fwd(X, weight(), out=torch.empty(2, 16))
    with pytest.raises(ValueError, match="CUDA device"):
        nf4.nf4_quantize(torch.zeros(16, 128))


def test_int8_and_fp4_weights_are_checked_by_their_own_layout():
    X = torch.zeros(2, 128, dtype=torch.float16)
    w8 = nf4.alloc_weight(16, 128, "cpu", "int8")
    assert w8.codes.dtype == torch.int8 and w8.absmax_q is None and w8.absmax_scale.numel() == 32
    with pytest.raises(ValueError, match="CUDA device"):
        nf4.nf4_matmul_fwd(X, w8)
    bad = nf4.NF4Weight(w8.codes, None, w8.absmax_scale[:-1], 16, 128, "int8")
    with pytest.raises(ValueError, match="absmax_scale"):
        nf4.nf4_matmul_fwd(X, bad)
    mixed = nf4.NF4Weight(w8.codes, torch.empty(32, dtype=torch.uint8), w8.absmax_scale, 16, 128,
                          "int8")
    with pytest.raises(ValueError, match="no absmax_q"):
        nf4.nf4_matmul_fwd(X, mixed)
    w4 = nf4.alloc_weight(16, 128, "cpu", "fp4")
    as_int8 = nf4.NF4Weight(w4.codes, None, w4.absmax_scale, 16, 128, "int8")
    with pytest.raises(ValueError, match="int8"):
        nf4.nf4_matmul_fwd(X, as_int8)
    with pytest.raises(ValueError, match="dtype"):
        nf4.alloc_weight(16, 128, "cpu", "int4")


def test_element_types_and_accumulate_are_checked():
    w = weight()
    with pytest.raises(ValueError, match="bfloat16 or float16"):
        nf4.nf4_matmul_fwd(torch.zeros(2, 128), w)
    with pytest.raises(ValueError, match="float32 or bfloat16"):
        nf4.nf4_matmul_fwd(torch.zeros(2, 128, dtype=torch.bfloat16), w, out_dtype=torch.float16)
    with pytest.raises(ValueError, match="accumulate"):
        nf4.nf4_matmul_bwd_dx(torch.zeros(2, 16, dtype=torch.float16), w, accumulate=True)
    with pytest.raises(ValueError, match="shape"):
        nf4.nf4_matmul_fwd(torch.zeros(2, 128, dtype=torch.bfloat16), w,
                           out=torch.empty(2, 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="float32 or bfloat16"):
        nf4.nf4_quantize(torch.zeros(16, 128, dtype=torch.float16))
    with pytest.raises(ValueError, match="nf4"):
        nf4.nf4_quantize(torch.zeros(16, 128), out=nf4.alloc_weight(16, 128, "cpu", "fp4"))
    with pytest.raises(ValueError, match="CUDA device"):
        nf4.nf4_quantize(torch.zeros(16, 128, dtype=torch.bfloat16), dtype="int8")
