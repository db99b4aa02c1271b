"""The C-ABI library loads, exports every symbol the header declares, carries
the oracle's NF4 table bit for bit, and rejects invalid arguments on the host
before touching a device (no compute call is made here)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import dequant_gemm_gb300 as nf4
from oracle import nf4_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf4gemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nf4_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(nf4.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = nf4.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_codebook_matches_oracle_bits():
    got = nf4.nf4_codebook().numpy().astype(np.float32)
    assert np.array_equal(got.view(np.uint32), o.nf4_levels().view(np.uint32))


def test_status_strings():
    for code in range(8):
        assert nf4.status_string(code)
    assert nf4.status_string(99) == "unknown status"


def _weight(rows=8, cols=64, codes=16, a8=16, s2=16, blocksize=64, group=256):
    return nf4.nf4_weight(codes, a8, s2, rows, cols, blocksize, group)


P = 1 << 20   # a fake, 16-byte aligned address: never dereferenced by validation


@pytest.mark.parametrize("blocksize", [32, 128, 0])
def test_quantize_rejects_blocksize(blocksize):
    assert nf4.lib().nf4_quantize(P, 8, 64, blocksize, P, P, P, None) == 4


def test_quantize_rejects_shapes_and_pointers():
    L = nf4.lib()
    assert L.nf4_quantize(P, -1, 64, 64, P, P, P, None) == 2
    assert L.nf4_quantize(P, 8, 96, 64, P, P, P, None) == 2      # cols % 64
    assert L.nf4_quantize(None, 8, 64, 64, P, P, P, None) == 1
    assert L.nf4_quantize(P, 8, 64, 64, P, None, P, None) == 1
    assert L.nf4_quantize(P + 4, 8, 64, 64, P, P, P, None) == 3
    assert L.nf4_quantize(P, 8, 64, 64, P, P + 8, P, None) == 3
    # empty extents are a no-op that touches no pointer
    assert L.nf4_quantize(None, 0, 64, 64, None, None, None, None) == 0
    assert L.nf4_quantize(None, 8, 0, 64, None, None, None, None) == 0


def test_matmul_validation():
    L = nf4.lib()
    w = _weight(codes=P, a8=P, s2=P)
    assert L.nf4_matmul_fwd(P, 4, None, P, None) == 1
    assert L.nf4_matmul_fwd(P, -1, ctypes.byref(w), P, None) == 2
    assert L.nf4_matmul_fwd(P, 0, ctypes.byref(w), None, None) == 0      # M = 0
    bad = _weight(blocksize=32, codes=P, a8=P, s2=P)
    assert L.nf4_matmul_fwd(P, 4, ctypes.byref(bad), P, None) == 4
    bad = _weight(group=128, codes=P, a8=P, s2=P)
    assert L.nf4_matmul_bwd_dx(P, 4, ctypes.byref(bad), P, None) == 4
    rag = _weight(rows=12, codes=P, a8=P, s2=P)                          # rows % 8
    assert L.nf4_matmul_fwd(P, 4, ctypes.byref(rag), P, None) == 2
    assert L.nf4_matmul_bwd_dx(P, 4, ctypes.byref(rag), P, None) == 2
    odd = _weight(cols=96, codes=P, a8=P, s2=P)
    assert L.nf4_matmul_fwd(P, 4, ctypes.byref(odd), P, None) == 2
    nul = _weight(codes=None, a8=P, s2=P)
    assert L.nf4_matmul_fwd(P, 4, ctypes.byref(nul), P, None) == 1
    assert L.nf4_matmul_fwd(None, 4, ctypes.byref(w), P, None) == 1
    assert L.nf4_matmul_bwd_dx(P, 4, ctypes.byref(w), None, None) == 1
    assert L.nf4_matmul_fwd(P + 2, 4, ctypes.byref(w), P, None) == 3
    assert L.nf4_matmul_bwd_dx(P, 4, ctypes.byref(w), P + 4, None) == 3
    mis = _weight(codes=P + 1, a8=P, s2=P)
    assert L.nf4_dequantize(ctypes.byref(mis), P, None) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_device_error():
    L = nf4.lib()
    w = _weight(codes=P, a8=P, s2=P)
    assert L.nf4_quantize(P, 8, 64, 64, P, P, P, None) == 5
    assert L.nf4_matmul_fwd(P, 4, ctypes.byref(w), P, None) == 5


def test_timeout_site_description():
    # kernel << 28 | role << 24 | CTA index, as the device records it
    assert nf4.describe_site(0) == "none"
    assert nf4.describe_site((3 << 28) | (2 << 24) | 77) == "tensor-core input gradient, MMA issuer, CTA 77"
    assert nf4.describe_site((1 << 28) | (1 << 24)) == "small-M forward, copy producer, CTA 0"
    assert nf4.describe_site(-((1 << 32) - ((2 << 28) | (4 << 24) | 5))) == "tensor-core forward, epilogue, CTA 5"


def test_autograd_wrapper_imports_and_validates_without_a_device():
    from dequant_gemm_gb300.autograd import NF4LinearFunction, nf4_linear  # noqa: F401
    q = nf4.NF4Weight(torch.empty(0, dtype=torch.uint8), torch.empty(0, dtype=torch.uint8),
                      torch.empty(0), 8, 64)
    with pytest.raises(ValueError):
        nf4_linear(torch.zeros(2, 64, dtype=torch.float32), q)      # not bf16
    with pytest.raises(ValueError):
        nf4_linear(torch.zeros(2, 32, dtype=torch.bfloat16), q)     # wrong width


def test_fp4_codebook_matches_oracle_bits():
    got = nf4.nf4_codebook("fp4").numpy().astype(np.float32)
    assert np.array_equal(got.view(np.uint32), o.fp4_levels().view(np.uint32))
    buf = (ctypes.c_float * 16)()
    assert nf4.lib().nf4_codebook_of(2, ctypes.cast(buf, ctypes.c_void_p)) == 2   # int8: no table
    assert nf4.lib().nf4_codebook_of(0, None) == 1


def test_quantize_ex_validation():
    L = nf4.lib()
    # dtype / element type
    assert L.nf4_quantize_ex(P, 0, 8, 64, 64, 3, P, P, P, None) == 2
    assert L.nf4_quantize_ex(P, 2, 8, 64, 64, 0, P, P, P, None) == 2       # fp16 weights
    assert L.nf4_quantize_ex(P, 1, 8, 64, 32, 0, P, P, P, None) == 4
    # int8 takes no absmax codes; 4-bit needs them
    assert L.nf4_quantize_ex(P, 0, 8, 64, 64, 2, P, P, P, None) == 1
    assert L.nf4_quantize_ex(P, 0, 8, 64, 64, 1, P, None, P, None) == 1
    assert L.nf4_quantize_ex(P + 8, 1, 8, 64, 64, 2, P, None, P, None) == 3
    assert L.nf4_quantize_ex(None, 1, 0, 64, 64, 2, None, None, None, None) == 0


def test_matmul_ex_validation():
    L = nf4.lib()
    w = _weight(codes=P, a8=P, s2=P)
    f, d = L.nf4_matmul_fwd_ex, L.nf4_matmul_bwd_dx_ex
    assert f(P, 0, 4, ctypes.byref(w), P, 0, 0, None) == 2       # fp32 activations
    assert f(P, 1, 4, ctypes.byref(w), P, 2, 0, None) == 2       # fp16 output
    assert d(P, 2, 4, ctypes.byref(w), P, 0, 4, None) == 2       # unknown flag
    assert f(P, 2, 0, ctypes.byref(w), None, 1, 1, None) == 0    # M = 0
    i8 = nf4.nf4_weight(P, None, P, 8, 64, 64, 0, 2)
    bad_group = nf4.nf4_weight(P, None, P, 8, 64, 64, 256, 2)
    assert f(P, 1, 4, ctypes.byref(bad_group), P, 0, 0, None) == 4
    four_no_group = nf4.nf4_weight(P, P, P, 8, 64, 64, 0, 1)
    assert f(P, 1, 4, ctypes.byref(four_no_group), P, 0, 0, None) == 4
    bad_dtype = nf4.nf4_weight(P, P, P, 8, 64, 64, 256, 7)
    assert d(P, 1, 4, ctypes.byref(bad_dtype), P, 0, 0, None) == 2
    assert f(P, 1, 4, ctypes.byref(i8), P + 4, 1, 0, None) == 3
    mis = nf4.nf4_weight(P, None, P + 4, 8, 64, 64, 0, 2)
    assert L.nf4_dequantize(ctypes.byref(mis), P, None) == 3
    # an empty reduction with accumulate leaves the output alone: no launch
    empty = nf4.nf4_weight(P, P, P, 8, 0, 64, 256, 0)
    assert f(P, 1, 4, ctypes.byref(empty), P, 0, 1, None) == 0
    assert L.nf4_set_mma_wait_limit(0) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_ex_calls_without_device_report_device_error():
    L = nf4.lib()
    i8 = nf4.nf4_weight(P, None, P, 8, 64, 64, 0, 2)
    assert L.nf4_matmul_fwd_ex(P, 2, 4, ctypes.byref(i8), P, 1, 1, None) == 5
    assert L.nf4_quantize_ex(P, 1, 8, 64, 64, 2, P, None, P, None) == 5


def test_matmul_group_validation():
    L = nf4.lib()
    a = nf4.nf4_weight(P, P, P, 8, 64, 64, 256, 0)
    b = nf4.nf4_weight(P, P, P, 24, 64, 64, 256, 0)
    ws = (nf4.nf4_weight * 2)(a, b)
    outs = (ctypes.c_void_p * 2)(P, P)
    g = L.nf4_matmul_fwd_group
    assert g(P, 1, 4, None, 2, outs, 0, 0, None) == 1                 # no weights
    assert g(P, 1, 4, ws, 2, None, 0, 0, None) == 1                   # no outputs
    assert g(P, 1, 4, ws, 0, outs, 0, 0, None) == 2                   # empty group
    assert g(P, 1, 4, (nf4.nf4_weight * 5)(*([a] * 5)), 5,
             (ctypes.c_void_p * 5)(*([P] * 5)), 0, 0, None) == 2      # above NF4_GROUP_MAX
    other_cols = (nf4.nf4_weight * 2)(a, nf4.nf4_weight(P, P, P, 8, 128, 64, 256, 0))
    assert g(P, 1, 4, other_cols, 2, outs, 0, 0, None) == 2
    other_dtype = (nf4.nf4_weight * 2)(a, nf4.nf4_weight(P, P, P, 8, 64, 64, 256, 1))
    assert g(P, 1, 4, other_dtype, 2, outs, 0, 0, None) == 2
    assert g(P, 0, 4, ws, 2, outs, 0, 0, None) == 2                   # fp32 activations
    assert g(P, 1, 4, ws, 2, (ctypes.c_void_p * 2)(P, P + 4), 0, 0, None) == 3
    assert g(P, 1, 4, ws, 2, (ctypes.c_void_p * 2)(P, None), 0, 0, None) == 1
    assert g(P, 1, 0, ws, 2, outs, 0, 0, None) == 0                   # M = 0: nothing to do


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_group_call_without_device_reports_device_error():
    a = nf4.nf4_weight(P, P, P, 8, 64, 64, 256, 0)
    ws = (nf4.nf4_weight * 2)(a, a)
    assert nf4.lib().nf4_matmul_fwd_group(P, 1, 4, ws, 2, (ctypes.c_void_p * 2)(P, P), 0, 0,
                                          None) == 5


def test_dequantize_ex_validation():
    L = nf4.lib()
    w = _weight(codes=P, a8=P, s2=P)
    g = L.nf4_dequantize_ex
    assert g(ctypes.byref(w), P, 3, None) == 2           # unknown output type
    assert g(ctypes.byref(w), P, -1, None) == 2
    assert g(ctypes.byref(w), None, 1, None) == 1        # no output
    assert g(ctypes.byref(w), P + 8, 2, None) == 3       # misaligned output
    empty = nf4.nf4_weight(P, P, P, 0, 64, 64, 256, 0)
    assert g(ctypes.byref(empty), None, 1, None) == 0    # nothing to write
    assert g(None, P, 0, None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_dequantize_ex_without_device_reports_device_error():
    w = _weight(codes=P, a8=P, s2=P)
    for elem in (0, 1, 2):
        assert nf4.lib().nf4_dequantize_ex(ctypes.byref(w), P, elem, None) == 5


def test_dequantize_binding_rejects_bad_output_types():
    w = nf4.NF4Weight(torch.zeros(256, dtype=torch.uint8), torch.zeros(8, dtype=torch.uint8),
                      torch.zeros(1), 8, 64)
    with pytest.raises(ValueError):
        nf4.nf4_dequantize(w, out_dtype=torch.int32)
    with pytest.raises(ValueError):
        nf4.nf4_dequantize(w, out=torch.zeros(8, 64, dtype=torch.float64))
    with pytest.raises(ValueError):
        nf4.nf4_dequantize(w, out=torch.zeros(8, 32, dtype=torch.bfloat16))
