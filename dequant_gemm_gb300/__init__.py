"""GB300-native NF4 quantization and fused NF4-dequant matmul.

A thin Python binding over the C ABI of ``libnf4gemm.so`` (declared in
``include/nf4gemm.h``): the functions below only allocate outputs with
PyTorch, marshal pointers and the current CUDA stream, and raise on a
non-OK status. Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing library is an
error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

BLOCKSIZE = 64
DQ_GROUP = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnf4gemm.so")

STATUS = {
    0: "NF4_OK", 1: "NF4_ERR_NULL", 2: "NF4_ERR_SHAPE", 3: "NF4_ERR_ALIGN",
    4: "NF4_ERR_BLOCKSIZE", 5: "NF4_ERR_DEVICE", 6: "NF4_ERR_LAUNCH",
    7: "NF4_ERR_DEVICE_TIMEOUT",
}

# Every symbol the header declares, for load checks.
EXPORTS = ("nf4_quantize", "nf4_quantize_ex", "nf4_dequantize", "nf4_dequantize_ex", "nf4_matmul_fwd",
           "nf4_matmul_bwd_dx", "nf4_matmul_fwd_ex", "nf4_matmul_bwd_dx_ex", "nf4_matmul_fwd_group",
           "nf4_poll_device_status", "nf4_poll_device_status_site", "nf4_codebook",
           "nf4_codebook_of", "nf4_set_mma_wait_limit", "nf4_last_cuda_error",
           "nf4_status_string")

# Weight data types (nf4_dtype) and element types (nf4_elem) of the C ABI.
DTYPES = {"nf4": 0, "fp4": 1, "int8": 2}
ELEM = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
ACCUMULATE = 1
GROUP_MAX = 4          # NF4_GROUP_MAX


class NF4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: {STATUS.get(status, status)} ({status_string(status)})"
        if status == 6:
            msg += f": {lib().nf4_last_cuda_error().decode()}"
        super().__init__(msg)


class nf4_weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("absmax_q", ctypes.c_void_p),
                ("absmax_scale", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("blocksize", ctypes.c_int32),
                ("dq_group", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m dequant_gemm_gb300.build` "
                    "(the NF4 kernels have no fallback)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
            W = ctypes.POINTER(nf4_weight)
            sig = {
                "nf4_quantize": [vp, i64, i64, i32, vp, vp, vp, vp],
                "nf4_quantize_ex": [vp, i32, i64, i64, i32, i32, vp, vp, vp, vp],
                "nf4_dequantize": [W, vp, vp],
                "nf4_dequantize_ex": [W, vp, i32, vp],
                "nf4_matmul_fwd": [vp, i64, W, vp, vp],
                "nf4_matmul_bwd_dx": [vp, i64, W, vp, vp],
                "nf4_matmul_fwd_ex": [vp, i32, i64, W, vp, i32, i32, vp],
                "nf4_matmul_bwd_dx_ex": [vp, i32, i64, W, vp, i32, i32, vp],
                "nf4_matmul_fwd_group": [vp, i32, i64, W, i32, vp, i32, i32, vp],
                "nf4_poll_device_status": [vp],
                "nf4_poll_device_status_site": [vp, vp],
                "nf4_codebook": [vp],
                "nf4_codebook_of": [i32, vp],
                "nf4_set_mma_wait_limit": [i64],
            }
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int32
            L.nf4_status_string.argtypes = [ctypes.c_int32]
            L.nf4_status_string.restype = ctypes.c_char_p
            L.nf4_last_cuda_error.argtypes = []
            L.nf4_last_cuda_error.restype = ctypes.c_char_p
            _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().nf4_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise NF4Error(fn, status)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


@dataclass
class NF4Weight:
    """A quantized weight: codes, scales, shape and data type (the QuantState
    of the bitsandbytes page). Plain tensors; save them with torch.save.

    dtype "nf4" / "fp4": codes uint8 [rows*cols/2] (two 4-bit codes a byte),
    absmax_q uint8 [rows*cols/64], absmax_scale float32 [ceil(rows*cols/16384)].
    dtype "int8": codes int8 [rows*cols], absmax_q None, absmax_scale float32
    [rows*cols/64] (the fp32 absmax of each 64-weight block)."""
    codes: torch.Tensor
    absmax_q: torch.Tensor | None
    absmax_scale: torch.Tensor
    rows: int
    cols: int
    dtype: str = "nf4"

    def c_struct(self) -> nf4_weight:
        four = self.dtype != "int8"
        return nf4_weight(self.codes.data_ptr(),
                          self.absmax_q.data_ptr() if four else None,
                          self.absmax_scale.data_ptr(), self.rows, self.cols, BLOCKSIZE,
                          DQ_GROUP if four else 0, DTYPES[self.dtype])

    @property
    def device(self) -> torch.device:
        return self.codes.device

    def nbytes(self) -> int:
        n = self.codes.numel() * self.codes.element_size() + 4 * self.absmax_scale.numel()
        return n + (self.absmax_q.numel() if self.absmax_q is not None else 0)


def _require(t, name: str, dtype: torch.dtype, shape=None, numel=None):
    """Dtype, contiguity and extent of one tensor argument (no device check)."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")


def _same_device(device: torch.device, **tensors):
    for name, t in tensors.items():
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")


def _require_cuda_device(device: torch.device):
    """Checked last, after every shape and device-equality check, so that the
    host-side checks can be exercised on CPU tensors."""
    if device.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {device}")


def _check_weight(w: "NF4Weight", device: torch.device):
    """The arrays of a quantized weight: dtypes, exact sizes for its shape and
    data type, contiguity, and the device of the call."""
    if w.dtype not in DTYPES:
        raise ValueError(f"unknown weight dtype {w.dtype!r}; expected one of {sorted(DTYPES)}")
    if w.rows < 0 or w.cols < 0 or w.cols % BLOCKSIZE:
        raise ValueError(f"weight shape {w.rows}x{w.cols}: cols must be a multiple of {BLOCKSIZE}")
    n = w.rows * w.cols
    nb = n // BLOCKSIZE
    if w.dtype == "int8":
        _require(w.codes, "weight.codes", torch.int8, numel=n)
        if w.absmax_q is not None:
            raise ValueError("an int8 weight has no absmax_q")
        _require(w.absmax_scale, "weight.absmax_scale", torch.float32, numel=nb)
        _same_device(device, **{"weight.codes": w.codes, "weight.absmax_scale": w.absmax_scale})
        return
    _require(w.codes, "weight.codes", torch.uint8, numel=n // 2)
    _require(w.absmax_q, "weight.absmax_q", torch.uint8, numel=nb)
    _require(w.absmax_scale, "weight.absmax_scale", torch.float32,
             numel=(nb + DQ_GROUP - 1) // DQ_GROUP)
    _same_device(device, **{"weight.codes": w.codes, "weight.absmax_q": w.absmax_q,
                            "weight.absmax_scale": w.absmax_scale})


def alloc_weight(rows: int, cols: int, device, dtype: str = "nf4") -> NF4Weight:
    if dtype not in DTYPES:
        raise ValueError(f"unknown weight dtype {dtype!r}")
    n = rows * cols
    nb = n // BLOCKSIZE
    if dtype == "int8":
        return NF4Weight(torch.empty(n, dtype=torch.int8, device=device), None,
                         torch.empty(nb, dtype=torch.float32, device=device), rows, cols, dtype)
    ng = (nb + DQ_GROUP - 1) // DQ_GROUP
    return NF4Weight(torch.empty(n // 2, dtype=torch.uint8, device=device),
                     torch.empty(nb, dtype=torch.uint8, device=device),
                     torch.empty(ng, dtype=torch.float32, device=device), rows, cols, dtype)


def nf4_quantize(W: torch.Tensor, out: NF4Weight | None = None,
                 dtype: str = "nf4") -> NF4Weight:
    """Quantize an fp32 or bf16 [rows, cols] CUDA tensor (blocksize 64):
    dtype "nf4" or "fp4" (double-quantized absmax) or "int8"."""
    if not isinstance(W, torch.Tensor) or W.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"W must be float32 or bfloat16, got {getattr(W, 'dtype', type(W))}")
    _require(W, "W", W.dtype)
    if W.dim() != 2:
        raise ValueError("W must be 2-D [rows, cols]")
    if dtype not in DTYPES:
        raise ValueError(f"unknown weight dtype {dtype!r}")
    rows, cols = W.shape
    if cols % BLOCKSIZE:
        raise ValueError(f"cols = {cols} is not a multiple of {BLOCKSIZE}")
    if out is not None:
        if (out.rows, out.cols) != (rows, cols):
            raise ValueError(f"out is a {out.rows}x{out.cols} weight, W is {rows}x{cols}")
        if out.dtype != dtype:
            raise ValueError(f"out holds a {out.dtype} weight, asked for {dtype}")
        _check_weight(out, W.device)
    _require_cuda_device(W.device)
    q = out if out is not None else alloc_weight(rows, cols, W.device, dtype)
    with torch.cuda.device(W.device):
        _check("nf4_quantize_ex", lib().nf4_quantize_ex(
            _ptr(W), ELEM[W.dtype], rows, cols, BLOCKSIZE, DTYPES[dtype], _ptr(q.codes),
            _ptr(q.absmax_q), _ptr(q.absmax_scale), _stream(W.device)))
    return q


def nf4_dequantize(w: NF4Weight, out: torch.Tensor | None = None,
                   out_dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """[rows, cols] dequantized weight in fp32, or rounded to nearest even in
    bf16 or fp16 (for export and for library GEMMs)."""
    if out is not None:
        if not isinstance(out, torch.Tensor):
            raise ValueError("out must be a tensor")
        out_dtype = out.dtype
    if out_dtype not in ELEM:
        raise ValueError(f"nf4_dequantize: output dtype {out_dtype} is not fp32, bf16 or fp16")
    _check_weight(w, w.device)
    if out is not None:
        _require(out, "out", out_dtype, shape=(w.rows, w.cols))
        _same_device(w.device, out=out)
    _require_cuda_device(w.device)
    y = out if out is not None else torch.empty(w.rows, w.cols, dtype=out_dtype, device=w.device)
    s = w.c_struct()
    with torch.cuda.device(w.device):
        _check("nf4_dequantize_ex", lib().nf4_dequantize_ex(ctypes.byref(s), _ptr(y), ELEM[out_dtype],
                                                           _stream(w.device)))
    return y


def _matmul(name: str, fn: str, A: torch.Tensor, w: NF4Weight, width: int, out_cols: int,
            out, out_dtype, accumulate: bool) -> torch.Tensor:
    if not isinstance(A, torch.Tensor) or A.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"{name} must be bfloat16 or float16, got {getattr(A, 'dtype', type(A))}")
    _require(A, name, A.dtype)
    if A.dim() != 2 or A.shape[1] != width:
        raise ValueError(f"{name} must be [M, {width}]")
    M = A.shape[0]
    _check_weight(w, A.device)
    if out is not None:
        out_dtype = out.dtype
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"the output must be float32 or bfloat16, got {out_dtype}")
    if out is not None:
        _require(out, "out", out_dtype, shape=(M, out_cols))
        _same_device(A.device, out=out)
    elif accumulate:
        raise ValueError("accumulate=True needs the output tensor to add to (out=)")
    _require_cuda_device(A.device)
    y = out if out is not None else torch.empty(M, out_cols, dtype=out_dtype, device=A.device)
    s = w.c_struct()
    with torch.cuda.device(A.device):
        _check(fn, getattr(lib(), fn)(_ptr(A), ELEM[A.dtype], M, ctypes.byref(s), _ptr(y),
                                      ELEM[out_dtype], ACCUMULATE if accumulate else 0,
                                      _stream(A.device)))
    return y


def nf4_matmul_fwd(X: torch.Tensor, w: NF4Weight, out: torch.Tensor | None = None,
                   out_dtype: torch.dtype = torch.float32, accumulate: bool = False) -> torch.Tensor:
    """Y = X * dequant(W)^T (+ out when accumulate): X bf16 or fp16 [M, cols]
    -> Y fp32 or bf16 [M, rows]."""
    return _matmul("X", "nf4_matmul_fwd_ex", X, w, w.cols, w.rows, out, out_dtype, accumulate)


def nf4_matmul_fwd_group(X: torch.Tensor, ws, outs=None, out_dtype: torch.dtype = torch.float32,
                         accumulate: bool = False) -> list:
    """Y_i = X * dequant(W_i)^T (+ outs[i] when accumulate) for up to
    GROUP_MAX weights that share X (same cols and data type, rows may
    differ); one launch of the small-M kernel for M <= 16. Returns the
    outputs, fp32 or bf16 [M, rows_i]."""
    ws = list(ws)
    if not 1 <= len(ws) <= GROUP_MAX:
        raise ValueError(f"a group has 1 to {GROUP_MAX} weights, got {len(ws)}")
    if not isinstance(X, torch.Tensor) or X.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError(f"X must be bfloat16 or float16, got {getattr(X, 'dtype', type(X))}")
    _require(X, "X", X.dtype)
    K = ws[0].cols
    if X.dim() != 2 or X.shape[1] != K:
        raise ValueError(f"X must be [M, {K}]")
    M = X.shape[0]
    for w in ws:
        if w.cols != K or w.dtype != ws[0].dtype:
            raise ValueError("the weights of a group must share cols and dtype")
        _check_weight(w, X.device)
    if outs is not None:
        outs = list(outs)
        if len(outs) != len(ws):
            raise ValueError("one output per weight")
        out_dtype = outs[0].dtype
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"the output must be float32 or bfloat16, got {out_dtype}")
    if outs is not None:
        for o, w in zip(outs, ws):
            _require(o, "out", out_dtype, shape=(M, w.rows))
            _same_device(X.device, out=o)
    elif accumulate:
        raise ValueError("accumulate=True needs the output tensors to add to (outs=)")
    _require_cuda_device(X.device)
    if outs is None:
        outs = [torch.empty(M, w.rows, dtype=out_dtype, device=X.device) for w in ws]
    structs = (nf4_weight * len(ws))(*[w.c_struct() for w in ws])
    ptrs = (ctypes.c_void_p * len(ws))(*[o.data_ptr() for o in outs])
    with torch.cuda.device(X.device):
        _check("nf4_matmul_fwd_group",
               lib().nf4_matmul_fwd_group(_ptr(X), ELEM[X.dtype], M, structs, len(ws),
                                          ctypes.cast(ptrs, ctypes.c_void_p),
                                          ELEM[out_dtype], ACCUMULATE if accumulate else 0,
                                          _stream(X.device)))
    return outs


def nf4_matmul_bwd_dx(dY: torch.Tensor, w: NF4Weight, out: torch.Tensor | None = None,
                      out_dtype: torch.dtype = torch.float32,
                      accumulate: bool = False) -> torch.Tensor:
    """dX = dY * dequant(W) (+ out when accumulate): dY bf16 or fp16 [M, rows]
    -> dX fp32 or bf16 [M, cols]. No dW."""
    return _matmul("dY", "nf4_matmul_bwd_dx_ex", dY, w, w.rows, w.cols, out, out_dtype,
                   accumulate)


def nf4_set_mma_wait_limit(cycles: int = 0) -> None:
    """Diagnostic: the tensor-core kernels' MMA issuer gives up waiting for a
    stage after `cycles` clock cycles (0 restores the default of about a
    second). For testing the timeout path only."""
    _check("nf4_set_mma_wait_limit", lib().nf4_set_mma_wait_limit(int(cycles)))


def nf4_poll_device_status(device=None) -> int:
    """Synchronize the current stream and return (and clear) the device status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().nf4_poll_device_status(_stream(dev)))


def nf4_poll_device_status_site(device=None) -> tuple[int, int]:
    """As nf4_poll_device_status, plus where the first timeout happened:
    (status, site), site = kernel << 28 | role << 24 | CTA index (0 if none)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    site = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        st = int(lib().nf4_poll_device_status_site(_stream(dev), ctypes.byref(site)))
    return st, int(site.value)


def describe_site(site: int) -> str:
    """Readable form of a timeout site."""
    if site == 0:
        return "none"
    kernel = {1: "small-M forward", 2: "tensor-core forward", 3: "tensor-core input gradient"}
    role = {1: "copy producer", 2: "MMA issuer", 3: "dequantizing warp", 4: "epilogue"}
    u = site & 0xffffffff
    return (f"{kernel.get(u >> 28, u >> 28)}, {role.get((u >> 24) & 15, (u >> 24) & 15)}, "
            f"CTA {u & 0xffffff}")


def nf4_codebook(dtype: str = "nf4") -> torch.Tensor:
    """The 16 fp32 levels of a 4-bit dtype compiled into the library, by code
    (host only)."""
    buf = (ctypes.c_float * 16)()
    _check("nf4_codebook_of", lib().nf4_codebook_of(DTYPES[dtype], ctypes.cast(buf, ctypes.c_void_p)))
    return torch.tensor(list(buf), dtype=torch.float32)
