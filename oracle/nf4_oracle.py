"""Plain, slow CPU oracle for NF4 blockwise quantization with double-quantized
absmax scales, dequantization, and the NF4-dequant matmul (forward and the
frozen-base input gradient).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code, table or constant generator with
the CUDA library; the two meet only on seeded inputs.

Every function computes the plain definition of one step, in the order the
method states it, with numpy:

* floating point decisions that the method fixes to fp32 (the normalisation
  ``w / absmax``, the double-quant rounding, the dequant products) are taken in
  numpy float32, which rounds each operation to nearest-even exactly as IEEE
  fp32 does;
* everything else (the NF4 level construction, nearest-level distances, the
  matmuls) is fp64.

Sources (page title, section):

* "Zenbit" (pypi.org/project/zenbit), "What's inside", ``zenbit.nf4`` bullet:
  NF4 blockwise quantization with double quantization, QLoRA style.
* same page, ``zenbit.pallas_nf4`` bullet: fused dequant + matmul with the
  full-precision weight never materialised; backward computes dL/dX only.
* "bitsandbytes" (unfragile.ai/artifact/bitsandbytes), NF4 paragraph: 16 levels
  from the inverse normal CDF, more levels near zero, values mapped through a
  lookup table, per-block scale.
* same page, double-quantization paragraph: absmax per 64-weight block, the
  absmax vector itself quantized to 8 bits with its own scale; at dequant time
  the scales are dequantized first, then the weights.
* same page, quantized-GEMM paragraph: dequantize on the fly, fp32 output;
  weights int8 or 4-bit, activations float16/float32.
* same page, 4-bit paragraph: NF4 or FP4 (standard floating-point 4-bit) data
  types with double quantization of the scales.
* "Zenbit", ``zenbit.int8`` bullet: uniform int8 weight quantization.

Where the pages leave a step open, the reading taken is stated in the
docstring of the function that takes it.

Parity status per function:
  nf4_levels        pinned (second inverse-CDF routine, forward CDF, invariants)
  nearest_code      pinned (exact rational brute force, midpoint counting)
  quantize_codes    pinned (exact-rational IEEE quotient on every decision edge;
                    a reciprocal multiply or the dequantized absmax fail it)
  double_quant      pinned (exact halves round to even, exact multiply-then-
                    divide chain; half-up and divide-first fail it)
  quantize_flat     pinned (special cases, round-trip bound, brute force)
  dequant_absmax    pinned (exact product-then-quotient chain)
  dequantize_codes  pinned (one exactly rounded product per weight)
  dequantize_flat   pinned (round-trip bound, special cases)
  matmul_fwd        pinned (one-hot rows, exact small integer case)
  matmul_bwd_dx     pinned (transpose identity against matmul_fwd, one-hot rows)
  fp4_levels        pinned (E2M1 decode from the format definition, exact)
  quantize_flat / dequantize_flat with the FP4 table
                    pinned (exact brute-force nearest incl. the signed-zero tie,
                    special cases, round-trip bound)
  int8_quantize_flat, int8_dequantize_flat
                    pinned (exact multiply-then-divide chain, halves to even,
                    range, round-trip bound, memory invariant)
  bf16_to_fp32      pinned (all 65536 bit patterns against torch's conversion)
"""
from __future__ import annotations

from statistics import NormalDist

import numpy as np

BLOCKSIZE = 64     # weights per absmax block ("absmax per 64-weight block")
DQ_GROUP = 256     # absmax values per second-level fp32 scale


# --------------------------------------------------------------------------
# NF4 levels
# --------------------------------------------------------------------------
def nf4_levels_fp64() -> np.ndarray:
    """The 16 NF4 levels in fp64, before rounding to fp32.

    The pages say only that the levels come from the inverse normal CDF, that
    they crowd near zero, and (for this build) that there are 7 negative
    levels, an exact zero and 8 positive levels normalised to [-1, 1].
    Reading taken (the QLoRA construction, Dettmers et al. 2023, restated from
    its definition): with delta = ((1 - 1/30) + (1 - 1/32)) / 2,

      positive levels = Phi^-1(p) for p on the 9-point grid from delta to 1/2,
                        last point (p = 1/2, i.e. 0) dropped          -> 8 values
      negative levels = -Phi^-1(p) for p on the 8-point grid from delta
                        to 1/2, last point dropped                    -> 7 values
      plus an exact 0, sorted, all divided by Phi^-1(delta).
    """
    inv = NormalDist().inv_cdf
    delta = 0.5 * ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0))
    pos = [inv(p) for p in np.linspace(delta, 0.5, 9)[:-1]]
    neg = [-inv(p) for p in np.linspace(delta, 0.5, 8)[:-1]]
    top = inv(delta)
    levels = sorted(pos + neg + [0.0])
    return np.array([v / top for v in levels], dtype=np.float64)


def nf4_levels() -> np.ndarray:
    """NF4 levels rounded once, to nearest-even, to fp32 (the stored table)."""
    return nf4_levels_fp64().astype(np.float32)


def fp4_levels() -> np.ndarray:
    """The 16 FP4 levels, indexed by the 4-bit code (fp32).

    The "bitsandbytes" page names FP4 "standard floating-point 4-bit" beside
    NF4, with the same blockwise scaling and double quantization. Reading
    taken: the E2M1 layout, code = sign (bit 3) | exponent (bits 2-1) |
    mantissa (bit 0), exponent bias 1, exponent 0 subnormal:
      magnitude = m / 2                     if e == 0
                = 2^(e-1) * (1 + m / 2)     otherwise,
    i.e. 0, 0.5, 1, 1.5, 2, 3, 4, 6; normalised to [-1, 1] by the largest
    magnitude 6 like the NF4 levels. Computed in fp64 and rounded once to
    fp32 (the thirds have non-terminating binary expansions, so no fp32 tie
    arises for the double rounding to break). Code 8 is -0.0.
    """
    out = np.empty(16, dtype=np.float64)
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m / 2.0 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
        out[code] = (-mag if s else mag) / 6.0
    return out.astype(np.float32)


def levels_of(dtype: str) -> np.ndarray:
    """The fp32 table of a 4-bit data type ("nf4" or "fp4")."""
    if dtype == "nf4":
        return nf4_levels()
    if dtype == "fp4":
        return fp4_levels()
    raise ValueError(f"no 4-bit table for {dtype!r}")


def zero_code(levels: np.ndarray) -> int:
    """The code an all-zero block gets: the first index holding level 0
    (NF4: 7; FP4: 0, ahead of -0.0 at 8)."""
    return int(np.flatnonzero(levels == 0)[0])


# --------------------------------------------------------------------------
# Quantization
# --------------------------------------------------------------------------
def nearest_code(x: np.ndarray, levels: np.ndarray | None = None) -> np.ndarray:
    """Index of the NF4 level nearest to each fp32 value in ``x``.

    Ties go to the lower index (np.argmin returns the first minimum).

    The distances are taken in fp64. For fp32 operands x and c in [-1, 1]
    the difference x - c is exact in fp64 whenever |x| >= 2**-29 (both are
    multiples of 2**-52 and smaller than 2 in magnitude), and subtracting the
    level 0 is always exact; the only inexact case, 0 < |x| < 2**-29, is
    nearest to level 0 by a margin of 0.079 that no rounding can close. So the
    argmin below is the exact nearest level.
    """
    lv = (nf4_levels() if levels is None else levels).astype(np.float64)
    xd = np.asarray(x, dtype=np.float32).astype(np.float64)
    dist = np.abs(xd[..., None] - lv)
    return np.argmin(dist, axis=-1).astype(np.uint8)


def block_absmax(w_flat: np.ndarray) -> np.ndarray:
    """Per-64-block max |w| (exact in fp32)."""
    return np.max(np.abs(w_flat.reshape(-1, BLOCKSIZE)), axis=1).astype(np.float32)


def quantize_codes(w_flat: np.ndarray, absmax: np.ndarray,
                   levels: np.ndarray | None = None) -> np.ndarray:
    """4-bit codes of every weight: nearest level of w / absmax (NF4 table
    unless another 4-bit table is given).

    Readings taken: the normalisation is the IEEE fp32 quotient
    fl32(w / absmax) with the block's true fp32 absmax (the scale is computed
    first and only then double-quantized); a block whose absmax is 0 has all
    codes equal to the index of the exact zero level (7 for NF4).
    """
    lv = nf4_levels() if levels is None else levels
    blocks = w_flat.reshape(-1, BLOCKSIZE).astype(np.float32)
    codes = np.full(blocks.shape, zero_code(lv), dtype=np.uint8)
    nz = absmax > 0
    rows = np.flatnonzero(nz)
    step = 1 << 12                                # bounded temporaries
    for i0 in range(0, rows.size, step):
        r = rows[i0:i0 + step]
        x = blocks[r] / absmax[r, None]           # float32 / float32: IEEE RN
        codes[r] = nearest_code(x, lv)
    return codes.reshape(-1)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Two codes per byte, the even-indexed element in the high nibble."""
    c = codes.reshape(-1, 2).astype(np.uint8)
    return ((c[:, 0] << 4) | c[:, 1]).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p >> 4
    out[1::2] = p & 15
    return out


def double_quant(absmax: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """8-bit double quantization of the absmax vector.

    s2_g = max of the absmax values in group g (256 consecutive blocks, the
    last group possibly shorter); a8 = round(255 * absmax / s2_g) as uint8.
    Readings taken: the product 255 * absmax and the quotient are each rounded
    to fp32, the multiply first; "round" is round-half-to-even of the fp32
    quotient; a group whose s2 is 0 stores a8 = 0.
    """
    nb = absmax.size
    ng = (nb + DQ_GROUP - 1) // DQ_GROUP
    s2 = np.empty(ng, dtype=np.float32)
    a8 = np.empty(nb, dtype=np.uint8)
    for g in range(ng):
        seg = absmax[g * DQ_GROUP:(g + 1) * DQ_GROUP].astype(np.float32)
        s = np.float32(seg.max())
        s2[g] = s
        if s == 0:
            a8[g * DQ_GROUP:(g + 1) * DQ_GROUP] = 0
        else:
            q = (np.float32(255.0) * seg) / s          # fp32 RN, multiply first
            a8[g * DQ_GROUP:(g + 1) * DQ_GROUP] = np.rint(q).astype(np.uint8)
    return a8, s2


def quantize_flat(w_flat: np.ndarray, levels: np.ndarray | None = None):
    """NF4 (or, given its table, FP4) + double-quant of a row-major flattened
    fp32 weight.

    Blocks of 64 and groups of 256 blocks run over the flattened weight.
    Returns (packed codes uint8 [n/2], a8 uint8 [n/64], s2 fp32 [ceil(n/16384)]).
    A slice of a larger weight that starts on a group boundary (a multiple of
    16384 elements) gives exactly the outputs of those groups.
    """
    w = np.ascontiguousarray(w_flat, dtype=np.float32).reshape(-1)
    assert w.size % BLOCKSIZE == 0
    absmax = block_absmax(w)
    codes = quantize_codes(w, absmax, levels)
    a8, s2 = double_quant(absmax)
    return pack_nibbles(codes), a8, s2


def quantize(W: np.ndarray, levels: np.ndarray | None = None):
    """quantize_flat over W [rows, cols] in row-major order."""
    return quantize_flat(np.asarray(W, dtype=np.float32).reshape(-1), levels)


# --------------------------------------------------------------------------
# Dequantization
# --------------------------------------------------------------------------
def dequant_absmax(a8: np.ndarray, s2: np.ndarray) -> np.ndarray:
    """Scales first: ahat = fl32(fl32(a8 * s2) / 255) for each block.

    Reading taken: the plain inverse of the double quantization, each of the
    two operations rounded to fp32.
    """
    g = np.arange(a8.size) // DQ_GROUP
    prod = a8.astype(np.float32) * s2[g]               # fp32 RN
    return (prod / np.float32(255.0)).astype(np.float32)


def dequantize_codes(codes: np.ndarray, ahat: np.ndarray,
                     levels: np.ndarray | None = None) -> np.ndarray:
    """Weights second: what = fl32(c[q] * ahat) for codes [nblocks, 64] and the
    blocks' dequantized absmax [nblocks] (fp32 [nblocks, 64])."""
    lv = nf4_levels() if levels is None else levels
    q = np.asarray(codes, dtype=np.uint8).reshape(-1, BLOCKSIZE)
    return (lv[q] * np.asarray(ahat, dtype=np.float32)[:, None]).astype(np.float32)


def dequantize_flat(packed: np.ndarray, a8: np.ndarray, s2: np.ndarray,
                    levels: np.ndarray | None = None) -> np.ndarray:
    """Dequantize a whole flat weight (fp32 [n])."""
    ahat = dequant_absmax(a8, s2)
    return dequantize_codes(unpack_nibbles(packed), ahat, levels).reshape(-1)


def dequantize(packed, a8, s2, rows: int, cols: int,
               levels: np.ndarray | None = None) -> np.ndarray:
    return dequantize_flat(packed, a8, s2, levels).reshape(rows, cols)


# --------------------------------------------------------------------------
# Uniform int8 weight quantization
# --------------------------------------------------------------------------
def int8_quantize_flat(w_flat: np.ndarray):
    """Uniform symmetric int8 quantization per 64-weight block ("Zenbit",
    zenbit.int8 bullet: uniform int8 weight quantization; "bitsandbytes",
    CPU paragraph: int8 dequantization with per-block scaling factors).

    Readings taken: the block is the NF4 path's 64-weight block over the
    row-major flattened weight; a = max |w| of the block, kept in fp32 (no
    double quantization); q = rint(fl32(fl32(127 w) / a)), the multiply
    first and round-half-to-even as in the double quantization; q = 0 when
    a = 0. Returns (q int8 [n], a fp32 [n/64]).
    """
    w = np.ascontiguousarray(w_flat, dtype=np.float32).reshape(-1, BLOCKSIZE)
    a = block_absmax(w)
    q = np.zeros(w.shape, dtype=np.int8)
    nz = np.flatnonzero(a > 0)
    step = 1 << 14
    for i0 in range(0, nz.size, step):
        r = nz[i0:i0 + step]
        t = (np.float32(127.0) * w[r]) / a[r, None]      # fp32 RN, multiply first
        q[r] = np.rint(t).astype(np.int8)
    return q.reshape(-1), a


def int8_dequantize_flat(q: np.ndarray, absmax: np.ndarray) -> np.ndarray:
    """what = fl32(fl32(q * a) / 127): the inverse of int8_quantize_flat,
    each operation rounded to fp32 (fp32 [n])."""
    qb = np.asarray(q, dtype=np.int8).reshape(-1, BLOCKSIZE).astype(np.float32)
    prod = qb * np.asarray(absmax, dtype=np.float32)[:, None]
    return (prod / np.float32(127.0)).astype(np.float32).reshape(-1)


# --------------------------------------------------------------------------
# bf16 inputs
# --------------------------------------------------------------------------
def bf16_to_fp32(bits: np.ndarray) -> np.ndarray:
    """The fp32 value of each bf16 bit pattern: bf16 is the upper half of an
    fp32 (sign, 8 exponent bits, 7 fraction bits), so the value is exact.
    A bf16 weight is quantized as this fp32 weight."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


# --------------------------------------------------------------------------
# Matmuls (fp64 dequantize-then-multiply)
# --------------------------------------------------------------------------
def matmul_fwd(X: np.ndarray, W_hat: np.ndarray) -> np.ndarray:
    """Y[m, n] = sum_k X[m, k] * What[n, k], in fp64.

    X holds the (bf16) activations as exact fp32/fp64 values; W_hat is the
    fp32 dequantized weight [N, K].
    """
    return np.asarray(X, dtype=np.float64) @ np.asarray(W_hat, dtype=np.float64).T


def matmul_bwd_dx(dY: np.ndarray, W_hat: np.ndarray) -> np.ndarray:
    """dX[m, k] = sum_n dY[m, n] * What[n, k], in fp64. dW is not computed."""
    return np.asarray(dY, dtype=np.float64) @ np.asarray(W_hat, dtype=np.float64)


# --------------------------------------------------------------------------
# Error measures used by the tolerance checks
# --------------------------------------------------------------------------
def rel_frobenius(Y: np.ndarray, Y_ref: np.ndarray) -> float:
    Y = np.asarray(Y, dtype=np.float64)
    Y_ref = np.asarray(Y_ref, dtype=np.float64)
    den = np.linalg.norm(Y_ref)
    return float(np.linalg.norm(Y - Y_ref) / den) if den > 0 else float(np.linalg.norm(Y))


def max_rel_to_max(Y: np.ndarray, Y_ref: np.ndarray) -> float:
    Y = np.asarray(Y, dtype=np.float64)
    Y_ref = np.asarray(Y_ref, dtype=np.float64)
    den = np.max(np.abs(Y_ref))
    err = np.max(np.abs(Y - Y_ref))
    return float(err / den) if den > 0 else float(err)
