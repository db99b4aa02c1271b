"""Exact-arithmetic pins for the oracle's fp32 decisions.

Each test recomputes one step from its definition with exact rationals and an
independent binary32 rounding (tests/exact_fp32.py), on inputs built so that
the plausible alternative readings of the step give different results, and
then checks that those alternatives (planted here, in a copy of the step, on
the CPU) really fail the pin:

* the normalisation x = fl32(w / absmax) of the "bitsandbytes" page's NF4
  paragraph ("map weights to quantization levels" after per-block scaling)
  with the block's true absmax, against a reciprocal multiply w * fl32(1/a)
  and against normalising by the double-quantized absmax;
* the double quantization a8 = rint(fl32(fl32(255 a) / s2)) of the same page's
  double-quantization paragraph, against round-half-up and against the
  divide-first order fl32(255 fl32(a / s2));
* the dequantization ahat = fl32(fl32(a8 s2) / 255) ("scaling factors are
  dequantized first"), against fl32(a8 fl32(s2 / 255));
* the weight dequantization w = fl32(c[q] ahat).
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import nf4_oracle as o
from tests.exact_fp32 import as_f32, f32, rne32, rne_int

LEVELS = [f32(v) for v in o.nf4_levels()]


def exact_nearest(x: Fraction, levels=LEVELS) -> int:
    """argmin_i |x - c_i| over exact rationals, the first index on a tie."""
    best, best_d = 0, abs(x - levels[0])
    for i in range(1, len(levels)):
        d = abs(x - levels[i])
        if d < best_d:
            best, best_d = i, d
    return best


# ------------------------------------------------------------ the helper --
def test_rne32_matches_float32_conversion_of_doubles():
    """np.float32(double) is one IEEE rounding of an exact value: the helper
    must agree with it everywhere, subnormals and ties included."""
    rng = np.random.default_rng(0)
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-45, 38, 2000))
    vals += [2.0 ** -149, 2.0 ** -150, 3 * 2.0 ** -151, 2.0 ** -126 * (1 - 2.0 ** -30),
             1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, -(1 + 2.0 ** -24), 0.1, 1 / 3]
    for v in vals:
        if abs(v) > 3.4e38:
            continue
        assert rne32(Fraction(v)) == Fraction(float(np.float32(v))), v
    assert rne_int(Fraction(5, 2)) == 2 and rne_int(Fraction(7, 2)) == 4
    assert rne_int(Fraction(-5, 2)) == -2 and rne_int(Fraction(11, 4)) == 3


# ---------------------------------------------------------- the quotient --
def edge_blocks(seed=17, nblocks=96):
    """Blocks whose first element is +-a (so the block absmax is a) and whose
    other elements sit within 3 ulps of m * a for a decision midpoint m of
    the table; a spans ordinary, tiny, subnormal-adjacent and huge scales."""
    rng = np.random.default_rng(seed)
    c = o.nf4_levels().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2
    k = nblocks // 4
    absmax = np.concatenate([
        rng.uniform(1e-3, 1.0, nblocks - 3 * k), 10.0 ** rng.uniform(-38, -30, k),
        10.0 ** rng.uniform(-44, -39, k // 2), 10.0 ** rng.uniform(20, 35, k - k // 2),
        rng.uniform(0.5, 2.0, k)]).astype(np.float32)[:nblocks]
    W = np.empty((nblocks, 64), dtype=np.float32)
    W[:, 0] = absmax * np.where(rng.random(nblocks) < 0.5, 1, -1).astype(np.float32)
    for j in range(1, 64):
        m = mids[rng.integers(0, 15, nblocks)] * np.where(rng.random(nblocks) < 0.5, 1, -1)
        base = np.abs(m * absmax.astype(np.float64)).astype(np.float32)
        step = rng.integers(-3, 4, nblocks).astype(np.int32)
        mag = np.maximum(base.view(np.int32) + step, 0).view(np.float32)
        W[:, j] = np.where(m < 0, -mag, mag)
    W = np.where(np.abs(W) > np.abs(W[:, :1]), W[:, :1], W).astype(np.float32)
    return W


def expected_codes(W):
    out = np.empty(W.shape, dtype=np.uint8)
    for b in range(W.shape[0]):
        a = max(abs(f32(v)) for v in W[b])
        for j in range(W.shape[1]):
            out[b, j] = 7 if a == 0 else exact_nearest(rne32(f32(W[b, j]) / a))
    return out.reshape(-1)


@pytest.fixture(scope="module")
def quotient_case():
    W = edge_blocks()
    return W, expected_codes(W)


def test_quantize_codes_are_the_nearest_level_of_the_ieee_quotient(quotient_case):
    W, want = quotient_case
    got = o.unpack_nibbles(o.quantize_flat(W.reshape(-1))[0])
    assert np.array_equal(got, want)


def _codes_by(W, normalise):
    """Codes of a planted variant of the normalisation (same nearest step)."""
    blocks = W.reshape(-1, 64)
    a = np.max(np.abs(blocks), axis=1).astype(np.float32)
    x = normalise(blocks, a)
    return o.nearest_code(x).reshape(-1)


def test_pin_rejects_a_reciprocal_multiply(quotient_case):
    W, want = quotient_case
    # only blocks whose reciprocal is finite, so that a mismatch is a rounding
    # difference and not an overflow
    ok = np.repeat(np.abs(W[:, 0]) >= np.float32(1e-37), 64)
    with np.errstate(over="ignore", invalid="ignore"):
        recip = _codes_by(W, lambda b, a: (b * (np.float32(1) / a)[:, None]).astype(np.float32))
    assert np.count_nonzero((recip != want) & ok) > 0


def test_pin_rejects_normalising_by_the_dequantized_absmax(quotient_case):
    W, want = quotient_case

    def by_ahat(b, a):
        a8, s2 = o.double_quant(a)
        ahat = o.dequant_absmax(a8, s2)
        return np.clip(b / np.where(ahat > 0, ahat, 1)[:, None], -1, 1).astype(np.float32)
    assert np.count_nonzero(_codes_by(W, by_ahat) != want) > 0


# -------------------------------------------------------- double quant --
def test_double_quant_rounds_exact_halves_to_even():
    """s2 = 255 and absmax = k + 1/2: fl32(255 a) = 255 k + 127.5 exactly and
    the quotient by 255 is exactly k + 1/2, so the code is the even one of k,
    k + 1. Round-half-up would give k + 1 for every k."""
    ks = np.arange(255)
    absmax = np.concatenate([[255.0], ks + 0.5]).astype(np.float32)
    a8, s2 = o.double_quant(absmax)
    assert s2.size == 1 and s2[0] == 255.0 and a8[0] == 255
    for k in range(255):
        want = k if k % 2 == 0 else k + 1
        assert a8[1 + k] == want, k
    half_up = np.floor(np.float32(255) * absmax[1:256] / np.float32(255) + 0.5)
    assert np.count_nonzero(half_up != a8[1:256]) > 100


def exact_a8(a, s2):
    if s2 == 0:
        return 0
    return rne_int(rne32(rne32(255 * f32(a)) / f32(s2)))


def test_double_quant_is_multiply_then_divide_exactly():
    """Random groups plus absmax values chosen where the two orders of the
    fp32 operations land on different codes: the oracle matches the exact
    multiply-first chain on all of them."""
    rng = np.random.default_rng(3)
    # candidates within a few ulps of a half-way quotient k + 1/2
    n = 200000
    s = rng.uniform(0.01, 3.0, n).astype(np.float32)
    k = rng.integers(0, 255, n)
    a = ((k + 0.5) * s.astype(np.float64) / 255).astype(np.float32)
    a = (a.view(np.int32) + rng.integers(-4, 5, n).astype(np.int32)).view(np.float32)
    keep = (a > 0) & (a <= s)
    mul_first = np.rint((np.float32(255) * a) / s)
    div_first = np.rint(np.float32(255) * (a / s))
    idx = np.flatnonzero(keep & (mul_first != div_first))[:40]
    assert idx.size == 40
    found = list(zip(a[idx], s[idx]))
    absmax = np.zeros(256 * len(found), dtype=np.float32)
    for g, (a, s) in enumerate(found):
        absmax[256 * g] = s
        absmax[256 * g + 1] = a
        absmax[256 * g + 2:256 * (g + 1)] = rng.uniform(0, 1, 254).astype(np.float32) * s
    a8, s2 = o.double_quant(absmax)
    for i in range(absmax.size):
        assert a8[i] == exact_a8(absmax[i], s2[i // 256]), i
    div_first = [np.rint(np.float32(255) * (a / s)) for a, s in found]
    assert all(a8[256 * g + 1] != d for g, d in enumerate(div_first))


# ------------------------------------------------------------ dequant --
def test_dequant_absmax_is_product_then_quotient_exactly():
    rng = np.random.default_rng(8)
    s2 = rng.uniform(1e-4, 10.0, 64).astype(np.float32)
    s2[:4] = [np.float32(1e-30), np.float32(3e30), np.float32(2.0 ** -120), np.float32(1.0)]
    a8 = np.tile(np.arange(256, dtype=np.uint8), 64)
    ahat = o.dequant_absmax(a8, s2)
    alt = []
    for i in range(a8.size):
        s = s2[i // 256]
        want = rne32(rne32(int(a8[i]) * f32(s)) / 255)
        assert Fraction(float(ahat[i])) == want, i
        alt.append(rne32(int(a8[i]) * rne32(f32(s) / 255)) != want)
    assert sum(alt) > 100      # the other order is a different function


def test_dequantize_codes_is_one_rounded_product():
    rng = np.random.default_rng(11)
    ahat = rng.uniform(1e-3, 2.0, 40).astype(np.float32)
    ahat[:3] = [np.float32(1e-38), np.float32(2.0 ** -130), np.float32(1e30)]
    codes = rng.integers(0, 16, (40, 64)).astype(np.uint8)
    what = o.dequantize_codes(codes, ahat)
    for b in range(40):
        for j in range(64):
            want = rne32(LEVELS[codes[b, j]] * f32(ahat[b]))
            assert Fraction(float(what[b, j])) == want
    assert as_f32(want) == what[39, 63]
