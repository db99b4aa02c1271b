"""Pins for the oracle's quantize / double-quant / dequantize steps:
special cases whose result the method fixes, a round-trip error bound derived
from the level spacing and the 8-bit scale step, brute force on tiny inputs,
and the memory-size invariant the pages quote."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import nf4_oracle as o


def _w(n, seed=0, std=0.02):
    return (np.random.default_rng(seed).standard_normal(n) * std).astype(np.float32)


def test_pack_layout_even_element_high_nibble():
    codes = np.array([1, 2, 3, 4, 15, 0], dtype=np.uint8)
    assert list(o.pack_nibbles(codes)) == [0x12, 0x34, 0xF0]
    assert list(o.unpack_nibbles(o.pack_nibbles(codes))) == list(codes)


def test_zero_block_and_zero_group():
    w = np.zeros(64 * 300, dtype=np.float32)
    w[64 * 5 + 3] = 0.5          # one nonzero in block 5 (group 0)
    packed, a8, s2 = o.quantize_flat(w)
    codes = o.unpack_nibbles(packed)
    assert codes[64 * 5 + 3] == 15
    assert np.all(np.delete(codes, 64 * 5 + 3) == 7)
    assert a8[5] == 255 and np.all(np.delete(a8, 5) == 0)
    assert s2[0] == np.float32(0.5) and s2[1] == 0.0       # group 1 all zero
    what = o.dequantize_flat(packed, a8, s2)
    assert what[64 * 5 + 3] == np.float32(0.5)
    assert np.all(np.delete(what, 64 * 5 + 3) == 0)


def test_extremes_map_to_end_levels():
    w = _w(64)
    w[10] = 0.1
    w[20] = -0.1
    w = np.clip(w, -0.1, 0.1)
    codes = o.unpack_nibbles(o.quantize_flat(w)[0])
    assert codes[10] == 15 and codes[20] == 0
    # negated weight maps code i -> mirrored codes only where the table is
    # symmetric; at the ends it must swap 0 <-> 15
    codes_neg = o.unpack_nibbles(o.quantize_flat(-w)[0])
    assert codes_neg[10] == 0 and codes_neg[20] == 15


def test_negative_zero_is_code_seven():
    w = np.zeros(64, dtype=np.float32)
    w[0] = 1.0
    w[1] = -0.0
    codes = o.unpack_nibbles(o.quantize_flat(w)[0])
    assert codes[1] == 7


def test_double_quant_attaining_block_is_255_and_range():
    absmax = np.abs(_w(1000, 3)) + 1e-3
    a8, s2 = o.double_quant(absmax.astype(np.float32))
    assert s2.size == 4
    for g in range(4):
        seg = absmax[g * 256:(g + 1) * 256]
        assert s2[g] == np.float32(seg.max())
        assert a8[g * 256 + int(np.argmax(seg))] == 255
    # brute force: nearest integer to the exact ratio, up to the fp32 roundings
    for i in range(0, 1000, 37):
        exact = Fraction(255) * Fraction(float(absmax[i])) / Fraction(float(s2[i // 256]))
        assert abs(Fraction(int(a8[i])) - exact) <= Fraction(1, 2) + Fraction(1, 1 << 15)


def test_partial_last_group():
    w = _w(64 * 300, 5)
    packed, a8, s2 = o.quantize_flat(w)
    assert packed.size == 64 * 300 // 2 and a8.size == 300 and s2.size == 2
    absmax = np.abs(w.reshape(-1, 64)).max(axis=1)
    assert s2[1] == absmax[256:].max()


def test_group_aligned_slice_gives_same_outputs():
    w = _w(16384 * 3 + 64 * 10, 6)
    packed, a8, s2 = o.quantize_flat(w)
    p2, a2, s22 = o.quantize_flat(w[16384:32768])
    assert np.array_equal(p2, packed[8192:16384])
    assert np.array_equal(a2, a8[256:512]) and s22[0] == s2[1]


def test_round_trip_error_bound():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal(16384 * 4) * 0.02).astype(np.float32)
    w[rng.random(w.size) < 0.001] = (rng.standard_normal(1) * 0.5).astype(np.float32)
    packed, a8, s2 = o.quantize_flat(w)
    what = o.dequantize_flat(packed, a8, s2).astype(np.float64)
    a = np.abs(w.reshape(-1, 64)).max(axis=1).astype(np.float64)
    s = s2[np.arange(a.size) // 256].astype(np.float64)
    ahat = o.dequant_absmax(a8, s2).astype(np.float64)
    # scale error: half an 8-bit step of s2 plus the fp32 roundings
    assert np.all(np.abs(a - ahat) <= s / 510 + s * 2.0 ** -21)
    # weight error: largest half-gap of the levels, the scale error, roundings
    bound = 0.1519036 * a + 2.0 ** -22 * a + s * (1 / 510 + 2.0 ** -21) + 2.0 ** -22 * np.maximum(a, ahat)
    err = np.abs(w.astype(np.float64) - what).reshape(-1, 64)
    assert np.all(err <= bound[:, None])
    # and the bound is not vacuous: typical error is far smaller
    assert err.mean() < 0.05 * a.mean()


def test_dequant_matches_exact_rational_on_tiny_input():
    w = _w(128, 12, std=1.0)
    packed, a8, s2 = o.quantize_flat(w)
    codes = o.unpack_nibbles(packed)
    c = [Fraction(float(v)) for v in o.nf4_levels()]
    what = o.dequantize_flat(packed, a8, s2)
    for i in range(128):
        b = i // 64
        ahat = np.float32(np.float32(np.float32(a8[b]) * s2[0]) / np.float32(255))
        exact = c[codes[i]] * Fraction(float(ahat))
        # fl32 of the exact product: within half an ulp
        ulp = np.spacing(np.float32(abs(float(exact)))) if exact != 0 else 0
        assert abs(Fraction(float(what[i])) - exact) <= Fraction(float(ulp)) / 2


def test_memory_size_invariant_matches_quoted_savings():
    rows, cols = 4096, 4096
    nb = rows * cols // 64
    ng = (nb + 255) // 256
    packed, a8, s2 = o.quantize(np.zeros((64, 4096), np.float32))  # shapes only
    assert packed.nbytes == 64 * 4096 // 2 and a8.nbytes == 64 * 4096 // 64
    total = rows * cols // 2 + nb + 4 * ng
    bits = 8 * total / (rows * cols)
    assert abs(bits - 4.127) < 1e-3
    saving_fp32 = 1 - bits / 32
    assert 0.75 <= saving_fp32 <= 0.89            # "~75-89% vs fp32"
    dq_extra = 1 - bits / 4.5                     # vs fp32 absmax per block
    assert 0.05 <= dq_extra <= 0.10               # "further 5-10%"


@pytest.mark.parametrize("dtype", ["nf4", "fp4", "int8"])
def test_oracle_views_match_full_dequant(dtype):
    from tests.oracle_views import OracleWeight
    W = (np.random.default_rng(21).standard_normal((24, 704)) * 0.02).astype(np.float32)
    if dtype == "int8":
        full = o.int8_dequantize_flat(*o.int8_quantize_flat(W.reshape(-1))).reshape(24, 704)
    else:
        lv = o.levels_of(dtype)
        full = o.dequantize(*o.quantize(W, lv), 24, 704, lv)
    ow = OracleWeight(W, dtype)
    assert np.array_equal(ow.rows([0, 5, 23]), full[[0, 5, 23]])
    cols = OracleWeight.columns_of([0, 3, 10])
    assert np.array_equal(ow.col_blocks([0, 3, 10]), full[:, cols])
