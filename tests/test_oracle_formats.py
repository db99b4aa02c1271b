"""Pins for the oracle's other weight formats: FP4 (E2M1) levels and codes
("bitsandbytes" page, 4-bit paragraph: NF4 or FP4), uniform int8 per-block
quantization ("Zenbit" page, zenbit.int8 bullet), and the bf16 decoding of
bf16 weights. Each is checked against exact arithmetic or a library routine,
and each plausible alternative reading is planted in a copy and shown to fail.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nf4_oracle as o
from tests.exact_fp32 import f32, rne32, rne_int

# E2M1 magnitudes written out from the format: exponent 0 holds 0 and the
# subnormal 0.5; exponents 1..3 hold 1, 1.5, 2, 3, 4, 6.
E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
        Fraction(4), Fraction(6)]
FP4 = [f32(v) for v in o.fp4_levels()]


def test_fp4_levels_are_e2m1_over_six():
    lv = o.fp4_levels()
    for code in range(16):
        mag = E2M1[code & 7]
        want = rne32((-mag if code & 8 else mag) / 6)
        assert FP4[code] == want, code
    assert lv[7] == 1.0 and lv[15] == -1.0
    assert lv[0] == 0.0 and not np.signbit(lv[0]) and lv[8] == 0.0 and np.signbit(lv[8])
    assert np.all(np.diff(lv[:8]) > 0) and np.array_equal(lv[8:], -lv[:8])
    assert o.zero_code(lv) == 0 and o.zero_code(o.nf4_levels()) == 7


def exact_nearest(x: Fraction, levels) -> int:
    best, best_d = 0, abs(x - levels[0])
    for i in range(1, len(levels)):
        d = abs(x - levels[i])
        if d < best_d:
            best, best_d = i, d
    return best


def fp4_edge_values(rng, n=3000):
    """fp32 values in [-1, 1] within a few ulps of the decision midpoints
    between neighbouring magnitudes, on both signs, plus random values."""
    mags = [Fraction(float(v)) for v in o.fp4_levels()[:8]]
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(7)]
    xs = []
    for _ in range(n):
        m = float(mids[rng.integers(0, 7)])
        v = np.float32(m)
        v = (v.view(np.int32) + np.int32(rng.integers(-3, 4))).view(np.float32)
        xs.append(-v if rng.random() < 0.5 else v)
    xs += list(rng.uniform(-1, 1, n).astype(np.float32))
    xs += [np.float32(0.0), np.float32(-0.0), np.float32(-1e-30), np.float32(1e-30)]
    return np.array(xs, dtype=np.float32)


def test_fp4_nearest_code_is_exact_argmin_with_ties_to_the_lower_code():
    rng = np.random.default_rng(4)
    xs = fp4_edge_values(rng)
    got = o.nearest_code(xs, o.fp4_levels())
    for x, g in zip(xs, got):
        assert g == exact_nearest(f32(x), FP4), x
    # the midpoint between 0 and 1/12 is an fp32 value: +-mid is a tie that
    # goes to code 0 (+0) on both signs, never to -0 (8) or -1/12 (9)
    mid = np.float32(float((FP4[0] + FP4[1]) / 2))
    assert Fraction(float(mid)) == (FP4[0] + FP4[1]) / 2
    assert list(o.nearest_code(np.array([mid, -mid, -0.0], np.float32), o.fp4_levels())) == [0, 0, 0]


def test_fp4_pin_rejects_sign_magnitude_rounding_away_from_zero_on_ties():
    """A plausible slip: rounding |x| to the nearest magnitude with ties to
    the larger one and then applying the sign. The fp32 midpoint between 0
    and 1/12 is a tie that the planted rule sends to 1/12 (code 1, or 9 when
    negative) and the pinned rule to code 0."""
    mags = o.fp4_levels()[:8].astype(np.float64)

    def planted(xs):
        d = np.abs(np.abs(xs.astype(np.float64))[:, None] - mags[None, :])
        mag = (7 - np.argmin(d[:, ::-1], axis=1)).astype(np.uint8)    # ties to the larger
        return np.where(mag == 0, 0, mag | np.where(xs < 0, 8, 0)).astype(np.uint8)

    mid = np.float32(float((FP4[0] + FP4[1]) / 2))
    xs = np.array([mid, -mid], dtype=np.float32)
    want = [exact_nearest(f32(x), FP4) for x in xs]
    assert want == [0, 0]
    assert list(o.nearest_code(xs, o.fp4_levels())) == want
    assert list(planted(xs)) == [1, 9]


def test_fp4_quantize_special_cases_and_round_trip_bound():
    lv = o.fp4_levels()
    rng = np.random.default_rng(6)
    w = (rng.standard_normal(64 * 512) * 0.02).astype(np.float32)
    w[:64] = 0.0
    w[64:128] = 0.0
    w[64 + 5] = -2.5                       # single nonzero: code of -1
    w[128] = 0.7
    w[129] = -0.7                          # +-absmax: codes 7 and 15
    w[130] = -0.0
    packed, a8, s2 = o.quantize_flat(w, lv)
    codes = o.unpack_nibbles(packed)
    assert np.all(codes[:64] == 0) and codes[64 + 5] == 15
    assert np.all(np.delete(codes[64:128], 5) == 0)
    assert codes[128] == 7 and codes[129] == 15 and codes[130] == 0
    what = o.dequantize_flat(packed, a8, s2, lv).astype(np.float64)
    a = np.abs(w.reshape(-1, 64)).max(axis=1).astype(np.float64)
    s = s2[np.arange(a.size) // 256].astype(np.float64)
    half_gap = float(np.max(np.diff(lv[:8].astype(np.float64)))) / 2     # 1/6
    assert abs(half_gap - 1 / 6) < 1e-7
    bound = (half_gap * a + 2.0 ** -22 * a + s * (1 / 510 + 2.0 ** -21)
             + 2.0 ** -22 * np.maximum(a, s))
    err = np.abs(w.astype(np.float64) - what).reshape(-1, 64)
    assert np.all(err <= bound[:, None])
    # and the codes of every block are the exact nearest levels of w / a
    blocks = w.reshape(-1, 64)
    for b in range(0, 512, 37):
        ab = max(abs(f32(v)) for v in blocks[b])
        for j in range(64):
            want = o.zero_code(lv) if ab == 0 else exact_nearest(rne32(f32(blocks[b, j]) / ab), FP4)
            assert codes[64 * b + j] == want


def test_fp4_dequant_uses_the_fp4_table():
    lv = o.fp4_levels()
    codes = np.arange(64, dtype=np.uint8) % 16
    ahat = np.array([np.float32(3.0)], dtype=np.float32)
    what = o.dequantize_codes(codes.reshape(1, 64), ahat, lv).reshape(-1)
    for j in range(64):
        assert Fraction(float(what[j])) == rne32(FP4[j % 16] * 3)


# ------------------------------------------------------------------ int8 --
def exact_q(w, a):
    if a == 0:
        return 0
    return rne_int(rne32(rne32(127 * f32(w)) / f32(a)))


def test_int8_codes_are_the_exact_multiply_then_divide_chain():
    rng = np.random.default_rng(7)
    nb = 200
    a = np.concatenate([rng.uniform(1e-3, 2.0, nb - 40), 10.0 ** rng.uniform(-36, -30, 20),
                        10.0 ** rng.uniform(20, 34, 20)]).astype(np.float32)
    W = (rng.uniform(-1, 1, (nb, 64)) * a[:, None]).astype(np.float32)
    W[:, 0] = a * np.where(rng.random(nb) < 0.5, 1, -1)
    # values near the half-way points k + 1/2 of 127 w / a
    k = rng.integers(-127, 127, (nb, 20))
    W[:, 1:21] = ((k + 0.5) * a[:, None].astype(np.float64) / 127).astype(np.float32)
    q, absmax = o.int8_quantize_flat(W.reshape(-1))
    assert np.array_equal(absmax, np.abs(W).max(axis=1))
    for b in range(nb):
        for j in range(64):
            assert q[64 * b + j] == exact_q(W[b, j], absmax[b]), (b, j)
    assert q.min() >= -127 and q.max() <= 127
    assert np.all(np.abs(q.reshape(nb, 64)[:, 0]) == 127)


def test_int8_rounds_exact_halves_to_even_and_rejects_other_readings():
    """absmax 127 and w = k + 1/2: 127 w = 127 k + 63.5 exactly and the
    quotient by 127 is k + 1/2, so q is the even neighbour."""
    ks = np.arange(-63, 63)
    w = np.zeros((2, 64), dtype=np.float32)
    w[:, 0] = 127.0                                   # each block's absmax is 127
    w[:, 1:] = (ks + 0.5).reshape(2, 63)
    q, a = o.int8_quantize_flat(w.reshape(-1))
    assert np.all(a == 127.0)
    got = q.reshape(2, 64)[:, 1:].reshape(-1)
    for i, kk in enumerate(ks):
        want = kk if kk % 2 == 0 else kk + 1
        assert got[i] == want, kk
    half_up = np.floor((np.float32(127) * (ks + 0.5).astype(np.float32)) / np.float32(127) + 0.5)
    assert np.count_nonzero(half_up != got) > 30
    # divide first: fl32(127 fl32(w / a)) lands on other codes near the halves
    rng = np.random.default_rng(9)
    n = 200000
    aa = rng.uniform(0.01, 3.0, n).astype(np.float32)
    kk = rng.integers(-127, 127, n)
    ww = ((kk + 0.5) * aa.astype(np.float64) / 127).astype(np.float32)
    ww = (ww.view(np.int32) + rng.integers(-3, 4, n).astype(np.int32)).view(np.float32)
    ok = np.abs(ww) <= aa
    mul = np.rint((np.float32(127) * ww) / aa)
    div = np.rint(np.float32(127) * (ww / aa))
    idx = np.flatnonzero(ok & (mul != div))[:30]
    assert idx.size == 30
    blocks = np.zeros((30, 64), dtype=np.float32)
    blocks[:, 0] = aa[idx]
    blocks[:, 1] = ww[idx]
    q2, _ = o.int8_quantize_flat(blocks.reshape(-1))
    for j, i in enumerate(idx):
        assert q2[64 * j + 1] == exact_q(ww[i], aa[i]) and q2[64 * j + 1] != div[i]


def test_int8_dequant_and_round_trip_bound():
    rng = np.random.default_rng(10)
    w = (rng.standard_normal(64 * 300) * 0.02).astype(np.float32)
    w[64:128] = 0.0
    q, a = o.int8_quantize_flat(w)
    assert np.all(q[64:128] == 0) and a[1] == 0
    what = o.int8_dequantize_flat(q, a)
    for i in range(0, w.size, 97):
        want = rne32(rne32(int(q[i]) * f32(a[i // 64])) / 127)
        assert Fraction(float(what[i])) == want
    err = np.abs(w.astype(np.float64) - what).reshape(-1, 64)
    ad = a.astype(np.float64)
    assert np.all(err <= (ad / 254 + 2.0 ** -21 * ad)[:, None])
    # memory: one byte per weight and an fp32 scale per 64: 8.5 bits, about
    # half of fp16 ("~50% memory savings vs fp16")
    bits = 8 + 32 / 64
    assert 0.45 <= 1 - bits / 16 <= 0.5


# ------------------------------------------------------------------ bf16 --
def test_bf16_decode_matches_torch_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = o.bf16_to_fp32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
