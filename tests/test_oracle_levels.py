"""Pins for the oracle's NF4 levels and nearest-level search.

The pages give no printed NF4 values; the levels are pinned by what defines
them (standard-normal quantiles at evenly spaced probabilities, normalised to
[-1, 1]) through routines the oracle does not use, and by the table's
invariants. The nearest-level search is pinned by exact rational brute force
and by an independent midpoint-counting formulation.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.special as sps

from oracle import nf4_oracle as o

DELTA = 0.5 * ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0))


def test_levels_match_second_inverse_cdf_routine():
    # scipy's ndtri is an independent implementation of Phi^-1
    pos = sps.ndtri(np.linspace(DELTA, 0.5, 9)[:-1])
    neg = -sps.ndtri(np.linspace(DELTA, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, neg, [0.0]])) / sps.ndtri(DELTA)
    assert np.array_equal(v.astype(np.float32).view(np.uint32), o.nf4_levels().view(np.uint32))


def test_levels_invert_through_forward_cdf():
    # Phi(c * Phi^-1(delta)) must land back on the evenly spaced probabilities
    lv = o.nf4_levels_fp64()
    top = sps.ndtri(DELTA)
    p = sps.ndtr(lv * top)
    assert np.allclose(p[8:], np.linspace(DELTA, 0.5, 9)[:-1][::-1], atol=1e-12, rtol=0)
    assert np.allclose(1.0 - p[:7], np.linspace(DELTA, 0.5, 8)[:-1], atol=1e-12, rtol=0)


def test_level_invariants():
    c = o.nf4_levels()
    assert c.dtype == np.float32 and c.size == 16
    assert np.all(np.diff(c) > 0)
    assert c[0] == -1.0 and c[15] == 1.0
    assert c[7] == 0.0 and not np.signbit(c[7])
    assert (c < 0).sum() == 7 and (c > 0).sum() == 8
    # more resolution near zero than at the extremes (non-uniform spacing)
    gaps = np.diff(c.astype(np.float64))
    assert gaps[7] < gaps[0] and gaps[8] < gaps[14]
    # largest half-gap (between the two lowest levels) bounds the rounding error
    assert abs(gaps.max() / 2 - 0.1519036) < 1e-6 and np.argmax(gaps) == 0


def _brute_nearest(x):
    c = [Fraction(float(v)) for v in o.nf4_levels()]
    fx = Fraction(float(x))
    d = [abs(fx - ci) for ci in c]
    return min(range(16), key=lambda i: (d[i], i))


def _near_midpoints(ulps):
    c = o.nf4_levels().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2          # exact in fp64
    out = []
    for m in mids:
        b = np.float32(m).view(np.int32).astype(np.int64)
        out.append(np.arange(b - ulps, b + ulps + 1, dtype=np.int64))
    v = np.concatenate(out)
    return v.astype(np.int32).view(np.float32), mids


def test_nearest_code_exact_rational_bruteforce():
    rng = np.random.default_rng(7)
    xs = list(rng.uniform(-1, 1, 400).astype(np.float32))
    near, _ = _near_midpoints(3)
    xs += list(near)
    xs += [np.float32(v) for v in (0.0, -0.0, 1.0, -1.0, 1e-30, -1e-30, 2.0 ** -40, 1e-45)]
    got = o.nearest_code(np.array(xs, dtype=np.float32))
    want = [_brute_nearest(x) for x in xs]
    assert list(got) == want


def test_nearest_code_equals_strict_midpoint_count():
    near, mids = _near_midpoints(1 << 13)
    rng = np.random.default_rng(11)
    rnd = rng.uniform(-1, 1, 1 << 18).astype(np.float32)
    tiny = (rng.uniform(-1, 1, 4096) * 2.0 ** -30).astype(np.float32)
    x = np.concatenate([near, rnd, tiny])
    x = x[(x >= -1) & (x <= 1)]
    # ties go to the lower index, so a value equal to a midpoint is not above it
    count = (x.astype(np.float64)[:, None] > mids[None, :]).sum(axis=1)
    assert np.array_equal(o.nearest_code(x), count.astype(np.uint8))


def test_representable_midpoints_tie_to_lower():
    c = o.nf4_levels().astype(np.float64)
    mids = (c[:-1] + c[1:]) / 2
    exact = [i for i, m in enumerate(mids) if float(np.float32(m)) == m]
    assert exact, "expected at least one fp32-representable midpoint"
    for i in exact:
        assert o.nearest_code(np.array([mids[i]], dtype=np.float32))[0] == i


def test_levels_match_stored_table():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "nf4_levels.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    bits = np.array([int(r[1], 16) for r in rows], dtype=np.uint32)
    assert np.array_equal(bits, o.nf4_levels().view(np.uint32))
