"""The fused attention kernel's polynomial 2^x (ex2_poly2 in
chunked_next_token_ttt_b300/csrc/attention_fused.cu), replayed step by step in
float32 NumPy with the constants read from the source, against 2^x in float64.

The kernel computes half of its probabilities P = 2^(S c - m) this way instead
of on the MUFU unit; P is then rounded to bf16 (relative spacing 2^-8), so the
polynomial's error must stay well below that.  Pins: the relative error over
the range P can take (x in [-126, TAU]), exact powers of two at integers, and a
result of at most 2^-125 for -inf (a masked score)."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "chunked_next_token_ttt_b300", "csrc", "attention_fused.cu")


def _poly_source():
    s = open(SRC).read()
    body = s[s.index("void ex2_poly2"):]
    body = body[:body.index("\n}\n")]
    return body


def _coefficients():
    body = _poly_source()
    cs = [float(c) for c in re.findall(r"f2make\(([0-9.]+)f, \1f\)", body)]
    assert len(cs) == 5 and cs[0] == 12582912.0     # the rounding constant, then c3, c2, c1, c0
    return np.float32(cs[0]), [np.float32(c) for c in cs[1:]]


def _ex2_poly(x):
    """The kernel's steps in float32: clamp, round by the 1.5 * 2^23 constant,
    cubic in Horner form, exponent-field add."""
    rnd, (c3, c2, c1, c0) = _coefficients()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-126.0))
    j = (x + rnd).astype(np.float32)
    f = (x - (j - rnd).astype(np.float32)).astype(np.float32)
    # fma rounds once: a float64 product of two float32 values is exact
    p = (np.float64(c3) * f + c2).astype(np.float32)
    p = (p.astype(np.float64) * f + c1).astype(np.float32)
    p = (p.astype(np.float64) * f + c0).astype(np.float32)
    bits = (p.view(np.int32).astype(np.int64) + (j.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_relative_error_over_the_range_of_p():
    x = np.concatenate([np.linspace(-126.0, 8.5, 400001), np.linspace(-1.0, 1.0, 100001)]).astype(np.float32)
    got = _ex2_poly(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    normal = want >= 2.0 ** -125
    rel = np.abs(got[normal] / want[normal] - 1.0)
    assert rel.max() < 1e-4, rel.max()          # bf16 spacing is 2^-8 = 3.9e-3
    assert np.all(got[~normal] >= 0) and np.all(got[~normal] <= 2.0 ** -124)


def test_integers_and_masked_scores():
    n = np.arange(-120, 9, dtype=np.float32)
    got = _ex2_poly(n).astype(np.float64)
    np.testing.assert_allclose(got, np.exp2(n.astype(np.float64)), rtol=1e-4)
    assert _ex2_poly(np.float32(-np.inf)) <= 2.0 ** -125
    assert _ex2_poly(np.float32(-1e30)) <= 2.0 ** -125
    assert np.all(np.diff(_ex2_poly(np.linspace(-3, 3, 10001).astype(np.float32))) >= 0)   # monotone
