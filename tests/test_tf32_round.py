"""The TF32 rounding helper the plain-TF32 parity tests use, against its definition
(nearest multiple of 2^(e-10) for a value in [2^e, 2^(e+1)), ties away from zero),
evaluated in exact rational arithmetic."""
import math
from fractions import Fraction

import numpy as np

from tests.parity import tf32_round


def _tf32_exact(v: float) -> float:
    if v == 0.0:
        return v
    m, e = math.frexp(v)              # v = m * 2^e, 0.5 <= |m| < 1
    quantum = Fraction(2) ** (e - 11)  # 11 significant bits
    q = Fraction(v) / quantum
    r = math.floor(abs(q) + Fraction(1, 2))
    return float(math.copysign(1, v) * r * quantum)


def test_tf32_round_matches_definition():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                           (rng.standard_normal(2000) * 1e-30).astype(np.float32),
                           (rng.standard_normal(2000) * 1e30).astype(np.float32)])
    # exact ties (a 1 in the first dropped bit only) and values just below / above them
    base = np.array([1.0, -1.0, 3.0, 0.75], np.float32).view(np.uint32)
    ties = (base[:, None] + np.array([0x1000, 0x0FFF, 0x1001, 0x3000], np.uint32)).ravel().view(np.float32)
    vals = np.concatenate([vals, ties, np.float32([0.0, -0.0, 2.0 ** -126, 1.9999999])])
    got = tf32_round(vals)
    want = np.array([_tf32_exact(float(v)) for v in vals], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_tf32_round_examples():
    one_tie = np.float32(1.0 + 2.0 ** -11)        # halfway between 1 and 1 + 2^-10
    assert tf32_round(np.float32([one_tie]))[0] == np.float32(1.0 + 2.0 ** -10)
    assert tf32_round(np.float32([-one_tie]))[0] == np.float32(-(1.0 + 2.0 ** -10))
    assert tf32_round(np.float32([1.0 + 2.0 ** -12]))[0] == np.float32(1.0)
