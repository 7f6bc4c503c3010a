"""The bulk append kernel's fast rule for Q4G32 and Q8G32 codes, modelled in numpy float32 (every
operation IEEE round-to-nearest, as on the GPU), against the codec's definition on groups chosen to
stress it: random, clamped (offset far above the spread), zero beyond fp16, subnormal fp16 scales,
constant, quarter-integer (tie-heavy) and many-decade groups.

The rule: q = RN(RN(y - z) * inv) (Q8: RN(y * inv)) with inv the hardware reciprocal of the scale,
which is within 1 ulp of 1/s: the model takes each of RN(1/s) and its two neighbours.  rint by
(q + 1.5 * 2^23) - 1.5 * 2^23; the code is the low nibble (byte) of the rint sum's bits.  The group is
redone with the IEEE quotient when a quotient lies within 2^-17 (Q8: 2^-14) of a half-integer, is NaN,
or when the codes of the group's extremes leave [0, 15] ([-127, 127]): the fast quotient is monotone
in y, so the extremes bound every code.  The claim checked: every code equals the definition's."""

import numpy as np
import pytest

F = np.float32
MAGIC = F(12582912.0)
LIM4 = F(0.5) - F(2.0 ** -17)
LIM8 = F(0.5) - F(2.0 ** -14)


def _groups(n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    kinds = np.arange(n) % 8
    x = rng.standard_normal((n, 32))
    x[kinds == 1] = 1000.0 + 0.01 * rng.standard_normal(((kinds == 1).sum(), 32))
    x[kinds == 2] = -1.0e5 + rng.standard_normal(((kinds == 2).sum(), 32))
    x[kinds == 3] = rng.integers(-8, 8, ((kinds == 3).sum(), 32)) * 0.5
    x[kinds == 4] *= 1e-6
    x[kinds == 5] = rng.standard_normal(((kinds == 5).sum(), 1))
    x[kinds == 6] *= np.exp(rng.uniform(-20, 20, ((kinds == 6).sum(), 1)))
    x[kinds == 7] = np.round(rng.standard_normal(((kinds == 7).sum(), 32)) * 8) / 4
    return x.astype(F)


def _neighbours(v: np.ndarray):
    return (np.nextafter(v, F(-np.inf)), v, np.nextafter(v, F(np.inf)))


def _rint_parts(q: np.ndarray):
    t = (q + MAGIC).astype(F)
    d = (q + (MAGIC - t).astype(F)).astype(F)           # q - rint(q), exact
    return t, d


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_q4_fast_rule_equals_definition():
    x = _groups(48000, 3)
    mn, mx = x.min(1, keepdims=True), x.max(1, keepdims=True)
    s = ((mx - mn).astype(F) / F(15)).astype(F).astype(np.float16).astype(F)
    z = mn.astype(np.float16).astype(F)
    want = np.clip(np.rint((((x - z).astype(F)) / s).astype(F)), 0, 15)
    want = np.where(s > 0, want, 0).astype(np.int64)
    n = (x - z).astype(F)
    for inv in _neighbours((F(1) / s).astype(F)):
        q = (n * inv).astype(F)
        t, d = _rint_parts(q)
        dmax = np.where(np.isnan(d).any(1, keepdims=True), np.nan, np.abs(d).max(1, keepdims=True))
        fast = (t.view(np.uint32) & 15).astype(np.int64)
        qlo = (((mn - z).astype(F)) * inv).astype(F)
        qhi = (((mx - z).astype(F)) * inv).astype(F)
        redo = ~(dmax <= LIM4) | ~(qlo >= -0.5) | ~(qhi < 15.5)
        got = np.where(s > 0, np.where(redo, want, fast), 0)
        assert np.array_equal(got, want)
        # the rule is not vacuous: the redo path is taken, and the fast codes alone are wrong somewhere
        assert redo.any() and not np.array_equal(np.where(s > 0, fast, 0), want)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_q8_fast_rule_equals_definition():
    x = _groups(48000, 4)
    amax = np.abs(x).max(1, keepdims=True)
    d = (amax / F(127)).astype(F).astype(np.float16).astype(F)
    want = np.clip(np.rint((x / d).astype(F)), -127, 127)
    want = np.where(d > 0, want, 0).astype(np.int64) + 128
    for inv in _neighbours((F(1) / d).astype(F)):
        q = (x * inv).astype(F)
        t, dd = _rint_parts(q)
        dmax = np.where(np.isnan(dd).any(1, keepdims=True), np.nan, np.abs(dd).max(1, keepdims=True))
        fast = ((t.view(np.uint32) & 0xFF) ^ 0x80).astype(np.int64)
        qmax = (amax * inv).astype(F)
        redo = ~(dmax <= LIM8) | ~(qmax < 127.5)
        got = np.where(d > 0, np.where(redo, want, fast), 128)
        assert np.array_equal(got, want)
        assert redo.any()
