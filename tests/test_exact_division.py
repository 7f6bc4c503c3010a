"""The bulk append kernel forms the group scales RN((max - min) / 15) and RN(max |y| / 127) without a
division: q0 = RN(a * c) with c = RN(1/D), the exact residual r = a - D * q0 (one fma), then
RN(q0 + r * c) (Markstein's correction step, IBM J. Res. Dev. 34(1), 1990).  Over the normal range
the result depends on a's 24-bit mantissa only (scaling a by 2^k scales every step), so an exact
integer model over all 2^23 mantissas proves the three steps give the correctly rounded quotient for
every normal a.  The model is checked to have teeth: the uncorrected q0 alone is wrong on some."""

import numpy as np
import pytest


def _rn_shift(v: np.ndarray, sh: np.ndarray) -> np.ndarray:
    """Round-half-even of v / 2^sh for v >= 0, sh >= 1."""
    q = v >> sh
    rem = v - (q << sh)
    half = np.int64(1) << (sh - 1)
    return q + ((rem > half) | ((rem == half) & ((q & 1) == 1)))


def _bitlen(v: np.ndarray) -> np.ndarray:
    b = np.floor(np.log2(v.astype(np.float64))).astype(np.int64) + 1
    b = np.where((v >> (b - 1)) == 0, b - 1, b)     # the float log2 may be one off near 2^k
    return np.where((v >> b) != 0, b + 1, b)


def _norm24(m: np.ndarray, e: np.ndarray):
    big = m >= (1 << 24)
    return np.where(big, m >> 1, m), np.where(big, e + 1, e)


@pytest.mark.parametrize("D", [15, 127])
def test_constant_division_is_correctly_rounded(D):
    k = int(np.floor(np.log2(D)))
    C = round((1 << (24 + k)) / D)                   # c = RN(1/D) = C * 2^ce, C a 24-bit mantissa
    ce = -(24 + k)
    assert (1 << 23) <= C < (1 << 24)
    assert np.float32(1.0 / D) == np.float32(C * 2.0 ** ce)
    A = np.arange(1 << 23, 1 << 24, dtype=np.int64)  # a = A * 2^ea, every mantissa
    P = A * C                                        # a * c exactly, 47 or 48 bits
    sh = np.where(P >= (1 << 47), 48, 47) - 24
    Q0 = _rn_shift(P, sh)                            # q0 = Q0 * 2^(ea + ce + sh)
    t = -(ce + sh)
    assert np.all(t >= 0)
    R = A * (np.int64(1) << t) - D * Q0              # r = R * 2^(ea + ce + sh), exact
    assert np.all(np.abs(R) < (1 << 24))
    N = Q0 * (np.int64(1) << (-ce)) + R * C          # q0 + r c = N * 2^(ea + ce + sh + ce)
    assert np.all((N > 0) & (N < (1 << 62)))
    bN = _bitlen(N)
    M1, E1 = _norm24(_rn_shift(N, bN - 24), 2 * ce + sh + bN - 24)
    # exact RN(a / D) from A * 2^36 / D: integer part X, remainder Rm (D odd: never a tie unless exact)
    X = (A << 36) // D
    Rm = (A << 36) - X * D
    bX = _bitlen(X)
    shX = bX - 24
    q = X >> shX
    rem = X - (q << shX)
    half = np.int64(1) << (shX - 1)
    up = (rem > half) | ((rem == half) & ((Rm > 0) | ((q & 1) == 1)))
    ME, EE = _norm24(q + up, shX - 36)
    assert np.array_equal(M1, ME) and np.array_equal(E1, EE)
    M0, E0 = _norm24(Q0, ce + sh)
    assert not (np.array_equal(M0, ME) and np.array_equal(E0, EE))   # the correction step matters
