"""Property tests of the oracle codec on arbitrary inputs within the documented value range.

Vectors are finite with Euclidean norm below the fp16 range (the library's stated precondition);
elements may be tiny, subnormal, zero or repeated.  Runs on the CPU only.
"""

import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402
from hypothesis.extra import numpy as hnp  # noqa: E402

from oracle import codec  # noqa: E402

SETTINGS = settings(max_examples=150, deadline=None, derandomize=True)

_elem = st.one_of(
    st.floats(-4000.0, 4000.0, allow_nan=False, allow_infinity=False, width=32),
    st.floats(-2.0 ** -100, 2.0 ** -100, allow_nan=False, allow_infinity=False, width=32),
    st.sampled_from([0.0, -0.0, 1.0, -1.0, 0.5]),
)
vectors = hnp.arrays(np.float32, (128,), elements=_elem)


def _in_range(y):
    return float(np.sqrt(np.sum(y.astype(np.float64) ** 2))) < 60000.0


@SETTINGS
@given(vectors)
def test_q4_codes_in_range_and_error_bounded(y):
    if not _in_range(y):
        return
    c, s, z = codec.q4g32_encode(y)
    assert c.dtype == np.uint8 and int(c.max()) <= 15
    assert np.all(np.isfinite(s.astype(np.float32))) and np.all(np.isfinite(z.astype(np.float32)))
    sg = np.repeat(s.astype(np.float64), 32)
    zg = np.repeat(z.astype(np.float64), 32)
    err = np.abs(codec.q4g32_decode(c, s, z).astype(np.float64) - y)
    # half a step, the fp16 rounding of zero and scale, and the float32 roundings of the decode
    bound = 0.5 * sg + 2.0 ** -10 * (np.abs(zg) + 15 * sg) + 2.0 ** -22 * np.abs(y) + 1e-36
    gmax = np.repeat(np.abs(y.reshape(4, 32)).max(1).astype(np.float64), 32)
    bound = bound + 2.0 ** -23 * gmax
    assert np.all(err <= bound * (1 + 1e-6) + 6e-8 * (gmax < 6.2e-5))


@SETTINGS
@given(vectors)
def test_q8_codes_in_range_and_error_bounded(y):
    if not _in_range(y):
        return
    c, d = codec.q8g32_encode(y)
    assert c.dtype == np.int8 and int(np.abs(c.astype(np.int32)).max()) <= 127
    dg = np.repeat(d.astype(np.float64), 32)
    gmax = np.repeat(np.abs(y.reshape(4, 32)).max(1).astype(np.float64), 32)
    err = np.abs(codec.q8g32_decode(c, d).astype(np.float64) - y)
    # fp16 d may round down (clipping the largest value) or flush a tiny group to zero
    assert np.all(err <= 0.5 * dg + 2.0 ** -10 * gmax + 6e-8 * (gmax < 7.8e-3))


@SETTINGS
@given(vectors)
def test_rotation_round_trip(y):
    if not _in_range(y):
        return
    s = codec.wht_signs(11)
    back = codec.unrotate(codec.rotate(y, s), s).astype(np.float64)
    scale = float(np.max(np.abs(y))) if np.any(y) else 0.0
    assert np.all(np.abs(back - y) <= 2.0 ** -19 * scale + 1e-40)


def _squares_underflow(y):
    """Nonzero, but every float32 square rounds to zero (all |y_j| <= 2^-75)."""
    return bool(np.any(y != 0)) and bool(np.all(y * y == 0))


@SETTINGS
@given(vectors)
def test_tq3_fields(y):
    if not _in_range(y) or _squares_underflow(y):
        return
    proj = np.random.default_rng(0).standard_normal((128, 128)).astype(np.float32)
    code, bits, n, gamma = codec.tq3_qjl_encode(y[None], proj)
    assert int(code.max()) <= 7 and bits.dtype == bool
    assert float(n[0]) >= 0 and np.isfinite(float(n[0]))
    g = float(gamma[0])
    # the residual of a unit vector against its nearest centroids: |r| <= |u| + |c| <= 1 + 0.2 * sqrt(128)
    assert np.isfinite(g) and 0.0 <= g <= 1.0 + 0.2 * np.sqrt(128)


def test_tq3_key_below_the_norm_guard():
    """The documented degenerate case of the 1/max(|y|, FLT_MIN) normalisation: a nonzero key whose
    squares all underflow has n = 0 and is scaled by 1/FLT_MIN, so its residual norm overflows fp16
    (gamma = inf) and 0 * inf makes its logits NaN.  Keys must be zero or have some |y_j| > 2^-75."""
    proj = np.random.default_rng(0).standard_normal((128, 128)).astype(np.float32)
    y = np.full((1, 128), 2.0 ** -80, np.float32)
    assert _squares_underflow(y[0])
    with np.errstate(over="ignore"):
        code, bits, n, gamma = codec.tq3_qjl_encode(y, proj)
    assert float(n[0]) == 0 and np.isinf(float(gamma[0]))
    y[0, 0] = 2.0 ** -74                                 # one square survives: a normal key again
    code, bits, n, gamma = codec.tq3_qjl_encode(y, proj)
    assert np.isfinite(float(gamma[0])) and float(gamma[0]) < 3.0


def test_sinkhorn_scale_outside_fp16():
    """sigma is stored as fp16: channel scales spread by 10^4 are recovered in ratio, while a channel
    10^8 below the others rounds to sigma = 0 (the calibration precondition in the header)."""
    x = np.random.default_rng(0).standard_normal((256, 128)).astype(np.float32)
    y = x.copy()
    y[:, 5] *= np.float32(1e4)
    s = codec.sinkhorn_sigma(y).astype(np.float64)
    others = np.delete(s, 5)
    assert 0.8e4 < s[5] / np.median(others) < 1.25e4
    y = x.copy()
    y[:, 5] *= np.float32(1e-8)
    with np.errstate(all="ignore"):
        s = codec.sinkhorn_sigma(y)
    assert float(s[5]) == 0.0 and np.all(np.delete(s, 5) > 0)


@settings(max_examples=40, deadline=None, derandomize=True)
@given(st.integers(0, 2), st.integers(1, 40), st.sampled_from([0, 4, 8]), st.integers(0, 2 ** 31 - 1))
def test_decode_output_is_a_convex_combination_of_values(kind, L, window, seed):
    """Softmax weights are non-negative and sum to 1, and the inverse rotation is linear, so every
    output coordinate lies between the smallest and largest value any attended token contributes
    (dequantised and un-rotated, or raw in the window)."""
    from oracle import attention

    kfmt = (attention.Q4G32, attention.Q8G32, attention.TQ3_QJL)[kind]
    rng = np.random.default_rng(seed)
    proj = rng.standard_normal((128, 128)).astype(np.float32) if kfmt == attention.TQ3_QJL else None
    cfg = attention.OracleConfig(n_layers=1, n_kv_heads=1, n_q_heads=2, max_batch=1, max_seq_len=48,
                                 window=window, k_format=kfmt, seed=seed % 7)
    c = attention.OracleCache(cfg, proj)
    k = (rng.standard_normal((1, 1, L, 128)) * rng.uniform(0.1, 5)).astype(np.float32)
    v = (rng.standard_normal((1, 1, L, 128)) * rng.uniform(0.1, 5)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = (rng.standard_normal((1, 2, 128)) * rng.uniform(0.1, 3)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))[0]
    Lq = max(0, L - window) if window > 0 else L
    vals = []
    if Lq:
        vd = codec.q4g32_decode(c.v["code"][0, 0, 0, :Lq], c.v["scale"][0, 0, 0, :Lq],
                                c.v["zero"][0, 0, 0, :Lq]).astype(np.float64)
        vals.append(codec.unrotate64(vd, c.signs))
    if L > Lq:
        vals.append(v[0, 0, Lq:L].astype(np.float64))
    vals = np.concatenate(vals)
    lo, hi = vals.min(0), vals.max(0)
    tol = 1e-9 * np.abs(vals).max()
    assert np.all(out >= lo - tol) and np.all(out <= hi + tol)
