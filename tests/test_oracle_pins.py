"""Pins of the CPU oracle against facts that the pages and mathematics fix (no GPU needed).

Each test checks the oracle against something other than itself: a textbook construction or
table, a library routine, a closed form, an invariant, or brute force on small inputs.
"""

import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg

from oracle import attention, codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ------------------------------------------------------------------ rotation
def test_splitmix64_published_outputs():
    want = [int(x, 16) for x in _golden_rows("splitmix64_seed0.txt")]
    assert codec.splitmix64(0, 3) == want


def test_signs_are_pm1_and_balanced():
    s = codec.wht_signs(0)
    assert s.dtype == np.float32 and set(np.unique(s)) <= {-1.0, 1.0}
    assert 40 < (s > 0).sum() < 88          # a fair coin over 128 draws
    assert not np.array_equal(s, codec.wht_signs(1))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_butterfly_is_sylvester_hadamard(dtype):
    """Butterfly applied to the unit vectors reproduces scipy's Sylvester H_128 exactly."""
    H = codec.hadamard_butterfly(np.eye(128, dtype=dtype))   # row j = H e_j = column j of H
    ref = scipy.linalg.hadamard(128).astype(dtype)
    assert np.array_equal(H.T, ref)
    assert np.array_equal(H @ H.T, 128 * np.eye(128, dtype=dtype))


def test_rotation_of_unit_vector_is_signed_hadamard_column():
    s = codec.wht_signs(0)
    ref = scipy.linalg.hadamard(128).astype(np.float32)
    for j in (0, 5, 77, 127):
        e = np.zeros(128, np.float32)
        e[j] = 1.0
        y = codec.rotate(e, s)
        assert np.array_equal(y, (ref[:, j] * s[j]) * codec.C_WHT)


def test_rotation_constant_bits():
    assert np.float32(codec.C_WHT).view(np.uint32) == 0x3DB504F3


def test_rotation_orthogonal_and_invertible():
    rng = np.random.default_rng(1)
    s = codec.wht_signs(3)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    y = codec.rotate(x, s)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x.astype(np.float64), axis=1), rtol=1e-6)
    xr = codec.unrotate(y, s)
    assert np.max(np.abs(xr - x)) <= 2.0 ** -20 * np.max(np.abs(x)) * 8
    # float64 version agrees with the float32 one to float32 rounding
    assert np.allclose(codec.rotate64(x, s), y, rtol=0, atol=1e-5)


def test_sumsq128_tree():
    rng = np.random.default_rng(2)
    # small integers: every partial sum is exact, so the tree equals the exact sum
    v = rng.integers(-50, 50, (16, 128)).astype(np.float32)
    assert np.array_equal(codec.sumsq128(v), (v.astype(np.int64) ** 2).sum(1).astype(np.float32))
    x = rng.standard_normal((16, 128)).astype(np.float32)
    exact = (x.astype(np.float64) ** 2).sum(1)
    assert np.allclose(codec.sumsq128(x), exact, rtol=8 * 2.0 ** -24 * 8)
    # a dropped or doubled block would be caught here
    e = np.zeros(128, np.float32)
    e[127] = 3.0
    assert codec.sumsq128(e) == 9.0


def test_sumsq128_tree_shape():
    """The documented tree pairs (v0^2 + v1^2) + (v2^2 + v3^2) within a block and block i with block
    i + 16, then i + 8, ...  Two squares of 2^-24 next to a 1 reach the exact (representable) sum
    1 + 2^-23 only when the tree adds them to each other before adding them to the 1; a
    left-to-right block sum or an adjacent-block pairing rounds each to even and returns 1."""
    exact = np.float32(1 + 2.0 ** -23)
    v = np.zeros(128, np.float32)
    v[0], v[2], v[3] = 1.0, 2.0 ** -12, 2.0 ** -12          # same block, second pair
    assert codec.sumsq128(v) == exact
    v = np.zeros(128, np.float32)
    v[0], v[4 * 1], v[4 * 17] = 1.0, 2.0 ** -12, 2.0 ** -12  # blocks 1 and 17 are siblings
    assert codec.sumsq128(v) == exact


def test_sumsq128_invariant_under_tree_symmetries():
    """IEEE addition commutes, so swapping the operands of any node of the tree leaves the result
    bit-identical: swaps within a pair, of the two pairs of a block, and block index b -> b xor m."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-8, 8, (64, 128)))).astype(np.float32)
    ref = codec.sumsq128(x)
    blk = x.reshape(64, 32, 4)
    assert np.array_equal(codec.sumsq128(blk[:, :, [1, 0, 2, 3]].reshape(64, 128)), ref)
    assert np.array_equal(codec.sumsq128(blk[:, :, [2, 3, 0, 1]].reshape(64, 128)), ref)
    for m in (1, 2, 4, 8, 16, 31):
        perm = np.arange(32) ^ m
        assert np.array_equal(codec.sumsq128(blk[:, perm].reshape(64, 128)), ref)


# ------------------------------------------------------------------ Q4G32
def test_q4_on_grid_round_trip_is_lossless():
    """Inputs already on a grid z + s*c (fp16 z, power-of-two s, codes using 0 and 15)."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        z = np.float16(rng.uniform(-4, 4)).astype(np.float32)
        s = np.float32(2.0 ** rng.integers(-6, 0))
        codes = rng.integers(0, 16, (4, 32))
        codes[:, 0] = 0
        codes[:, 1] = 15
        y = (z + s * codes.astype(np.float32)).astype(np.float32).reshape(128)
        c, sc, zc = codec.q4g32_encode(y)
        assert np.array_equal(c, codes.reshape(128).astype(np.uint8))
        assert np.all(sc.astype(np.float32) == s) and np.all(zc.astype(np.float32) == z)
        assert np.array_equal(codec.q4g32_decode(c, sc, zc), y)


def test_q4_constant_group():
    y = np.full(128, 0.3, np.float32)
    c, s, z = codec.q4g32_encode(y)
    assert np.all(c == 0) and np.all(s == 0)
    assert np.all(codec.q4g32_decode(c, s, z) == np.float16(0.3).astype(np.float32))


def test_q4_codes_are_nearest_grid_points():
    """Brute force: each code minimises |y - (z + s*c)| over c in 0..15 (ties excluded)."""
    rng = np.random.default_rng(4)
    y = (rng.standard_normal((200, 128)) * rng.uniform(0.1, 10, (200, 1))).astype(np.float32)
    c, s, z = codec.q4g32_encode(y)
    sg = np.repeat(s.astype(np.float64), 32, axis=-1)
    zg = np.repeat(z.astype(np.float64), 32, axis=-1)
    grid = zg[..., None] + sg[..., None] * np.arange(16)
    dist = np.abs(y.astype(np.float64)[..., None] - grid)
    best = dist.argmin(-1)
    tie = np.sort(dist, -1)[..., 1] - np.sort(dist, -1)[..., 0] < 1e-6 * sg
    assert np.array_equal(c[~tie], best[~tie])
    # error bound: half a step plus the fp16 rounding of the zero and the scale
    err = np.abs(codec.q4g32_decode(c, s, z) - y)
    assert np.all(err <= 0.5 * sg + 2.0 ** -10 * (np.abs(zg) + 15 * sg) + 1e-6)


def test_q4_scale_and_zero_formula_brute_force():
    rng = np.random.default_rng(5)
    y = rng.standard_normal(128).astype(np.float32)
    c, s, z = codec.q4g32_encode(y)
    for gi in range(4):
        g = y[32 * gi:32 * gi + 32]
        assert z[gi] == np.float16(float(g.min()))
        want = np.float16(np.float32(np.float32(g.max()) - np.float32(g.min())) / np.float32(15))
        assert s[gi] == want


def test_q4_ties_round_to_even():
    """A group spanning exactly [0, 15] has scale 1 and zero 0, so (y - zero) / scale = y is exact and
    values halfway between codes take the even code (IEEE round-half-even)."""
    y = np.full(128, 7.0, np.float32)
    y[:9] = [0, 15, 0.5, 1.5, 2.5, 3.5, 4.5, 13.5, 14.5]
    c, s, z = codec.q4g32_encode(y)
    assert s[0] == 1 and z[0] == 0
    assert list(c[:9]) == [0, 15, 0, 2, 2, 4, 4, 14, 14]


# ------------------------------------------------------------------ Q8G32 (8-bit keys)
def test_q8_on_grid_round_trip_is_lossless():
    """Inputs d * c with a power-of-two d and integer c in [-127, 127], one |c| = 127 per group."""
    rng = np.random.default_rng(30)
    for _ in range(20):
        d = np.float32(2.0 ** rng.integers(-12, 2))
        codes = rng.integers(-127, 128, (4, 32))
        codes[:, 0] = 127 * rng.choice([-1, 1], 4)
        y = (d * codes.astype(np.float32)).reshape(128)
        c, dc = codec.q8g32_encode(y)
        assert np.array_equal(c, codes.reshape(128).astype(np.int8))
        assert np.all(dc.astype(np.float32) == d)
        assert np.array_equal(codec.q8g32_decode(c, dc), y)


def test_q8_codes_are_nearest_grid_points():
    """Brute force over the 255 levels d * c; error at most half a step plus the fp16 rounding of d
    (which can push max |y| / d just past 127, where the code clips)."""
    rng = np.random.default_rng(31)
    y = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    c, d = codec.q8g32_encode(y)
    dg = np.repeat(d.astype(np.float64), 32, axis=-1)
    grid = dg[..., None] * np.arange(-127, 128)
    dist = np.abs(y.astype(np.float64)[..., None] - grid)
    best = dist.argmin(-1) - 127
    sd = np.sort(dist, -1)
    tie = sd[..., 1] - sd[..., 0] < 1e-6 * dg
    assert np.array_equal(c[~tie].astype(np.int64), best[~tie])
    amax = np.repeat(np.abs(y.reshape(200, 4, 32)).max(-1).astype(np.float64), 32, axis=-1)
    err = np.abs(codec.q8g32_decode(c, d).astype(np.float64) - y)
    assert np.all(err <= 0.5 * dg + 2.0 ** -11 * amax * 1.01)


def test_q8_zero_group_sign_symmetry_and_ties():
    z = np.zeros(128, np.float32)
    c, d = codec.q8g32_encode(z)
    assert np.all(c == 0) and np.all(d == 0)
    rng = np.random.default_rng(32)
    y = rng.standard_normal((50, 128)).astype(np.float32)
    c1, d1 = codec.q8g32_encode(y)
    c2, d2 = codec.q8g32_encode(-y)
    assert np.array_equal(c2, -c1) and np.array_equal(d2, d1)
    # a group with max |y| = 127 has d = 1: halves go to the even code (IEEE round-half-even)
    y = np.zeros(128, np.float32)
    y[:8] = [127, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5]
    c, d = codec.q8g32_encode(y)
    assert d[0] == 1 and list(c[:8]) == [127, 0, 2, 2, 0, -2, -2, 126]


def test_q8_key_record_is_8_5_bits():
    """An 8-bit block format of 32 values with one fp16 scale stores 34 bytes per 32 values."""
    assert attention.REC_BYTES[attention.Q8G32] * 8 / 128 == 8.5
    cfg = attention.OracleConfig(1, 1, 1, 1, 1, k_format=attention.Q8G32)
    assert attention.payload_bytes_per_token_head(cfg) == 136 + 80


def test_q8_keys_score_far_closer_than_q4_keys():
    """[TQ] "rules": K at Q8 is the safe setting.  On outlier-bearing keys the Q8 logit error is at
    least ten times below the Q4 one (step 2 max|y| / 254 against (max - min) / 15)."""
    rng = np.random.default_rng(33)
    k = rng.standard_normal((1000, 128)).astype(np.float32)
    k[:, :3] *= 8
    s = codec.wht_signs(0)
    y = codec.rotate(k, s)
    q = rng.standard_normal(128)
    true = y.astype(np.float64) @ q
    e8 = np.abs(codec.q8g32_decode(*codec.q8g32_encode(y)).astype(np.float64) @ q - true).mean()
    e4 = np.abs(codec.q4g32_decode(*codec.q4g32_encode(y)).astype(np.float64) @ q - true).mean()
    assert e8 * 10 < e4


# ------------------------------------------------------------------ Lloyd-Max / TQ3
def test_lloyd_max_matches_textbook_table():
    rows = _golden_rows("lloyd_max_gaussian_8.txt")
    levels = np.array([float(x) for x in rows[0].split()])
    thresholds = np.array([float(x) for x in rows[1].split()])
    c, b = codec.lloyd_max_gaussian(8)
    assert np.allclose(c[4:], levels, atol=1.5e-4)
    assert np.allclose(c[:4], -levels[::-1], atol=1.5e-4)
    assert np.allclose(b[3:], thresholds, atol=1.5e-4)


def test_lloyd_max_fixed_point_conditions_by_quadrature():
    """Centroid condition checked with numerical integration, independent of the closed form."""
    c, b = codec.lloyd_max_gaussian(8)
    edges = np.concatenate(([-np.inf], b, [np.inf]))
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)
    for k in range(8):
        m0 = scipy.integrate.quad(pdf, edges[k], edges[k + 1], epsabs=1e-14)[0]
        m1 = scipy.integrate.quad(lambda x: x * pdf(x), edges[k], edges[k + 1], epsabs=1e-14)[0]
        assert abs(m1 / m0 - c[k]) < 1e-9
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), atol=1e-15)
    assert np.allclose(c, -c[::-1], atol=1e-12)


def test_tq3_codebook_is_fp16_scaled_lloyd_max():
    cent, bnd = codec.tq3_codebook()
    c64, _ = codec.lloyd_max_gaussian(8)
    assert cent.dtype == np.float16
    assert np.allclose(cent.astype(np.float64), c64 / math.sqrt(128), rtol=2.0 ** -11)
    assert np.all(np.diff(cent.astype(np.float32)) > 0)
    assert np.all((bnd > cent[:-1].astype(np.float32)) & (bnd < cent[1:].astype(np.float32)))


def test_tq3_codes_are_nearest_centroid_and_norms():
    rng = np.random.default_rng(6)
    proj = rng.standard_normal((128, 128)).astype(np.float32)
    y = rng.standard_normal((100, 128)).astype(np.float32) * 3
    code, bits, n, gamma = codec.tq3_qjl_encode(y, proj)
    cent, _ = codec.tq3_codebook()
    c32 = cent.astype(np.float32)
    nrm = np.linalg.norm(y.astype(np.float64), axis=1)
    assert np.allclose(n.astype(np.float64), nrm, rtol=2.0 ** -10)
    u = y.astype(np.float64) / nrm[:, None]
    d = np.abs(u[..., None] - c32.astype(np.float64))
    best = d.argmin(-1)
    sd = np.sort(d, -1)
    clear = sd[..., 1] - sd[..., 0] > 1e-6
    assert np.array_equal(code[clear], best[clear])
    r = u - c32[code]
    assert np.allclose(gamma.astype(np.float64), np.linalg.norm(r, axis=1), rtol=2.0 ** -10, atol=1e-6)
    t = r @ proj.T.astype(np.float64)
    far = np.abs(t) > 1e-5
    assert np.array_equal(bits[far], t[far] >= 0)


def test_tq3_codes_are_scale_invariant():
    """u = y / |y| does not depend on the scale of y: a power-of-two scale (exact in float32) leaves
    codes and signs unchanged and scales n exactly, down to norms far below any small epsilon."""
    rng = np.random.default_rng(22)
    proj = rng.standard_normal((128, 128)).astype(np.float32)
    y = rng.standard_normal((50, 128)).astype(np.float32)
    c0, b0, n0, g0 = codec.tq3_qjl_encode(y, proj)
    for e in (-30, -12, 10):
        c, b, n, g = codec.tq3_qjl_encode(y * np.float32(2.0 ** e), proj)
        assert np.array_equal(c, c0) and np.array_equal(b, b0) and np.array_equal(g, g0)
        if e == 10:
            assert np.array_equal(n.astype(np.float32), n0.astype(np.float32) * np.float32(2.0 ** e))


def test_tq3_zero_vector():
    """y = 0: n = 0 and u = 0 (the guard max(n, eps) keeps the division finite); 0 is the middle
    boundary of the symmetric codebook and a coordinate on a boundary takes the upper cell, so every
    code is 4, the residual is -c4 in every coordinate and gamma = sqrt(128) * c4."""
    rng = np.random.default_rng(23)
    proj = rng.standard_normal((128, 128)).astype(np.float32)
    c, b, n, g = codec.tq3_qjl_encode(np.zeros((1, 128), np.float32), proj)
    cent, bnd = codec.tq3_codebook()
    assert bnd[3] == 0 and n[0] == 0
    assert np.all(c == 4)
    assert g[0] == np.float16(math.sqrt(128) * float(cent[4]))
    assert np.array_equal(b[0], proj.astype(np.float64).sum(1) * -float(cent[4]) >= 0)


def test_qjl_estimator_is_unbiased():
    """E_S[sqrt(pi/2)/m * |r| * <S q, sign(S r)>] = <q, r> for Gaussian S (QJL)."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128)
    r = rng.standard_normal(128) * 0.1
    est = []
    for _ in range(2000):
        S = rng.standard_normal((128, 128))
        est.append(codec.QJL_CONST * np.linalg.norm(r) * (S @ q) @ np.sign(S @ r))
    est = np.array(est)
    se = est.std() / math.sqrt(len(est))
    assert abs(est.mean() - q @ r) < 3.5 * se


def test_tq3_estimate_tracks_true_inner_product():
    rng = np.random.default_rng(8)
    proj = rng.standard_normal((128, 128)).astype(np.float32)
    y = rng.standard_normal((400, 128)).astype(np.float32)
    q = rng.standard_normal(128)
    code, bits, n, gamma = codec.tq3_qjl_encode(y, proj)
    est = codec.tq3_qjl_dot64(q, code, bits, n, gamma, proj)
    true = y.astype(np.float64) @ q
    assert np.corrcoef(est, true)[0, 1] > 0.97
    assert abs(np.mean(est - true)) < 4 * np.std(est - true) / math.sqrt(len(true))
    # unbiased means the estimate is on the scale of <q, y>: least-squares slope 1
    slope = np.dot(est, true) / np.dot(true, true)
    assert abs(slope - 1) < 0.05


# ------------------------------------------------------------------ Sinkhorn invariants
def test_sinkhorn_recovers_planted_column_scales():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((1024, 128))
    a /= np.sqrt((a ** 2).mean(0))               # unit column RMS
    cscale = np.exp(rng.uniform(np.log(0.2), np.log(5), 128))
    x = (a * cscale).astype(np.float32)
    sig = codec.sinkhorn_sigma(x).astype(np.float64)
    ratio = sig / cscale
    assert np.std(ratio) / np.mean(ratio) < 0.03


def test_sinkhorn_recovers_column_scales_under_planted_row_scales():
    """X = diag(r) A diag(c) with balanced A: alternating row and column normalisation (Sinkhorn)
    removes the row factors, so sigma is proportional to c even when r spans four decades; column
    normalisation alone would weight each column by a few dominant rows."""
    rng = np.random.default_rng(24)
    a = rng.standard_normal((1024, 128))
    a /= np.sqrt((a ** 2).mean(0))
    r = np.exp(rng.uniform(np.log(0.01), np.log(100), (1024, 1)))
    cscale = np.exp(rng.uniform(np.log(0.2), np.log(5), 128))
    sig = codec.sinkhorn_sigma((r * a * cscale).astype(np.float32)).astype(np.float64)
    ratio = sig / cscale
    assert np.std(ratio) / np.mean(ratio) < 0.03


def test_sinkhorn_zero_rows_and_zero_block():
    """Degenerate blocks: an all-zero token contributes nothing and keeps sigma finite; an all-zero
    block has no scale to balance and gives sigma = 1."""
    rng = np.random.default_rng(25)
    a = rng.standard_normal((1024, 128))
    a /= np.sqrt((a ** 2).mean(0))
    cscale = np.exp(rng.uniform(np.log(0.2), np.log(5), 128))
    x = (a * cscale).astype(np.float32)
    x[::7] = 0
    sig = codec.sinkhorn_sigma(x).astype(np.float64)
    ratio = sig / cscale
    assert np.all(np.isfinite(sig)) and np.std(ratio) / np.mean(ratio) < 0.03
    assert np.all(codec.sinkhorn_sigma(np.zeros((64, 128), np.float32)) == 1)


def test_sinkhorn_balanced_input_gives_unit_sigma():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((1024, 128)).astype(np.float32)
    sig = codec.sinkhorn_sigma(x).astype(np.float64)
    assert np.all(np.abs(sig - 1) < 0.12)


def test_sinkhorn_balanced_block_has_unit_column_rms():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((512, 128)) * np.exp(rng.uniform(-2, 2, 128))).astype(np.float32)
    sig = codec.sinkhorn_sigma(x).astype(np.float64)
    bal = x / sig
    rows = np.sqrt((bal.astype(np.float64) ** 2).mean(1, keepdims=True))
    cols = np.sqrt(((bal / rows) ** 2).mean(0))
    assert np.all(np.abs(cols - 1) < 0.05)


# ------------------------------------------------------------------ attention
def _cache(window, T, B=1, H=1, Hq=2, kfmt=attention.Q4G32, seed=0, sink=False, proj=None):
    cfg = attention.OracleConfig(n_layers=1, n_kv_heads=H, n_q_heads=Hq, max_batch=B,
                                 max_seq_len=T, window=window, k_format=kfmt, sinkhorn=sink,
                                 seed=seed)
    return attention.OracleCache(cfg, proj)


@pytest.mark.parametrize("L", [1, 7, 100, 128])
def test_window_covering_context_is_plain_attention(L):
    rng = np.random.default_rng(12)
    c = _cache(128, 256)
    k = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    ref = attention.plain_attention64(q[0], k[0, 0], v[0, 0])
    assert np.allclose(out[0], ref, rtol=0, atol=1e-12)


def _brute_force_unit(cache, q, L, k_raw, v_raw):
    """Token-by-token loop with Python floats for sequence 0, kv-head 0 of layer 0.

    Quantised tokens are dequantised from the stored records (Q4G32: zero + scale * code, times
    sigma when balanced; TQ3+QJL: n * (<q~, c[code]> + sqrt(pi/2)/128 * gamma * <S q~, 2b - 1>)) and
    scored against the rotated query; window tokens are scored from the raw inputs ``k_raw``,
    ``v_raw`` [L][128], not from the ring, so that the ring's slot bookkeeping is checked too.
    """
    cfg = cache.cfg
    s = cache.signs.astype(np.float64)
    W = cfg.window
    Lq = max(0, L - W) if W > 0 else L
    sk = [float(x) for x in cache.sigma_k[0, 0]] if cfg.sinkhorn else [1.0] * 128
    sv = [float(x) for x in cache.sigma_v[0, 0]] if cfg.sinkhorn else [1.0] * 128
    cent = [float(x) for x in codec.tq3_codebook()[0]]
    outs = []
    for qh in q:
        qt = codec.hadamard_butterfly(qh.astype(np.float64) * s) * float(codec.C_WHT)
        ws, vals = [], []
        for t in range(L):
            if t < Lq:
                if cfg.k_format == attention.TQ3_QJL:
                    code = cache.k["code"][0, 0, 0, t]
                    bits = cache.k["bits"][0, 0, 0, t]
                    dot_c = sum(qt[j] * cent[code[j]] for j in range(128))
                    dot_s = 0.0
                    for i in range(128):
                        sq_i = sum(float(cache.proj[i, j]) * qt[j] for j in range(128))
                        dot_s += sq_i * (1.0 if bits[i] else -1.0)
                    est = float(cache.k["norm"][0, 0, 0, t]) * (
                        dot_c + math.sqrt(math.pi / 2) / 128 * float(cache.k["gamma"][0, 0, 0, t]) * dot_s)
                    lg = est / math.sqrt(128)
                elif cfg.k_format == attention.Q8G32:
                    code = cache.k["code"][0, 0, 0, t]
                    kv = [sk[j] * float(np.float32(cache.k["scale"][0, 0, 0, t, j // 32]) * np.float32(code[j]))
                          for j in range(128)]
                    lg = sum(qt[j] * kv[j] for j in range(128)) / math.sqrt(128)
                else:
                    code = cache.k["code"][0, 0, 0, t]
                    kv = [sk[j] * (float(cache.k["zero"][0, 0, 0, t, j // 32]) +
                                   float(np.float32(cache.k["scale"][0, 0, 0, t, j // 32]) * np.float32(code[j])))
                          for j in range(128)]
                    lg = sum(qt[j] * kv[j] for j in range(128)) / math.sqrt(128)
                vc = cache.v["code"][0, 0, 0, t]
                vr = np.array([sv[j] * (float(cache.v["zero"][0, 0, 0, t, j // 32]) +
                                        float(np.float32(cache.v["scale"][0, 0, 0, t, j // 32]) * np.float32(vc[j])))
                               for j in range(128)])
                vals.append(s * (codec.hadamard_butterfly(vr) * float(codec.C_WHT)))
            else:
                lg = sum(float(qh[j]) * float(k_raw[t, j]) for j in range(128)) / math.sqrt(128)
                vals.append(v_raw[t].astype(np.float64))
            ws.append(lg)
        m = max(ws)
        e = [math.exp(w - m) for w in ws]
        z = sum(e)
        outs.append(sum(ei / z * vi for ei, vi in zip(e, vals)))
    return np.array(outs)


@pytest.mark.parametrize("window,L", [(4, 9), (0, 6), (2, 2), (8, 3), (4, 13)])
def test_decode_matches_brute_force_on_tiny_inputs(window, L):
    rng = np.random.default_rng(13)
    c = _cache(window, 16, seed=5)
    k = (rng.standard_normal((1, 1, L, 128)) * 2).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    assert np.allclose(out[0], _brute_force_unit(c, q[0], L, k[0, 0], v[0, 0]), rtol=0, atol=1e-10)


@pytest.mark.parametrize("window,L", [(4, 9), (0, 5)])
def test_decode_tq_keys_matches_brute_force(window, L):
    rng = np.random.default_rng(17)
    proj = rng.standard_normal((128, 128)).astype(np.float32)
    c = _cache(window, 16, kfmt=attention.TQ3_QJL, seed=2, proj=proj)
    k = (rng.standard_normal((1, 1, L, 128)) * 2).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    assert np.allclose(out[0], _brute_force_unit(c, q[0], L, k[0, 0], v[0, 0]), rtol=0, atol=1e-10)


@pytest.mark.parametrize("window,L,sink", [(4, 9, False), (0, 5, False), (4, 10, True)])
def test_decode_q8_keys_matches_brute_force(window, L, sink):
    rng = np.random.default_rng(34)
    c = _cache(window, 16, kfmt=attention.Q8G32, seed=6, sink=sink)
    if sink:
        blk = (rng.standard_normal((1, 256, 128)) * np.exp(rng.uniform(-2, 2, 128))).astype(np.float32)
        c.calibrate(0, blk, blk * np.float32(0.5))
    k = (rng.standard_normal((1, 1, L, 128)) * 2).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    assert np.allclose(out[0], _brute_force_unit(c, q[0], L, k[0, 0], v[0, 0]), rtol=0, atol=1e-10)


def _planted_column_block(rng, n, cscale, signs):
    """Raw vectors whose ROTATED coordinates have column RMS ``cscale`` (unit-RMS Gaussian core)."""
    a = rng.standard_normal((n, 128))
    a /= np.sqrt((a ** 2).mean(0))
    return codec.unrotate((a * cscale).astype(np.float32), signs)


def test_decode_balanced_matches_brute_force():
    rng = np.random.default_rng(18)
    c = _cache(4, 16, sink=True, seed=1)
    ck = np.exp(rng.uniform(np.log(0.1), np.log(10), 128))
    cv = np.exp(rng.uniform(np.log(0.1), np.log(10), 128))
    c.calibrate(0, _planted_column_block(rng, 256, ck, c.signs)[None],
                _planted_column_block(rng, 256, cv, c.signs)[None])
    assert not np.all(c.sigma_k == 1) and not np.all(c.sigma_v == 1)
    L = 11
    k = _planted_column_block(rng, L, ck, c.signs)[None, None]
    v = _planted_column_block(rng, L, cv, c.signs)[None, None]
    c.append(0, k, v, np.array([0]))
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    assert np.allclose(out[0], _brute_force_unit(c, q[0], L, k[0, 0], v[0, 0]), rtol=0, atol=1e-10)


@pytest.mark.parametrize("kfmt", [attention.Q4G32, attention.Q8G32])
def test_balanced_records_reconstruct_the_rotated_input(kfmt):
    """[KV] TLDR: the balanced value y / sigma is what is quantised, so sigma * dequant(code) is y
    to within half a quantisation step of the balanced group (times sigma) plus fp16 rounding."""
    rng = np.random.default_rng(19)
    c = _cache(0, 64, sink=True, seed=4, kfmt=kfmt)
    ck = np.exp(rng.uniform(np.log(0.05), np.log(20), 128))
    cv = np.exp(rng.uniform(np.log(0.05), np.log(20), 128))
    c.calibrate(0, _planted_column_block(rng, 512, ck, c.signs)[None],
                _planted_column_block(rng, 512, cv, c.signs)[None])
    for sg16, cs in ((c.sigma_k, ck), (c.sigma_v, cv)):    # each from its own block
        ratio = sg16[0, 0].astype(np.float64) / cs
        assert np.std(ratio) / np.mean(ratio) < 0.03
    k = _planted_column_block(rng, 64, ck, c.signs)[None, None]
    v = _planted_column_block(rng, 64, cv, c.signs)[None, None]
    c.append(0, k, v, np.array([0]))
    for rec, sg16, x in ((c.k, c.sigma_k, k), (c.v, c.sigma_v, v)):
        sig = sg16[0, 0].astype(np.float64)
        y = codec.rotate(x[0, 0], c.signs).astype(np.float64)
        sg = np.repeat(rec["scale"][0, 0, 0].astype(np.float64), 32, axis=-1)
        if "zero" in rec:
            deq = codec.q4g32_decode(rec["code"][0, 0, 0], rec["scale"][0, 0, 0], rec["zero"][0, 0, 0])
            zg = np.repeat(rec["zero"][0, 0, 0].astype(np.float64), 32, axis=-1)
            step = 0.5 * sg + 2.0 ** -10 * (np.abs(zg) + 15 * sg)
        else:
            deq = codec.q8g32_decode(rec["code"][0, 0, 0], rec["scale"][0, 0, 0])
            step = 0.5 * sg + 2.0 ** -11 * 127 * sg * 1.01
        bound = sig * step + 2.0 ** -20 * np.abs(y) + 1e-6
        assert np.all(np.abs(sig * deq - y) <= bound)


def test_gqa_query_head_i_reads_kv_head_i_div_g():
    """Grouped-query attention (Llama convention): query head i attends with kv-head i // g; each
    sequence attends to its own first seq_lens[b] tokens."""
    rng = np.random.default_rng(20)
    B, H, Hq, T = 2, 2, 6, 60
    c = _cache(128, 64, B=B, H=H, Hq=Hq)
    k = rng.standard_normal((B, H, T, 128)).astype(np.float32)
    v = rng.standard_normal((B, H, T, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0, 0]))
    q = rng.standard_normal((B, Hq, 128)).astype(np.float32)
    lens = np.array([T, 37])
    out = c.decode(0, q, lens)
    for b in range(B):
        for i in range(Hq):
            ref = attention.plain_attention64(q[b, i:i + 1], k[b, i // 3, :lens[b]], v[b, i // 3, :lens[b]])
            assert np.allclose(out[b, i], ref[0], rtol=0, atol=1e-12)


def test_bulk_append_equals_token_by_token():
    rng = np.random.default_rng(14)
    k = rng.standard_normal((2, 2, 40, 128)).astype(np.float32)
    v = rng.standard_normal((2, 2, 40, 128)).astype(np.float32)
    a = _cache(16, 64, B=2, H=2, Hq=4)
    b = _cache(16, 64, B=2, H=2, Hq=4)
    a.append(0, k, v, np.array([3, 10]))
    for t in range(40):
        b.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1], np.array([3 + t, 10 + t]))
    for name in ("code", "scale", "zero"):
        assert np.array_equal(a.k[name], b.k[name]) and np.array_equal(a.v[name], b.v[name])
    assert np.array_equal(a.ring_k, b.ring_k) and np.array_equal(a.ring_v, b.ring_v)


def test_append_skips_sequences_with_negative_position():
    """pos[b] < 0 leaves sequence b untouched (records and ring), the others are written."""
    rng = np.random.default_rng(26)
    c = _cache(8, 32, B=3, H=1, Hq=2)
    k = rng.standard_normal((3, 1, 5, 128)).astype(np.float32)
    c.append(0, k, k, np.array([-1, 2, -1]))
    for rec in (c.k, c.v):
        for name in ("code", "scale", "zero"):
            assert not rec[name][0, 0].any() and not rec[name][0, 2].any()
            assert rec[name][0, 1, 0, 2:7].any()
    assert not c.ring_k[0, 0].any() and not c.ring_k[0, 2].any() and c.ring_k[0, 1].any()


def test_large_logits_stay_finite():
    """The softmax is taken relative to the running maximum, so logits of order 10^4 neither
    overflow nor lose the result (scipy's softmax as the reference)."""
    rng = np.random.default_rng(27)
    L = 40
    c = _cache(128, 64)
    k = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    c.append(0, k, v, np.array([0]))
    q = (rng.standard_normal((1, 2, 128)) * 1000).astype(np.float32)
    out = c.decode(0, q, np.array([L]))
    ref = attention.plain_attention64(q[0], k[0, 0], v[0, 0])
    assert np.all(np.isfinite(out)) and np.allclose(out[0], ref, rtol=0, atol=1e-12)


def test_empty_sequence_gives_zero_output():
    c = _cache(128, 16)
    out = c.decode(0, np.ones((1, 2, 128), np.float32), np.array([0]))
    assert np.all(out == 0)


def test_rotation_reduces_q4_error_with_outlier_channels():
    """[KV] TLDR: the Walsh-Hadamard rotation before 4-bit avoids the loss of flat q4 on outliers."""
    rng = np.random.default_rng(15)
    k = rng.standard_normal((512, 128)).astype(np.float32)
    k[:, :4] *= 10
    s = codec.wht_signs(0)
    flat = codec.q4g32_decode(*codec.q4g32_encode(k))
    rot = codec.unrotate(codec.q4g32_decode(*codec.q4g32_encode(codec.rotate(k, s))), s)
    err_flat = np.mean((flat - k) ** 2)
    err_rot = np.mean((rot - k) ** 2)
    assert err_rot < 0.7 * err_flat


def test_quantised_attention_tracks_full_precision():
    rng = np.random.default_rng(16)
    L = 600
    k = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 128)).astype(np.float32)
    q = rng.standard_normal((1, 2, 128)).astype(np.float32)
    c = _cache(0, L)
    c.append(0, k, v, np.array([0]))
    out = c.decode(0, q, np.array([L]))[0]
    ref = attention.plain_attention64(q[0], k[0, 0], v[0, 0])
    assert np.corrcoef(out.ravel(), ref.ravel())[0, 1] > 0.95


# ------------------------------------------------------------------ bytes ([QC] tables)
def test_compression_ratio_is_6_4():
    """[QC]: 6.4x KV compression = 32 bits / (4 + (16 + 16) / 32) bits per value."""
    cfg = attention.OracleConfig(1, 1, 1, 1, 1)
    per_value_bits = attention.payload_bytes_per_token_head(cfg) * 8 / (2 * 128)
    assert per_value_bits == 5.0 and 32 / per_value_bits == 6.4


def test_fp32_kv_at_32k_is_7_17_gb():
    """[QC] PPL table: FP32 KV memory at 32K for Llama 3.2 3B (28 layers, 8 kv heads) 7.17 GB."""
    b = attention.fp32_kv_bytes(28, 8, 32768)
    assert b == 7_516_192_768
    assert round(b / 2 ** 20 / 1000, 2) == 7.17


def test_progressive_window_costs_0_03_gb():
    """[QC] PPL table: 4-bit + progressive 2.33 GB vs 4-bit flat 2.30 GB -> window ~0.03 GB."""
    cfg = attention.OracleConfig(n_layers=28, n_kv_heads=8, n_q_heads=24, max_batch=1,
                                 max_seq_len=32768, window=128)
    w = attention.window_bytes(cfg)
    assert w == 28 * 8 * 128 * 128 * 4 * 2
    assert round(w / 1e9, 2) == 0.03


def test_tq_record_is_4_25_bits_and_compresses_over_4_5x():
    """[TQ] comparison table: compression >= 4.5x at ~3.5 bits; our key record is 4.25 bits."""
    assert attention.REC_BYTES[attention.TQ3_QJL] * 8 / 128 == 4.25
    assert 16 / 3.5 >= 4.5
    assert 32 / 4.25 > 4.5


# ------------------------------------------------------------------ chunked prefill (T queries)
def _prefill_case(window, p0, T, B=1, H=1, Hq=2, seed=40):
    rng = np.random.default_rng(seed)
    cap = p0 + T + 4
    c = _cache(window, cap, B=B, H=H, Hq=Hq, seed=3)
    kp = rng.standard_normal((B, H, p0, 128)).astype(np.float32)
    vp = rng.standard_normal((B, H, p0, 128)).astype(np.float32)
    if p0:
        c.append(0, kp, vp, np.zeros(B, int))
    k = rng.standard_normal((B, H, T, 128)).astype(np.float32)
    v = rng.standard_normal((B, H, T, 128)).astype(np.float32)
    q = rng.standard_normal((B, Hq, T, 128)).astype(np.float32)
    return c, np.concatenate([kp, k], axis=2), np.concatenate([vp, v], axis=2), k, v, q


@pytest.mark.parametrize("p0", [0, 20])
def test_prefill_with_covering_window_is_causal_attention(p0):
    """Window >= context: query t is exactly softmax attention over raw positions 0 .. p0 + t."""
    c, kall, vall, k, v, q = _prefill_case(128, p0, 40, B=2, H=2, Hq=6)
    out = attention.prefill(c, 0, k, v, q, np.array([p0, p0]))
    for b in range(2):
        for i in range(6):
            for t in range(40):
                L = p0 + t + 1
                ref = attention.plain_attention64(q[b, i:i + 1, t], kall[b, i // 3, :L], vall[b, i // 3, :L])
                assert np.allclose(out[b, i, t], ref[0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("window,p0,T", [(0, 3, 6), (4, 3, 10), (8, 0, 12)])
def test_prefill_matches_brute_force_with_sliding_window(window, p0, T):
    """Query t sees positions [0, L - W) through their records and [L - W, L) raw, L = p0 + t + 1;
    the brute force reads the raw window from the inputs, not from the ring."""
    c, kall, vall, k, v, q = _prefill_case(window, p0, T)
    out = attention.prefill(c, 0, k, v, q, np.array([p0]))
    for t in range(T):
        L = p0 + t + 1
        ref = _brute_force_unit(c, q[0, :, t], L, kall[0, 0], vall[0, 0])
        assert np.allclose(out[0, :, t], ref, rtol=0, atol=1e-10)


def test_prefill_is_causal_and_leaves_the_bulk_append_state():
    """Changing the chunk's tokens after t leaves query t's output unchanged; the cache afterwards
    holds exactly what one bulk append of the chunk writes ([QC] v3.2 note)."""
    c1, _, _, k, v, q = _prefill_case(4, 5, 9)
    c2, _, _, _, _, _ = _prefill_case(4, 5, 9)
    c3, _, _, _, _, _ = _prefill_case(4, 5, 9)
    out1 = attention.prefill(c1, 0, k, v, q, np.array([5]))
    k2, v2, q2 = k.copy(), v.copy(), q.copy()
    k2[:, :, 6:] += 1.0
    v2[:, :, 6:] -= 2.0
    q2[:, :, 6:] *= 3.0
    out2 = attention.prefill(c2, 0, k2, v2, q2, np.array([5]))
    assert np.array_equal(out1[:, :, :6], out2[:, :, :6])
    assert not np.allclose(out1[:, :, 6:], out2[:, :, 6:])
    c3.append(0, k, v, np.array([5]))
    for name in ("code", "scale", "zero"):
        assert np.array_equal(c1.k[name], c3.k[name]) and np.array_equal(c1.v[name], c3.v[name])
    assert np.array_equal(c1.ring_k, c3.ring_k) and np.array_equal(c1.ring_v, c3.ring_v)


def test_prefill_skips_inactive_sequences():
    c, _, _, k, v, q = _prefill_case(8, 0, 5, B=2)
    out = attention.prefill(c, 0, k, v, q, np.array([-1, 0]))
    assert not out[0].any() and out[1].any()
    assert not c.k["code"][0, 0].any()


def test_q4_key_codes_are_8x_fewer_bytes_than_fp32_keys():
    """[TQ] "inference cost" row: logits up to 8x faster at 4-bit than at 32-bit keys, i.e. the
    bytes a bandwidth-bound logit pass reads per key: 128 nibbles against 128 floats; with the
    group scales and zeros the Q4G32 record is 6.4x smaller."""
    fp32_key = 128 * 4
    codes = 128 // 2
    assert fp32_key / codes == 8
    assert fp32_key / attention.REC_BYTES[attention.Q4G32] == 6.4
