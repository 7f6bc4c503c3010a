"""Pins of the block-codec oracle (oracle/blocks.py): the outlier-channel split and TBQ blocks.

Each function is checked against something other than itself: the Max (1960) Gaussian quantizer
tables, scipy's Sylvester Hadamard matrices, the cache's own rotation signs and summation tree,
brute-force nearest centroids, the optimal quantizers' published distortions, a hand-computed
bit stream, and the bit widths the pages print (3.0625 / 4.0625 for the TBQ blocks, 2.5 / 3.5 for
the split).
"""

import os

import numpy as np
import pytest

from oracle import blocks, codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# mean squared error of the optimal 2^b-level quantizer of a unit Gaussian (Max 1960, Table I)
LLOYD_MAX_MSE = {2: 0.1175, 3: 0.03454, 4: 0.009497}


def _golden(name):
    rows = [r for r in open(os.path.join(GOLDEN, name)).read().splitlines() if r and not r.startswith("#")]
    return [np.array([float(x) for x in r.split()]) for r in rows]


@pytest.mark.parametrize("levels,name", [(4, "lloyd_max_gaussian_4.txt"), (16, "lloyd_max_gaussian_16.txt")])
def test_lloyd_max_tables(levels, name):
    out, thr = _golden(name)
    c, b = codec.lloyd_max_gaussian(levels)
    assert np.allclose(c[levels // 2:], out, atol=6e-4)
    assert np.allclose(b[levels // 2 - 1:], thr, atol=6e-4)
    assert np.allclose(c, -c[::-1], atol=1e-12)


@pytest.mark.parametrize("n", [8, 64, 256])
def test_hadamard_n_is_sylvester(n):
    from scipy.linalg import hadamard

    assert np.array_equal(blocks.hadamard_n(np.eye(n)), hadamard(n))
    h = blocks.hadamard_n(np.eye(n))
    assert np.array_equal(h @ h.T, n * np.eye(n))


def test_normalisations_are_exact_powers_of_two():
    assert blocks.c_n(64) == np.float32(0.125) and blocks.c_n(256) == np.float32(0.0625)
    assert blocks.c_n(128) == codec.C_WHT


def test_signs_extend_the_cache_signs():
    for seed in (0, 7, 12345):
        assert np.array_equal(blocks.signs_n(seed, 256)[:128], codec.wht_signs(seed))


@pytest.mark.parametrize("n", [64, 256])
def test_rotation_is_orthonormal_and_inverted(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal((50, n)).astype(np.float32)
    s = blocks.signs_n(3, n)
    y = blocks.rotate_n(x, s)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-5)
    assert np.allclose(blocks.unrotate_n(y, s), x, atol=2e-6 * np.abs(x).max())
    # rotated unit vectors are signed, scaled Hadamard columns
    e = np.eye(n, dtype=np.float32)
    from scipy.linalg import hadamard

    assert np.array_equal(blocks.rotate_n(e, s), (hadamard(n) * s[None, :] * blocks.c_n(n)).T.astype(np.float32))


def test_sum_tree_is_the_cache_tree_at_128():
    x = np.random.default_rng(1).standard_normal((500, 128)).astype(np.float32)
    assert np.array_equal(blocks.sumsq_tree(x).view(np.uint32), codec.sumsq128(x).view(np.uint32))


@pytest.mark.parametrize("n", [64, 256])
def test_sum_tree_shape(n):
    """1 and two squares of 2^-24 in blocks 1 and 1 + n/8: the tree adds the small ones first and
    reaches 1 + 2^-23 exactly; left to right, each small one rounds away."""
    v = np.zeros(n, np.float32)
    v[0] = 1.0
    v[4] = v[4 + n // 2] = 2.0 ** -12
    assert blocks.sumsq_tree(v) == np.float32(1.0 + 2.0 ** -23)
    seq = np.float32(0.0)
    for x in v:
        seq = np.float32(seq + np.float32(x * x))
    assert seq == np.float32(1.0)


def test_codebook_at_128_is_the_cache_tq3_codebook():
    """The 3-bit codebook of a 128-dimensional unit vector is the one the cache's TQ3 keys use."""
    cent, bnd = blocks.mse_codebook(3, 128)
    c3, b3 = codec.tq3_codebook()
    assert np.array_equal(cent.view(np.uint16), c3.view(np.uint16))
    assert np.array_equal(bnd.view(np.uint32), b3.view(np.uint32))


@pytest.mark.parametrize("bits,dim", [(2, 64), (3, 64), (4, 64), (3, 256), (4, 256)])
def test_codes_are_nearest_centroids(bits, dim):
    rng = np.random.default_rng(bits * 1000 + dim)
    y = rng.standard_normal((400, dim)).astype(np.float32) * np.float32(3.0)
    code, norm = blocks.mse_encode(y, bits)
    cent, _ = blocks.mse_codebook(bits, dim)
    n = np.sqrt(blocks.sumsq_tree(y))
    u = (y * (np.float32(1.0) / n)[:, None]).astype(np.float64)
    best = np.argmin(np.abs(u[..., None] - cent.astype(np.float64)), axis=-1)
    assert np.array_equal(code, best)
    assert np.array_equal(norm, n.astype(np.float16))
    assert code.max() <= 2 ** bits - 1


@pytest.mark.parametrize("bits,dim", [(2, 64), (3, 64), (4, 64), (3, 256), (4, 256)])
def test_distortion_is_the_optimal_quantizers(bits, dim):
    """Per-coordinate squared error of the unit vector, times dim, is the Lloyd-Max distortion of a
    unit Gaussian (a wrong 1/sqrt(dim) scale or codebook would miss it by far)."""
    rng = np.random.default_rng(7 + bits)
    y = rng.standard_normal((6000, dim)).astype(np.float32)
    code, norm = blocks.mse_encode(y, bits)
    cent, _ = blocks.mse_codebook(bits, dim)
    u = y / np.linalg.norm(y, axis=1, keepdims=True)
    mse = np.mean((u - cent.astype(np.float64)[code]) ** 2) * dim
    assert abs(mse / LLOYD_MAX_MSE[bits] - 1.0) < 0.06


def test_bit_stream_order():
    code = np.array([1, 2, 3, 4, 5, 6, 7, 0], np.uint8)
    # little endian: code j at bits 3j .. 3j+2 of the stream
    bits = "".join(format(c, "03b")[::-1] for c in code)
    want = np.array([int(bits[8 * i:8 * i + 8][::-1], 2) for i in range(3)], np.uint8)
    assert np.array_equal(blocks.pack_bits(code, 3), want)
    assert want[0] == 0xD1
    rng = np.random.default_rng(0)
    for b in (2, 3, 4):
        c = rng.integers(0, 2 ** b, (10, 256)).astype(np.uint8)
        assert np.array_equal(blocks.unpack_bits(blocks.pack_bits(c, b), b, 256), c)


def test_record_sizes_are_the_pages_bit_widths():
    """[TQ]: TBQ3_0 / TBQ4_0 about 3.0625 / 4.0625 bits; TurboQuant at 2.5 / 3.5 bits a channel."""
    assert blocks.tbq_block_bytes(3) == 98 and 8 * 98 / 256 == 3.0625
    assert blocks.tbq_block_bytes(4) == 130 and 8 * 130 / 256 == 4.0625
    assert blocks.split_record_bytes(3) == 44 and 8 * (44 - 4) / 128 == 2.5
    assert blocks.split_record_bytes(4) == 60 and 8 * (60 - 4) / 128 == 3.5


@pytest.mark.parametrize("bits", [3, 4])
def test_tbq_roundtrip(bits):
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((300, 256)).astype(np.float32) * np.float32(2.0)
    blk = blocks.tbq_encode(x, bits, seed=5)
    assert blk.shape == (300, blocks.tbq_block_bytes(bits))
    xr = blocks.tbq_decode(blk, bits, seed=5)
    rel = np.mean((xr - x) ** 2) / np.mean(x ** 2)
    assert abs(rel / LLOYD_MAX_MSE[bits] - 1.0) < 0.08
    # the decoded block re-encodes to the same codes (its rotation is centroids times the norm)
    assert np.array_equal(blocks.unpack_bits(blocks.tbq_encode(xr, bits, 5)[:, 2:], bits, 256),
                          blocks.unpack_bits(blk[:, 2:], bits, 256))


def test_tbq_zero_block_and_seed():
    blk = blocks.tbq_encode(np.zeros((2, 256), np.float32), 4, 0)
    # u = 0 lies on the middle boundary (midpoint of +-c): ties go up, to code 2^(b-1)
    assert (blocks.unpack_bits(blk[:, 2:], 4, 256) == 8).all()
    z = blocks.tbq_decode(blk, 4, 0)
    assert not z.any()
    x = np.random.default_rng(2).standard_normal((4, 256)).astype(np.float32)
    assert not np.array_equal(blocks.tbq_encode(x, 3, 0), blocks.tbq_encode(x, 3, 1))


def test_split_outliers_are_the_largest_channels():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1000, 128))
    big = np.sort(rng.permutation(128)[:64])
    x[:, big] *= 5.0
    assert np.array_equal(blocks.split_outliers(x), big)
    assert np.array_equal(blocks.split_outliers(np.ones((10, 128))), np.arange(64))


@pytest.mark.parametrize("hi", [3, 4])
def test_split_roundtrip_and_partition(hi):
    rng = np.random.default_rng(hi)
    x = rng.standard_normal((400, 128)).astype(np.float32)
    o = np.sort(rng.permutation(128)[:64]).astype(np.int16)
    x[:, o] *= np.float32(6.0)
    rec = blocks.split_encode(x, o, hi, seed=0)
    assert rec.shape == (400, blocks.split_record_bytes(hi))
    xr = blocks.split_decode(rec, o, hi, seed=0)
    r = np.setdiff1d(np.arange(128), o)
    for idx, bits in ((o, hi), (r, hi - 1)):
        rel = np.mean((xr[:, idx] - x[:, idx]) ** 2) / np.mean(x[:, idx] ** 2)
        assert abs(rel / LLOYD_MAX_MSE[bits] - 1.0) < 0.1
    # the outlier set's norm goes first: scaling only the outliers changes only the first norm
    x2 = x.copy()
    x2[:, o] *= np.float32(2.0)
    rec2 = blocks.split_encode(x2, o, hi, seed=0)
    assert np.array_equal(rec2[:, 2:4], rec[:, 2:4]) and not np.array_equal(rec2[:, 0:2], rec[:, 0:2])
