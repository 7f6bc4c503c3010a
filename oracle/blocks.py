"""Oracle of the two block codecs next to the cache: the outlier-channel split behind TurboQuant's
non-integer bit widths, and TBQ3_0 / TBQ4_0-style 256-value blocks (test infrastructure only).

Both are the TurboQuant MSE quantiser of [TQ] "key idea" row -- a random rotation, then a
per-coordinate optimal (Lloyd-Max) scalar quantiser of the unit vector, plus its norm -- applied to
blocks other than one 128-value head vector:

* Outlier split ([TQ] "method comparison" table: LongBench at 2.5 and 3.5 bits; "what the blogbot
  verified" list: the non-integer widths come from splitting off outlier channels, the page's own
  worked example being garbled).  Reading: the 128 channels of a vector are split into the 64
  outlier channels (largest mean square over a calibration block, ties to the lower index) and the
  64 others, each set in ascending channel order; the outlier set is coded at ``hi_bits`` and the
  other at ``hi_bits - 1`` bits, so (64 hi + 64 (hi - 1)) / 128 = hi - 0.5 bits per channel: 3.5
  bits for hi = 4, 2.5 for hi = 3 (the fp16 norms not counted, like the page's figures).  Each
  64-value set is rotated by a 64-point randomized Walsh-Hadamard transform with signs 0..63 (outlier
  set) or 64..127 (the others) of the cache's sign vector, c = 1/8.
* TBQ blocks ([TQ] "what the blogbot verified": the llama.cpp proposal adding TBQ3_0 / TBQ4_0;
  "limits and counterpoints": about 3.0625 / 4.0625 bits per value).  Reading: 3.0625 = 3 + 16/256,
  one fp16 value per 256 codes: a block is 256 consecutive values of a row (two 128-value heads of a
  token), rotated by a 256-point randomized Walsh-Hadamard transform (signs: the first 256 outputs
  of the SplitMix64 sign stream, c = 1/16), stored as its fp16 norm followed by the 256 b-bit codes:
  2 + 32 b bytes (98 B at 3 bits, 130 B at 4 bits).

Every float32 step is one numpy ufunc call on float32 operands (one rounding, no FMA), in the
order stated; the GPU kernels must reproduce the codes and the decoded values bit for bit.
"""

from __future__ import annotations

import numpy as np

from . import codec

F32 = np.float32
F16 = np.float16
FLT_MIN = codec.FLT_MIN


def signs_n(seed: int, n: int) -> np.ndarray:
    """The first ``n`` random +-1 signs of the SplitMix64 stream of ``seed`` (sign j = -1 when bit
    0 of output j+1 is set); its first 128 are the cache's rotation signs."""
    return np.array([-1.0 if (v & 1) else 1.0 for v in codec.splitmix64(seed, n)], dtype=F32)


def hadamard_n(x: np.ndarray) -> np.ndarray:
    """Unnormalised Sylvester-Hadamard product along the last axis (a power of two): stages
    h = 1, 2, 4, ... ascending, pairs (j, j + h) of each block of 2h becoming (a + b, a - b)."""
    x = np.asarray(x)
    n = x.shape[-1]
    lead = x.shape[:-1]
    h = 1
    while h < n:
        v = x.reshape(lead + (n // (2 * h), 2, h))
        a = v[..., 0, :]
        b = v[..., 1, :]
        x = np.stack((a + b, a - b), axis=-2).reshape(lead + (n,))
        h *= 2
    return x


def c_n(n: int):
    """float32 round-to-nearest of 1/sqrt(n) (exact for n = 64: 1/8, and n = 256: 1/16)."""
    return F32(1.0 / np.sqrt(float(n)))


def rotate_n(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = c H (s . x) in float32 over the last axis: sign flip, butterfly, one multiply by c."""
    x = np.asarray(x, dtype=F32)
    return hadamard_n(x * signs) * c_n(x.shape[-1])


def unrotate_n(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """x = s . (c H y), float32, same stage order."""
    y = np.asarray(y, dtype=F32)
    return (hadamard_n(y) * c_n(y.shape[-1])) * signs


def sumsq_tree(v: np.ndarray) -> np.ndarray:
    """Fixed-order float32 sum of squares over the last axis (n a power of two, n >= 8): squares
    rounded first, blocks of four consecutive ((v0^2 + v1^2) + (v2^2 + v3^2)), then the block sums
    halved: s[i] + s[i + n/8], then s[i] + s[i + n/16], ..., s[0] + s[1] (for n = 128 this is the
    cache's tree)."""
    v = np.asarray(v, dtype=F32)
    n = v.shape[-1]
    sq = v * v
    b = sq.reshape(sq.shape[:-1] + (n // 4, 4))
    s = (b[..., 0] + b[..., 1]) + (b[..., 2] + b[..., 3])
    m = n // 4
    while m > 1:
        m //= 2
        s = s[..., :m] + s[..., m:2 * m]
    return s[..., 0]


def mse_codebook(bits: int, dim: int):
    """2^bits-level codebook for a coordinate of a unit vector in R^dim, i.e. of N(0, 1/dim): the
    unit-variance Lloyd-Max centroids times 1/sqrt(dim) (float64), rounded to fp16; boundaries are
    the float32 midpoints of adjacent fp16 centroids.  Returns (centroids f16, boundaries f32)."""
    c64, _ = codec.lloyd_max_gaussian(2 ** bits)
    cent = (c64 / np.sqrt(float(dim))).astype(F16)
    c32 = cent.astype(F32)
    return cent, (c32[:-1] + c32[1:]) / F32(2.0)


def mse_encode(y: np.ndarray, bits: int):
    """Norm and codes of rotated vectors y [..., dim]: n = sqrt(sumsq), u = y * (1 / max(n, FLT_MIN))
    ([QC] v3.19 normalisation form), code = number of boundaries <= u (ties go up).  Returns
    (codes uint8 [..., dim], norm f16 [...])."""
    y = np.asarray(y, dtype=F32)
    dim = y.shape[-1]
    _, bnd = mse_codebook(bits, dim)
    n = np.sqrt(sumsq_tree(y))
    inv = F32(1.0) / np.maximum(n, FLT_MIN)
    u = y * inv[..., None]
    code = (u[..., None] >= bnd).sum(axis=-1).astype(np.uint8)
    return code, n.astype(F16)


def mse_decode(code: np.ndarray, norm: np.ndarray, bits: int) -> np.ndarray:
    """Rotated-space value f32(norm) * f32(centroid[code]) (one rounding)."""
    cent, _ = mse_codebook(bits, code.shape[-1])
    return norm.astype(F32)[..., None] * cent.astype(F32)[code]


def pack_bits(code: np.ndarray, bits: int) -> np.ndarray:
    """Codes [..., n] as a little-endian bit stream: code j at bits [bits j, bits j + bits)."""
    code = np.asarray(code, dtype=np.uint8)
    bitarr = ((code[..., None] >> np.arange(bits, dtype=np.uint8)) & 1).reshape(code.shape[:-1] + (-1,))
    return np.packbits(bitarr, axis=-1, bitorder="little")


def unpack_bits(stream: np.ndarray, bits: int, n: int) -> np.ndarray:
    bitarr = np.unpackbits(np.asarray(stream, np.uint8), axis=-1, bitorder="little")[..., :bits * n]
    bitarr = bitarr.reshape(bitarr.shape[:-1] + (n, bits))
    return (bitarr << np.arange(bits, dtype=np.uint8)).sum(axis=-1).astype(np.uint8)


def _f16_bytes(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, F16)[..., None].view(np.uint8)


# ------------------------------------------------------------------------------ TBQ blocks
TBQ_N = 256


def tbq_block_bytes(bits: int) -> int:
    return 2 + TBQ_N * bits // 8


def tbq_encode(x: np.ndarray, bits: int, seed: int) -> np.ndarray:
    """Blocks of 256 values x [..., 256] -> bytes [..., 2 + 32 bits]: fp16 norm, then the codes."""
    y = rotate_n(x, signs_n(seed, TBQ_N))
    code, norm = mse_encode(y, bits)
    return np.concatenate([_f16_bytes(norm), pack_bits(code, bits)], axis=-1)


def tbq_decode(blocks: np.ndarray, bits: int, seed: int) -> np.ndarray:
    """bytes [..., 2 + 32 bits] -> values [..., 256] float32: centroid times norm, inverse rotation."""
    blocks = np.asarray(blocks, np.uint8)
    norm = np.ascontiguousarray(blocks[..., :2]).view(F16)[..., 0]
    code = unpack_bits(blocks[..., 2:], bits, TBQ_N)
    return unrotate_n(mse_decode(code, norm, bits), signs_n(seed, TBQ_N))


# ------------------------------------------------------------------------------ outlier split
SPLIT_N = 64


def split_record_bytes(hi_bits: int) -> int:
    """fp16 norms of both sets, then 64 hi-bit codes and 64 (hi - 1)-bit codes."""
    return 4 + SPLIT_N * hi_bits // 8 + SPLIT_N * (hi_bits - 1) // 8


def split_outliers(calib: np.ndarray) -> np.ndarray:
    """The 64 channels with the largest mean square over a calibration block [T][128], ascending.
    Each channel's sum of squares is taken in float64, token by token in order (the squares of
    float32 inputs are exact in float64); ties go to the lower channel index."""
    x = np.asarray(calib, np.float64)
    ss = np.zeros(codec.D, np.float64)
    for t in range(x.shape[0]):
        ss = ss + x[t] * x[t]
    order = np.lexsort((np.arange(codec.D), -ss))  # largest first, lower index first among equals
    return np.sort(order[:SPLIT_N]).astype(np.int16)


def _split_sets(outliers: np.ndarray):
    o = np.asarray(outliers, np.int64)
    r = np.setdiff1d(np.arange(codec.D), o)
    return o, r


def split_encode(x: np.ndarray, outliers: np.ndarray, hi_bits: int, seed: int) -> np.ndarray:
    """Vectors x [..., 128] -> records [..., split_record_bytes(hi_bits)]."""
    x = np.asarray(x, F32)
    o, r = _split_sets(outliers)
    s = signs_n(seed, codec.D)
    co, no = mse_encode(rotate_n(x[..., o], s[:SPLIT_N]), hi_bits)
    cr, nr = mse_encode(rotate_n(x[..., r], s[SPLIT_N:]), hi_bits - 1)
    return np.concatenate([_f16_bytes(no), _f16_bytes(nr), pack_bits(co, hi_bits), pack_bits(cr, hi_bits - 1)],
                          axis=-1)


def split_decode(rec: np.ndarray, outliers: np.ndarray, hi_bits: int, seed: int) -> np.ndarray:
    """records [..., split_record_bytes(hi_bits)] -> vectors [..., 128] float32."""
    rec = np.asarray(rec, np.uint8)
    o, r = _split_sets(outliers)
    s = signs_n(seed, codec.D)
    no = np.ascontiguousarray(rec[..., 0:2]).view(F16)[..., 0]
    nr = np.ascontiguousarray(rec[..., 2:4]).view(F16)[..., 0]
    nbo = SPLIT_N * hi_bits // 8
    co = unpack_bits(rec[..., 4:4 + nbo], hi_bits, SPLIT_N)
    cr = unpack_bits(rec[..., 4 + nbo:], hi_bits - 1, SPLIT_N)
    out = np.zeros(rec.shape[:-1] + (codec.D,), F32)
    out[..., o] = unrotate_n(mse_decode(co, no, hi_bits), s[:SPLIT_N])
    out[..., r] = unrotate_n(mse_decode(cr, nr, hi_bits - 1), s[SPLIT_N:])
    return out
