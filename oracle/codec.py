"""Oracle codec: rotation, balancing and quantisers of the KV cache (test infrastructure only).

Every float32 step below is one numpy ufunc call on float32 operands, so it rounds exactly once
(IEEE round-to-nearest-even) and never fuses a multiply with an add.  The order of operations is
the one stated in each docstring; the GPU library must reproduce the codes bit for bit.

Page references:
  [QC] "Beyond RAG: load the whole document on your laptop" (quant.cpp summary)
  [KV] "Running Bonsai ternary 27B at 120K context in under 10 GB of VRAM" (KVarN port)
  [TQ] "LLM memory saving: weights vs KV-cache quantization (2026)"
"""

from __future__ import annotations

import numpy as np

F32 = np.float32
F16 = np.float16
D = 128                      # head_dim: every workload on the pages' models uses 128
GROUP = 32                   # Q4 group size along head_dim
N_GROUPS = D // GROUP
FLT_MIN = F32(np.finfo(np.float32).tiny)
# c = float32 round-to-nearest of 1/sqrt(128) = 2^-3.5 (bit pattern 0x3DB504F3); applied after the
# unnormalised butterfly so that c*H is orthogonal up to the rounding of c.
C_WHT = F32(1.0 / np.sqrt(128.0))

_M64 = (1 << 64) - 1


# --------------------------------------------------------------------------------------------
# Random signs of the rotation: SplitMix64 (Steele, Lea & Flood 2014; Vigna's splitmix64.c).
# --------------------------------------------------------------------------------------------
def splitmix64(seed: int, n: int) -> list[int]:
    """First ``n`` outputs of the SplitMix64 sequence whose state starts at ``seed``.

    state += 0x9E3779B97F4A7C15; z = state; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9;
    z = (z ^ z>>27) * 0x94D049BB133111EB; output z ^ z>>31 (all mod 2^64).
    """
    out = []
    state = seed & _M64
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _M64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        out.append(z ^ (z >> 31))
    return out


def wht_signs(seed: int) -> np.ndarray:
    """The random +-1 diagonal of the randomized Walsh-Hadamard rotation.

    [KV] TLDR (Walsh-Hadamard before 4-bit) and [TQ] "key idea" row (random rotation).  The pages
    give no generator; reading: sign_j = -1 when bit 0 of the (j+1)-th SplitMix64 output is 1,
    one vector for every layer and head.
    """
    return np.array([-1.0 if (v & 1) else 1.0 for v in splitmix64(seed, D)], dtype=F32)


# --------------------------------------------------------------------------------------------
# Walsh-Hadamard transform
# --------------------------------------------------------------------------------------------
def hadamard_butterfly(x: np.ndarray) -> np.ndarray:
    """Unnormalised Sylvester-Hadamard product H x along the last axis (length 128).

    Stages h = 1, 2, 4, ..., 64 in that order; in each, the element pairs (j, j+h) of every block of
    2h elements become (a + b, a - b).  The dtype of ``x`` is kept (float32 or float64).
    """
    x = np.asarray(x)
    lead = x.shape[:-1]
    h = 1
    while h < D:
        v = x.reshape(lead + (D // (2 * h), 2, h))
        a = v[..., 0, :]
        b = v[..., 1, :]
        x = np.stack((a + b, a - b), axis=-2).reshape(lead + (D,))
        h *= 2
    return x


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """y = c * H (s (.) x) in float32: sign flip (exact), butterfly, then one multiply by c."""
    x = np.asarray(x, dtype=F32)
    return hadamard_butterfly(x * signs) * C_WHT


def unrotate(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Inverse rotation x = s (.) (c * H y), float32, same stage order as ``rotate``."""
    y = np.asarray(y, dtype=F32)
    return (hadamard_butterfly(y) * C_WHT) * signs


def rotate64(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Same rotation in float64 (for the attention oracle), with the float32 value of c."""
    return hadamard_butterfly(np.asarray(x, np.float64) * signs.astype(np.float64)) * float(C_WHT)


def unrotate64(y: np.ndarray, signs: np.ndarray) -> np.ndarray:
    return (hadamard_butterfly(np.asarray(y, np.float64)) * float(C_WHT)) * signs.astype(np.float64)


# --------------------------------------------------------------------------------------------
# Fixed-order sums used by the norm, the Sinkhorn row statistic and the residual norm
# --------------------------------------------------------------------------------------------
def sumsq128(v: np.ndarray) -> np.ndarray:
    """Sum of squares over the last axis (128) in a fixed float32 tree.

    Squares are rounded first.  Blocks of four consecutive elements are added as
    ((v0^2 + v1^2) + (v2^2 + v3^2)); the 32 block sums are then halved: s[i] + s[i+16], then
    s[i] + s[i+8], ..., s[0] + s[1].  (The pages fix only that the reduction order is fixed:
    [QC] v3.18 note on determinism.)
    """
    v = np.asarray(v, dtype=F32)
    sq = v * v
    b = sq.reshape(sq.shape[:-1] + (D // 4, 4))
    s = (b[..., 0] + b[..., 1]) + (b[..., 2] + b[..., 3])
    n = D // 4
    while n > 1:
        n //= 2
        s = s[..., :n] + s[..., n:2 * n]
    return s[..., 0]


# --------------------------------------------------------------------------------------------
# 4-bit asymmetric group quantiser (Q4G32)
# --------------------------------------------------------------------------------------------
def q4g32_encode(y: np.ndarray):
    """4-bit codes with per-group fp16 scale and zero for groups of 32 consecutive channels.

    [QC] "how it works": everything outside the FP32 window is 4-bit.  Per group: exact min and
    max; scale = f16(f32(max - min) / 15); zero = f16(min); code = clamp(rint(f32(y - zero) /
    scale), 0, 15) with round-half-even, or 0 when scale == 0.  Returns (codes uint8 [...,128],
    scale f16 [...,4], zero f16 [...,4]).
    """
    y = np.asarray(y, dtype=F32)
    g = y.reshape(y.shape[:-1] + (N_GROUPS, GROUP))
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    scale = ((mx - mn) / F32(15.0)).astype(F16)
    zero = mn.astype(F16)
    s = scale.astype(F32)[..., None]
    z = zero.astype(F32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (g - z) / s
    code = np.where(s > 0, np.clip(np.rint(t), 0, 15), 0).astype(np.uint8)
    return code.reshape(y.shape), scale, zero


def q4g32_decode(code: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """Dequantised value f32(zero + f32(scale * code)) (two roundings, no FMA)."""
    c = np.asarray(code).reshape(code.shape[:-1] + (N_GROUPS, GROUP)).astype(F32)
    out = zero.astype(F32)[..., None] + scale.astype(F32)[..., None] * c
    return out.reshape(code.shape)


# --------------------------------------------------------------------------------------------
# 8-bit symmetric group quantiser (Q8G32) for keys kept at 8 bits
# --------------------------------------------------------------------------------------------
def q8g32_encode(y: np.ndarray):
    """8-bit codes with one fp16 scale per group of 32 consecutive channels, no zero point.

    [TQ] "when to use what" and "rules" lists: keep K at Q8 and cut only V to low bits.  The page
    names the llama.cpp cache type without defining it; reading: its 8-bit block format (32 values,
    one fp16 scale d = max|y| / 127, signed codes).  Per group: d = f16(f32(max |y|) / 127);
    code = clamp(rint(y / f32(d)), -127, 127) with round-half-even against the STORED scale, or 0
    when d == 0.  Returns (codes int8 [...,128], d f16 [...,4]).
    """
    y = np.asarray(y, dtype=F32)
    g = y.reshape(y.shape[:-1] + (N_GROUPS, GROUP))
    amax = np.abs(g).max(axis=-1)
    d = (amax / F32(127.0)).astype(F16)
    df = d.astype(F32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = g / df
    code = np.where(df > 0, np.clip(np.rint(t), -127, 127), 0).astype(np.int8)
    return code.reshape(y.shape), d


def q8g32_decode(code: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Dequantised value f32(d * code) (one rounding; exact, since |code| < 2^8 and d is fp16)."""
    c = np.asarray(code).reshape(code.shape[:-1] + (N_GROUPS, GROUP)).astype(F32)
    return (d.astype(F32)[..., None] * c).reshape(code.shape)


# --------------------------------------------------------------------------------------------
# Lloyd-Max scalar quantiser for a Gaussian and the 3-bit TurboQuant key codec
# --------------------------------------------------------------------------------------------
def lloyd_max_gaussian(levels: int = 8, tol: float = 1e-15, max_iter: int = 200000):
    """Lloyd-Max (minimum-MSE) quantiser of N(0, 1) in float64.

    [TQ] "key idea" row: the per-coordinate optimal scalar quantiser after a random rotation.
    Lloyd's iteration alternates the midpoint condition (boundaries halfway between centroids)
    and the centroid condition (each centroid is E[X | X in its cell], closed form
    (phi(a) - phi(b)) / (Phi(b) - Phi(a))).  Returns (centroids, boundaries), ascending.
    """
    from scipy.special import ndtr

    c = np.linspace(-2.0, 2.0, levels)
    for _ in range(max_iter):
        b = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-np.inf], b, [np.inf]))
        pdf = np.exp(-0.5 * edges * edges) / np.sqrt(2.0 * np.pi)
        mass = ndtr(edges[1:]) - ndtr(edges[:-1])
        c_new = (pdf[:-1] - pdf[1:]) / mass
        done = np.max(np.abs(c_new - c)) < tol
        c = c_new
        if done:
            break
    return c, 0.5 * (c[:-1] + c[1:])


def tq3_codebook():
    """3-bit codebook for a coordinate of a unit vector in R^128, i.e. of N(0, 1/128).

    Centroids: the unit-variance Lloyd-Max values times 1/sqrt(128) (float64), rounded to fp16.
    Boundaries: float32 midpoints of adjacent fp16 centroids (exact in float32).
    Returns (centroids f16 [8], boundaries f32 [7]).
    """
    c64, _ = lloyd_max_gaussian(8)
    cent = (c64 / np.sqrt(128.0)).astype(F16)
    c32 = cent.astype(F32)
    bnd = (c32[:-1] + c32[1:]) / F32(2.0)
    return cent, bnd


def tq3_qjl_encode(y: np.ndarray, proj: np.ndarray):
    """TurboQuant-style key code: 3-bit Lloyd-Max codes of the unit vector plus a QJL sign sketch.

    [TQ] "key idea" row: random rotation (applied by the caller), per-coordinate optimal scalar
    quantiser, 1-bit QJL on the residual for an unbiased inner product.  [QC] v3.19 note gives the
    normalisation form 1/max(sqrt(ss), eps); eps = FLT_MIN (the page states none).

    Steps (float32): n = sqrt(sumsq128(y)); inv = 1 / max(n, FLT_MIN); u = y * inv;
    code_j = number of boundaries <= u_j; r = u - centroid[code]; gamma = sqrt(sumsq128(r));
    t_i = sum over j = 0..127 in order of f32(proj[i, j] * r_j); bit_i = (t_i >= 0).
    Returns (codes uint8 [...,128], bits bool [...,128], n f16 [...], gamma f16 [...]).
    """
    y = np.asarray(y, dtype=F32)
    proj = np.asarray(proj, dtype=F32)
    cent, bnd = tq3_codebook()
    n = np.sqrt(sumsq128(y))
    inv = F32(1.0) / np.maximum(n, FLT_MIN)
    u = y * inv[..., None]
    code = (u[..., None] >= bnd).sum(axis=-1).astype(np.uint8)
    r = u - cent.astype(F32)[code]
    gamma = np.sqrt(sumsq128(r))
    t = np.zeros(y.shape[:-1] + (D,), dtype=F32)
    for j in range(D):
        t = t + proj[:, j] * r[..., j:j + 1]
    bits = t >= 0
    return code, bits, n.astype(F16), gamma.astype(F16)


QJL_CONST = np.sqrt(np.pi / 2.0) / D   # sqrt(pi/2)/m with m = 128 projections


def tq3_qjl_dot64(q: np.ndarray, code, bits, n, gamma, proj) -> np.ndarray:
    """Estimated <q, y> of a TQ3+QJL key, in float64 (for the attention oracle).

    <q, y> ~= n * (<q, c[code]> + sqrt(pi/2)/128 * gamma * <S q, 2 bits - 1>), with the stored fp16
    n and gamma.  ``q``: [..., 128] float64 (already rotated); key arrays [..., T, ...].
    Returns [..., T].
    """
    cent, _ = tq3_codebook()
    khat = cent.astype(np.float64)[code]                      # [..., T, 128]
    sq = np.einsum("ij,...j->...i", proj.astype(np.float64), q)  # [..., 128]
    sgn = np.where(bits, 1.0, -1.0)
    dot_c = np.einsum("...tj,...j->...t", khat, q)
    dot_s = np.einsum("...ti,...i->...t", sgn, sq)
    return n.astype(np.float64) * (dot_c + QJL_CONST * gamma.astype(np.float64) * dot_s)


# --------------------------------------------------------------------------------------------
# Sinkhorn variance balancing (KVarN)
# --------------------------------------------------------------------------------------------
SINKHORN_ITERS = 8


def sinkhorn_sigma(x_rot: np.ndarray, iters: int = SINKHORN_ITERS) -> np.ndarray:
    """Per-channel balancing scale sigma (fp16 [128]) from a rotated calibration block [n, 128].

    [KV] TLDR: Sinkhorn variance balancing after the Walsh-Hadamard transform, before 4-bit.  The
    page names the method only; reading (float32 throughout):
      repeat ``iters`` times:
        row step:    rho_i   = sqrt(sumsq128(X_i) / 128);      X_i /= rho_i   (rho_i = 0 -> 1)
        column step: kappa_j = sqrt(S_j / n), S_j = sum over tokens t = 0..n-1 in order of X_tj^2;
                     X_j /= kappa_j (kappa_j = 0 -> 1);        sigma_j *= kappa_j
      sigma -> fp16.
    Parity of this reading is unpinned by the pages; invariants checked instead: a block with
    planted column scales gives sigma proportional to them, a balanced block gives sigma ~ 1, and
    the balanced block has unit column RMS.
    """
    x = np.array(x_rot, dtype=F32, copy=True)
    ntok = x.shape[0]
    sigma = np.ones(D, dtype=F32)
    for _ in range(iters):
        rho = np.sqrt(sumsq128(x) / F32(D))
        rho = np.where(rho > 0, rho, F32(1.0))
        x = x / rho[:, None]
        s = np.zeros(D, dtype=F32)
        for t in range(ntok):
            s = s + x[t] * x[t]
        kappa = np.sqrt(s / F32(ntok))
        kappa = np.where(kappa > 0, kappa, F32(1.0))
        x = x / kappa[None, :]
        sigma = sigma * kappa
    return sigma.astype(F16)
