"""The oracle's pins catch plausible mistakes: each mutant below plants one in a copy of the oracle.

Each case loads ``oracle/`` from source with one textual change applied (in memory, in a child
interpreter, nothing is written to disk) and runs ``tests/test_oracle_pins.py`` against it; the
pins must fail.  The mistakes are the kinds a restatement of the pages could plausibly contain:
a dropped factor or term, a wrong constant, a transposed operand, a wrong index, a changed
tie or rounding rule, a different summation tree, a dropped step of an iteration.

Mutants that are equivalent to the original are not listed: reading the window's slots in another
order (the same set of tokens), writing every appended token to the ring instead of only the last
``window`` ones (later writes win), another softmax shift at moderate logits.  The choice of bit in
the sign generator is a reading the pages leave open; the GPU parity tests fix it instead.
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (file, original text, mutated text); the original must occur exactly once.
MUTANTS = [
    # rotation and the fixed-order sum
    ("codec.py", "x = np.stack((a + b, a - b), axis=-2)", "x = np.stack((a + b, b - a), axis=-2)"),
    ("codec.py", "return hadamard_butterfly(x * signs) * C_WHT", "return hadamard_butterfly(x) * C_WHT"),
    ("codec.py", "return (hadamard_butterfly(y) * C_WHT) * signs", "return hadamard_butterfly(y * signs) * C_WHT"),
    ("codec.py", "z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9)", "z = ((z ^ (z >> 31)) * 0xBF58476D1CE4E5B9)"),
    ("codec.py", "s = (b[..., 0] + b[..., 1]) + (b[..., 2] + b[..., 3])",
                 "s = ((b[..., 0] + b[..., 1]) + b[..., 2]) + b[..., 3]"),
    ("codec.py", "s = s[..., :n] + s[..., n:2 * n]", "s = s[..., 0:2 * n:2] + s[..., 1:2 * n:2]"),
    # Q4G32
    ("codec.py", "scale = ((mx - mn) / F32(15.0)).astype(F16)", "scale = ((mx - mn) / F32(16.0)).astype(F16)"),
    ("codec.py", "zero = mn.astype(F16)", "zero = (mn - F32(0.0009765625)).astype(F16)"),
    ("codec.py", "t = (g - z) / s", "t = (g - mn[..., None]) / s"),
    ("codec.py", "code = np.where(s > 0, np.clip(np.rint(t), 0, 15), 0)",
                 "code = np.where(s > 0, np.clip(np.floor(t + F32(0.5)), 0, 15), 0)"),
    ("codec.py", "code = np.where(s > 0, np.clip(np.rint(t), 0, 15), 0)",
                 "code = np.where(s > 0, np.clip(np.floor(t), 0, 15), 0)"),
    ("codec.py", "out = zero.astype(F32)[..., None] + scale.astype(F32)[..., None] * c",
                 "out = (zero.astype(F32)[..., None] / scale.astype(F32)[..., None] + c)"
                 " * scale.astype(F32)[..., None]"),
    # Q8G32 keys
    ("codec.py", "d = (amax / F32(127.0)).astype(F16)", "d = (amax / F32(128.0)).astype(F16)"),
    ("codec.py", "amax = np.abs(g).max(axis=-1)", "amax = g.max(axis=-1)"),
    ("codec.py", "code = np.where(df > 0, np.clip(np.rint(t), -127, 127), 0)",
                 "code = np.where(df > 0, np.clip(np.trunc(t), -127, 127), 0)"),
    ("codec.py", "return (d.astype(F32)[..., None] * c).reshape(code.shape)",
                 "return (d.astype(F32)[..., None] * (c + F32(0.5))).reshape(code.shape)"),
    ("attention.py", "c, s = codec.q8g32_encode(self._balanced(k[b, h], sk))",
                     "c, s = codec.q8g32_encode(codec.rotate(k[b, h], self.signs))"),
    ("attention.py", "kd = codec.q8g32_decode(self.k[\"code\"][layer, b, h, :Lq],",
                     "kd = -codec.q8g32_decode(self.k[\"code\"][layer, b, h, :Lq],"),
    # Lloyd-Max codebook and TQ3 + QJL keys
    ("codec.py", "b = 0.5 * (c[:-1] + c[1:])\n        edges", "b = 0.45 * (c[:-1] + c[1:])\n        edges"),
    ("codec.py", "cent = (c64 / np.sqrt(128.0)).astype(F16)", "cent = (c64 / np.sqrt(127.0)).astype(F16)"),
    ("codec.py", "bnd = (c32[:-1] + c32[1:]) / F32(2.0)", "bnd = c32[:-1] + (c32[1:] - c32[:-1]) / F32(3.0)"),
    ("codec.py", "inv = F32(1.0) / np.maximum(n, FLT_MIN)", "inv = F32(1.0) / np.maximum(n, F32(1e-3))"),
    ("codec.py", "u = y * inv[..., None]", "u = y / n[..., None]"),
    ("codec.py", "code = (u[..., None] >= bnd).sum", "code = (u[..., None] > bnd).sum"),
    ("codec.py", "r = u - cent.astype(F32)[code]", "r = u"),
    ("codec.py", "gamma = np.sqrt(sumsq128(r))", "gamma = np.sqrt(sumsq128(r) / F32(D))"),
    ("codec.py", "t = t + proj[:, j] * r[..., j:j + 1]", "t = t + proj[j, :] * r[..., j:j + 1]"),
    ("codec.py", "bits = t >= 0", "bits = t < 0"),
    ("codec.py", "QJL_CONST = np.sqrt(np.pi / 2.0) / D", "QJL_CONST = np.sqrt(2.0 / np.pi) / D"),
    ("codec.py", 'sq = np.einsum("ij,...j->...i"', 'sq = np.einsum("ji,...j->...i"'),
    ("codec.py", "return n.astype(np.float64) * (dot_c + QJL_CONST", "return (dot_c + QJL_CONST"),
    ("codec.py", "QJL_CONST * gamma.astype(np.float64) * dot_s", "QJL_CONST * dot_s"),
    # Sinkhorn balancing
    ("codec.py", "        rho = np.sqrt(sumsq128(x) / F32(D))\n", "        rho = np.ones(x.shape[0], F32)\n"),
    ("codec.py", "rho = np.where(rho > 0, rho, F32(1.0))", "rho = np.where(rho > 0, rho, F32(0.0))"),
    ("codec.py", "kappa = np.sqrt(s / F32(ntok))", "kappa = np.sqrt(s)"),
    ("codec.py", "x = x / kappa[None, :]", "x = x"),
    ("codec.py", "sigma = sigma * kappa", "sigma = kappa"),
    # cache: append
    ("attention.py", "y = y / sigma.astype(F32)", "y = y"),
    ("attention.py", "self.sigma_v[layer, h] = codec.sinkhorn_sigma(codec.rotate(v_calib[h], self.signs))",
                     "self.sigma_v[layer, h] = codec.sinkhorn_sigma(codec.rotate(k_calib[h], self.signs))"),
    ("attention.py", "if p0 < 0:              # sequence not part of this append\n                continue",
                     "if p0 < -1:\n                continue"),
    ("attention.py", "self.ring_k[layer, b, h, p % W] = k[b, h, t]", "self.ring_k[layer, b, h, t % W] = k[b, h, t]"),
    # cache: decode
    ("attention.py", "heads = range(h * cfg.gqa, (h + 1) * cfg.gqa)",
                     "heads = range(h, cfg.n_q_heads, cfg.n_kv_heads)"),
    ("attention.py", "Lq = max(0, L - W) if W > 0 else L", "Lq = max(0, L - W + 1) if W > 0 else L"),
    ("attention.py", "lq = np.stack([codec.tq3_qjl_dot64(qt[i]", "lq = np.stack([codec.tq3_qjl_dot64(q64[i]"),
    ("attention.py", "kd = kd * self.sigma_k[layer, h].astype(np.float64)", "kd = kd"),
    ("attention.py", "vd = vd * self.sigma_v[layer, h].astype(np.float64)", "vd = vd"),
    ("attention.py", "logits.append(lq * inv_sqrt_d)", "logits.append(lq)"),
    ("attention.py", "logits.append((q64 @ kw.T) * inv_sqrt_d)",
                     "logits.append((qt @ kw.T) * inv_sqrt_d if Lq > 0 else (q64 @ kw.T) * inv_sqrt_d)"),
    ("attention.py", "m = lg.max(axis=1, keepdims=True)", "m = lg.max(axis=1, keepdims=True) * 0 + 50"),
    ("attention.py", "out += codec.unrotate64(p[:, :Lq] @ vd, self.signs)", "out += p[:, :Lq] @ vd"),
    # chunked prefill
    ("attention.py", "lens = np.where(active, p + 1, 0)", "lens = np.where(active, p, 0)"),
    ("attention.py", "p = np.where(active, np.asarray(pos) + t, -1)", "p = np.where(active, np.asarray(pos), -1)"),
    ("attention.py", "out[:, :, t] = cache.decode(layer, q[:, :, t], lens)",
                     "out[:, :, t] = cache.decode(layer, q[:, :, 0], lens)"),
    # block codecs: TBQ blocks and the outlier-channel split
    ("blocks.py", "x = np.stack((a + b, a - b), axis=-2).reshape(lead + (n,))",
                  "x = np.stack((a - b, a + b), axis=-2).reshape(lead + (n,))"),
    ("blocks.py", "return hadamard_n(x * signs) * c_n(x.shape[-1])", "return hadamard_n(x) * c_n(x.shape[-1])"),
    ("blocks.py", "return (hadamard_n(y) * c_n(y.shape[-1])) * signs", "return hadamard_n(y * signs) * c_n(y.shape[-1])"),
    ("blocks.py", "s = (b[..., 0] + b[..., 1]) + (b[..., 2] + b[..., 3])",
                  "s = ((b[..., 0] + b[..., 1]) + b[..., 2]) + b[..., 3]"),
    ("blocks.py", "s = s[..., :m] + s[..., m:2 * m]", "s = s[..., 0:2 * m:2] + s[..., 1:2 * m:2]"),
    ("blocks.py", "cent = (c64 / np.sqrt(float(dim))).astype(F16)", "cent = (c64 / np.sqrt(float(dim + 1))).astype(F16)"),
    ("blocks.py", "return cent, (c32[:-1] + c32[1:]) / F32(2.0)",
                  "return cent, c32[:-1] + (c32[1:] - c32[:-1]) / F32(3.0)"),
    ("blocks.py", "code = (u[..., None] >= bnd).sum(axis=-1)", "code = (u[..., None] > bnd).sum(axis=-1)"),
    ("blocks.py", "u = y * inv[..., None]", "u = y"),
    ("blocks.py", "return norm.astype(F32)[..., None] * cent.astype(F32)[code]", "return cent.astype(F32)[code]"),
    ("blocks.py", "bitarr = ((code[..., None] >> np.arange(bits, dtype=np.uint8)) & 1)",
                  "bitarr = ((code[..., None] >> np.arange(bits - 1, -1, -1, dtype=np.uint8)) & 1)"),
    ("blocks.py", "order = np.lexsort((np.arange(codec.D), -ss))", "order = np.lexsort((-np.arange(codec.D), -ss))"),
    ("blocks.py", "cr, nr = mse_encode(rotate_n(x[..., r], s[SPLIT_N:]), hi_bits - 1)",
                  "cr, nr = mse_encode(rotate_n(x[..., r], s[:SPLIT_N]), hi_bits - 1)"),
    ("blocks.py", "return np.concatenate([_f16_bytes(no), _f16_bytes(nr),", "return np.concatenate([_f16_bytes(nr), _f16_bytes(no),"),
]

# Child interpreter: build the ``oracle`` package from its sources with one replacement applied,
# then run the pins.  Exit status is pytest's.
_CHILD = r"""
import sys, types
import pytest
fn, old, new = sys.argv[1], sys.argv[2], sys.argv[3]
pkg = types.ModuleType("oracle")
pkg.__path__ = []
sys.modules["oracle"] = pkg
for name in ("codec", "attention", "blocks"):
    path = "oracle/%s.py" % name
    src = open(path).read()
    if name + ".py" == fn and old:
        assert src.count(old) == 1, "mutant text must occur once"
        src = src.replace(old, new)
    mod = types.ModuleType("oracle." + name)
    mod.__package__ = "oracle"
    mod.__file__ = path
    sys.modules["oracle." + name] = mod
    setattr(pkg, name, mod)
    exec(compile(src, path, "exec"), mod.__dict__)
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", "-W", "ignore::RuntimeWarning",
                      "tests/test_oracle_pins.py", "tests/test_oracle_blocks.py"]))
"""


def _run(fn, old, new):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-c", _CHILD, fn, old, new], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


@pytest.fixture(scope="module")
def results():
    jobs = [("codec.py", "", "")] + MUTANTS          # first: unchanged, must pass
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        return list(ex.map(lambda m: _run(*m), jobs))


def test_unmutated_oracle_passes_its_pins(results):
    rc, log = results[0]
    assert rc == 0, log[-2000:]


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_mutant_is_caught(results, i):
    fn, old, new = MUTANTS[i]
    with open(os.path.join(ROOT, "oracle", fn)) as f:
        assert f.read().count(old) == 1, "mutant text no longer in the oracle"
    rc, log = results[i + 1]
    assert rc == 1, f"pins did not catch: {fn}: {old!r} -> {new!r}\n{log[-1500:]}"
