"""Oracle cache model and float64 decode attention (test infrastructure only).

The cache keeps, for every (layer, sequence, kv-head):
  * a quantised record for EVERY appended token (quantise-on-append), and
  * a ring of the ``window`` most recent tokens in raw float32 (slot = position mod window).
Decode attends to positions [0, L - window) through the quantised records (in rotated space) and
to [L - window, L) through the raw ring, with one softmax over all L tokens.

[QC] "how it works": 128 FP32 tokens plus 4-bit for everything else; the same 128-token window
at every context length.  [QC] v3.2 note: a batched write of T tokens equals T single-token
writes bit for bit -- holds here because each record depends on its own token only.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import codec

F32 = np.float32
Q4G32 = "q4g32"
Q8G32 = "q8g32"
TQ3_QJL = "tq3_qjl"
REC_BYTES = {Q4G32: 64 + 8 + 8,          # 128 nibbles, 4 fp16 scales, 4 fp16 zeros
             Q8G32: 128 + 8,             # 128 signed bytes, 4 fp16 scales
             TQ3_QJL: 48 + 16 + 2 + 2}   # 128 x 3-bit codes, 128 sign bits, fp16 norm, fp16 gamma


@dataclass
class OracleConfig:
    n_layers: int
    n_kv_heads: int
    n_q_heads: int
    max_batch: int
    max_seq_len: int
    window: int = 128
    k_format: str = Q4G32
    v_format: str = Q4G32
    sinkhorn: bool = False
    seed: int = 0

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads


def payload_bytes_per_token_head(cfg: OracleConfig) -> int:
    """Bytes the quantised store holds per token and kv-head (K record + V record)."""
    return REC_BYTES[cfg.k_format] + REC_BYTES[cfg.v_format]


def window_bytes(cfg: OracleConfig) -> int:
    """Raw float32 K and V of the window, per (layer, sequence, kv-head) summed over all."""
    return cfg.n_layers * cfg.max_batch * cfg.n_kv_heads * cfg.window * codec.D * 4 * 2


def fp32_kv_bytes(n_layers: int, n_kv_heads: int, ctx: int) -> int:
    """Unquantised float32 K+V bytes of one sequence (the FP32 baseline row of [QC]'s table)."""
    return 2 * n_layers * n_kv_heads * codec.D * 4 * ctx


class OracleCache:
    """Plain per-position arrays; slow and obviously indexed."""

    def __init__(self, cfg: OracleConfig, qjl_proj: np.ndarray | None = None):
        self.cfg = cfg
        self.signs = codec.wht_signs(cfg.seed)
        L, B, H, P = cfg.n_layers, cfg.max_batch, cfg.n_kv_heads, cfg.max_seq_len
        self.sigma_k = np.ones((L, H, codec.D), np.float16)
        self.sigma_v = np.ones((L, H, codec.D), np.float16)
        self.proj = None if qjl_proj is None else np.asarray(qjl_proj, F32)
        if cfg.k_format == TQ3_QJL:
            assert self.proj is not None, "TQ3_QJL keys need the projection matrix"
            self.k = dict(code=np.zeros((L, B, H, P, codec.D), np.uint8),
                          bits=np.zeros((L, B, H, P, codec.D), bool),
                          norm=np.zeros((L, B, H, P), np.float16),
                          gamma=np.zeros((L, B, H, P), np.float16))
        elif cfg.k_format == Q8G32:
            self.k = dict(code=np.zeros((L, B, H, P, codec.D), np.int8),
                          scale=np.zeros((L, B, H, P, 4), np.float16))
        else:
            self.k = dict(code=np.zeros((L, B, H, P, codec.D), np.uint8),
                          scale=np.zeros((L, B, H, P, 4), np.float16),
                          zero=np.zeros((L, B, H, P, 4), np.float16))
        self.v = dict(code=np.zeros((L, B, H, P, codec.D), np.uint8),
                      scale=np.zeros((L, B, H, P, 4), np.float16),
                      zero=np.zeros((L, B, H, P, 4), np.float16))
        W = max(cfg.window, 1)
        self.ring_k = np.zeros((L, B, H, W, codec.D), F32)
        self.ring_v = np.zeros((L, B, H, W, codec.D), F32)

    # ---------------------------------------------------------------- calibration (KVarN)
    def calibrate(self, layer: int, k_calib: np.ndarray, v_calib: np.ndarray):
        """sigma for each kv-head from a raw calibration block [H][n][128] of K and of V.

        The block is rotated first ([KV]: Walsh-Hadamard, then Sinkhorn balancing).
        """
        for h in range(self.cfg.n_kv_heads):
            self.sigma_k[layer, h] = codec.sinkhorn_sigma(codec.rotate(k_calib[h], self.signs))
            self.sigma_v[layer, h] = codec.sinkhorn_sigma(codec.rotate(v_calib[h], self.signs))

    # ---------------------------------------------------------------- append
    def _balanced(self, x: np.ndarray, sigma: np.ndarray | None):
        y = codec.rotate(x, self.signs)
        if sigma is not None:
            y = y / sigma.astype(F32)          # balanced value y / sigma (float32 division)
        return y

    def _encode_q4(self, x: np.ndarray, sigma: np.ndarray | None):
        return codec.q4g32_encode(self._balanced(x, sigma))

    def append(self, layer: int, k: np.ndarray, v: np.ndarray, pos: np.ndarray):
        """Append T tokens per sequence: k, v [B][H][T][128] float32; pos [B] first position."""
        cfg = self.cfg
        B, H, T, _ = k.shape
        for b in range(B):
            p0 = int(pos[b])
            if p0 < 0:              # sequence not part of this append
                continue
            assert p0 + T <= cfg.max_seq_len
            sl = slice(p0, p0 + T)
            for h in range(H):
                sk = self.sigma_k[layer, h] if cfg.sinkhorn else None
                sv = self.sigma_v[layer, h] if cfg.sinkhorn else None
                if cfg.k_format == TQ3_QJL:
                    y = codec.rotate(k[b, h], self.signs)
                    c, bits, n, g = codec.tq3_qjl_encode(y, self.proj)
                    self.k["code"][layer, b, h, sl] = c
                    self.k["bits"][layer, b, h, sl] = bits
                    self.k["norm"][layer, b, h, sl] = n
                    self.k["gamma"][layer, b, h, sl] = g
                elif cfg.k_format == Q8G32:
                    c, s = codec.q8g32_encode(self._balanced(k[b, h], sk))
                    self.k["code"][layer, b, h, sl] = c
                    self.k["scale"][layer, b, h, sl] = s
                else:
                    c, s, z = self._encode_q4(k[b, h], sk)
                    self.k["code"][layer, b, h, sl] = c
                    self.k["scale"][layer, b, h, sl] = s
                    self.k["zero"][layer, b, h, sl] = z
                c, s, z = self._encode_q4(v[b, h], sv)
                self.v["code"][layer, b, h, sl] = c
                self.v["scale"][layer, b, h, sl] = s
                self.v["zero"][layer, b, h, sl] = z
                W = cfg.window
                if W > 0:
                    for t in range(max(0, T - W), T):
                        p = p0 + t
                        self.ring_k[layer, b, h, p % W] = k[b, h, t]
                        self.ring_v[layer, b, h, p % W] = v[b, h, t]

    # ---------------------------------------------------------------- decode
    def decode(self, layer: int, q: np.ndarray, seq_lens: np.ndarray) -> np.ndarray:
        """One decode step for every sequence: q [B][Hq][128] float32 -> out [B][Hq][128] float64."""
        cfg = self.cfg
        B = q.shape[0]
        out = np.zeros((B, cfg.n_q_heads, codec.D), np.float64)
        for b in range(B):
            for h in range(cfg.n_kv_heads):
                heads = range(h * cfg.gqa, (h + 1) * cfg.gqa)
                out[b, heads.start:heads.stop] = self.decode_unit(layer, b, h, q[b, heads.start:heads.stop],
                                                                  int(seq_lens[b]))
        return out

    def decode_unit(self, layer: int, b: int, h: int, qg: np.ndarray, L: int) -> np.ndarray:
        """Attention of the g query heads ``qg`` [g][128] over sequence b, kv-head h, length L."""
        cfg = self.cfg
        D = codec.D
        g = qg.shape[0]
        if L <= 0:
            return np.zeros((g, D))
        W = cfg.window
        Lq = max(0, L - W) if W > 0 else L
        q64 = np.asarray(qg, np.float64)
        inv_sqrt_d = 1.0 / np.sqrt(float(D))
        logits = []
        # quantised part, rotated space
        if Lq > 0:
            qt = codec.rotate64(q64, self.signs)                                  # [g][128]
            if cfg.k_format == TQ3_QJL:
                kk = {n: a[layer, b, h, :Lq] for n, a in self.k.items()}
                lq = np.stack([codec.tq3_qjl_dot64(qt[i], kk["code"], kk["bits"], kk["norm"],
                                                   kk["gamma"], self.proj) for i in range(g)])
            else:
                if cfg.k_format == Q8G32:
                    kd = codec.q8g32_decode(self.k["code"][layer, b, h, :Lq],
                                            self.k["scale"][layer, b, h, :Lq]).astype(np.float64)
                else:
                    kd = codec.q4g32_decode(self.k["code"][layer, b, h, :Lq], self.k["scale"][layer, b, h, :Lq],
                                            self.k["zero"][layer, b, h, :Lq]).astype(np.float64)
                if cfg.sinkhorn:
                    kd = kd * self.sigma_k[layer, h].astype(np.float64)
                lq = qt @ kd.T                                                    # [g][Lq]
            logits.append(lq * inv_sqrt_d)
            vd = codec.q4g32_decode(self.v["code"][layer, b, h, :Lq], self.v["scale"][layer, b, h, :Lq],
                                    self.v["zero"][layer, b, h, :Lq]).astype(np.float64)
            if cfg.sinkhorn:
                vd = vd * self.sigma_v[layer, h].astype(np.float64)
        # window part, raw values
        if L > Lq:
            slots = np.arange(Lq, L) % W
            kw = self.ring_k[layer, b, h, slots].astype(np.float64)
            vw = self.ring_v[layer, b, h, slots].astype(np.float64)
            logits.append((q64 @ kw.T) * inv_sqrt_d)
        lg = np.concatenate(logits, axis=1)
        m = lg.max(axis=1, keepdims=True)
        p = np.exp(lg - m)
        p /= p.sum(axis=1, keepdims=True)
        out = np.zeros((g, D))
        if Lq > 0:
            out += codec.unrotate64(p[:, :Lq] @ vd, self.signs)
        if L > Lq:
            out += p[:, Lq:] @ vw
        return out


def prefill(cache: "OracleCache", layer: int, k: np.ndarray, v: np.ndarray, q: np.ndarray,
            pos: np.ndarray) -> np.ndarray:
    """Chunked prefill over the compressed cache: T new tokens per sequence with their queries.

    [QC] v3.2 note: a batched prefill writes exactly what T single-token steps write.  Reading for
    the attention of the chunk: also exactly what T single-token steps compute, so query t of
    sequence b attends causally to positions [0, pos[b] + t] with the window of that step (the
    newest ``window`` of those positions raw, the rest through their quantised records).  Written as
    that definition: append token t, then decode at L = pos[b] + t + 1.

    k, v [B][H][T][128]; q [B][Hq][T][128]; pos [B] (pos[b] < 0: sequence b takes no part, its
    outputs are zero).  Returns out [B][Hq][T][128] float64.
    """
    B, _, T, _ = k.shape
    out = np.zeros((B, cache.cfg.n_q_heads, T, codec.D), np.float64)
    active = np.asarray(pos) >= 0
    for t in range(T):
        p = np.where(active, np.asarray(pos) + t, -1)
        cache.append(layer, k[:, :, t:t + 1], v[:, :, t:t + 1], p)
        lens = np.where(active, p + 1, 0)
        out[:, :, t] = cache.decode(layer, q[:, :, t], lens)
    return out


def plain_attention64(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Textbook softmax(q k^T / sqrt(d)) v in float64 via scipy's softmax; q [g][d], k, v [L][d]."""
    from scipy.special import softmax

    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    return softmax(q @ k.T / np.sqrt(q.shape[-1]), axis=-1) @ v
