"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds random-number generation only -- none of the method's arithmetic -- and is the
one piece of Python that both the CUDA path's callers and the CPU oracle's callers use.  It also
draws the method's own random matrix (the QJL Gaussian projection), which is then passed to both
sides as an input.

Workloads (names are the shapes they stand in for; no dataset or weights are used):
  tiny                : 1 layer, B=1, 4 query / 1 kv head, context 512, fp32 N(0,1), K channels
                        0-3 x10, window 128, Q4G32 K and V, WHT seed 0.
  llama3.2-3b-32k     : 28 layers, 24/8 heads, B=1, context 32768, bf16 N(0,1) with 2% of channels
                        (3 of 128 per layer and kv-head) x8 in K and V, Q4G32, window 128.
  qwen3-4b-kvarn-128k : 36 layers, 32/8 heads, B=1, context 131072, bf16 K/V with per-channel std
                        log-uniform in [0.1, 10], Sinkhorn balancing calibrated on the first 1024
                        tokens, Q4G32, window 128.
  llama3.1-8b-tq-b8-32k: 32 layers, 32/8 heads, B=8 x 32768, bf16 N(0,1) with 4 channels x12,
                        K = TQ3 + QJL, V = Q4G32, window 128.
  llama3.2-3b-32k-k8v4: the llama3.2-3b-32k shape and inputs (same seeds) with keys at 8 bits
                        (Q8G32) and values at 4 bits (Q4G32): the asymmetric K/V split.
  dense27b-ragged-b32 : 62 layers (one allocated and timed), 32/16 heads, B=32 with lengths
                        uniform in [1024, 65536] (numpy default_rng(7)), 64-token pages, bf16
                        N(0,1) with 1% of channels (1 of 128) x10 in K and V, Q4G32, window 128;
                        bulk append of an 8192-token prefill chunk per sequence.
"""

from __future__ import annotations

import math

import numpy as np
import torch

D = 128

WORKLOADS = {
    "tiny": dict(index=1, n_layers=1, batch=1, n_q_heads=4, n_kv_heads=1, ctx=512, window=128,
                 k_format="q4g32", v_format="q4g32", sinkhorn=False, in_dtype="f32", wht_seed=0,
                 outlier_channels=(0, 1, 2, 3), outlier_scale=10.0, outliers_in_v=False),
    "llama3.2-3b-32k": dict(index=2, n_layers=28, batch=1, n_q_heads=24, n_kv_heads=8, ctx=32768,
                            window=128, k_format="q4g32", v_format="q4g32", sinkhorn=False,
                            in_dtype="bf16", wht_seed=0, outlier_frac=0.02, outlier_scale=8.0,
                            outliers_in_v=True),
    "qwen3-4b-kvarn-128k": dict(index=3, n_layers=36, batch=1, n_q_heads=32, n_kv_heads=8,
                                ctx=131072, window=128, k_format="q4g32", v_format="q4g32",
                                sinkhorn=True, calib_tokens=1024, in_dtype="bf16", wht_seed=0,
                                channel_std_loguniform=(0.1, 10.0)),
    "llama3.1-8b-tq-b8-32k": dict(index=4, n_layers=32, batch=8, n_q_heads=32, n_kv_heads=8,
                                  ctx=32768, window=128, k_format="tq3_qjl", v_format="q4g32",
                                  sinkhorn=False, in_dtype="bf16", wht_seed=0, qjl_seed=4242,
                                  outlier_count=4, outlier_scale=12.0, outliers_in_v=True),
    # same index as llama3.2-3b-32k: the same seeded K, V and q, only the key format differs
    "llama3.2-3b-32k-k8v4": dict(index=2, n_layers=28, batch=1, n_q_heads=24, n_kv_heads=8, ctx=32768,
                                 window=128, k_format="q8g32", v_format="q4g32", sinkhorn=False,
                                 in_dtype="bf16", wht_seed=0, outlier_frac=0.02, outlier_scale=8.0,
                                 outliers_in_v=True),
    "dense27b-ragged-b32": dict(index=5, n_layers=62, alloc_layers=1, batch=32, n_q_heads=32,
                                n_kv_heads=16, ctx_range=(1024, 65536), len_seed=7, window=128,
                                page_tokens=64, k_format="q4g32", v_format="q4g32", sinkhorn=False,
                                in_dtype="bf16", wht_seed=0, outlier_frac=0.01,
                                outlier_scale=10.0, outliers_in_v=True, prefill_chunk=8192),
}


def ragged_lengths(lo: int = 1024, hi: int = 65536, n: int = 32, seed: int = 7) -> np.ndarray:
    """Sequence lengths uniform in [lo, hi] (inclusive) from numpy's default_rng(seed)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, n).astype(np.int32)


def qjl_projection(seed: int) -> np.ndarray:
    """The 128 x 128 Gaussian projection of the QJL sketch: i.i.d. N(0, 1), float32, row-major."""
    return np.random.default_rng(seed).standard_normal((D, D)).astype(np.float32)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def n_outliers(w: dict) -> int:
    if "outlier_channels" in w:
        return len(w["outlier_channels"])
    if "outlier_count" in w:
        return int(w["outlier_count"])
    if "outlier_frac" in w:
        return int(round(w["outlier_frac"] * D))
    return 0


def layer_seed(w: dict, layer: int, stream: int = 0) -> int:
    return 1000 * w["index"] + layer + 100003 * stream


def channel_scales(w: dict, layer: int, n_kv_heads: int, which: str, device="cpu") -> torch.Tensor:
    """Per-(kv-head, channel) multiplier of the unit-variance draws for K ('k') or V ('v')."""
    sc = torch.ones(n_kv_heads, D, dtype=torch.float32)
    if "channel_std_loguniform" in w:
        lo, hi = w["channel_std_loguniform"]
        g = _gen(layer_seed(w, layer, 7 if which == "k" else 8), "cpu")
        u = torch.rand(n_kv_heads, D, generator=g, dtype=torch.float64)
        sc = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).float()
    else:
        n_out = n_outliers(w)
        if n_out and (which == "k" or w.get("outliers_in_v", False)):
            if "outlier_channels" in w:
                for h in range(n_kv_heads):
                    sc[h, list(w["outlier_channels"])] = w["outlier_scale"]
            else:
                g = _gen(layer_seed(w, layer, 9), "cpu")
                for h in range(n_kv_heads):
                    ch = torch.randperm(D, generator=g)[:n_out]
                    sc[h, ch] = w["outlier_scale"]
    return sc.to(device)


def kv_tokens(w: dict, layer: int, batch: int, n_kv_heads: int, t0: int, T: int, device="cpu",
              dtype=None):
    """K and V for positions [t0, t0+T) of every sequence: ([B][H][T][128], [B][H][T][128]).

    Drawn per (layer, position block) so that any slice of the context can be regenerated; the
    block size is 4096 tokens and each block has its own generator stream.
    """
    dt = dtype or (torch.float32 if w["in_dtype"] == "f32" else torch.bfloat16)
    sk = channel_scales(w, layer, n_kv_heads, "k", device)
    sv = channel_scales(w, layer, n_kv_heads, "v", device)
    BLK = 4096
    ks, vs = [], []
    t = t0
    while t < t0 + T:
        blk = t // BLK
        lo = t - blk * BLK
        n = min(BLK - lo, t0 + T - t)
        g = _gen(layer_seed(w, layer, 1000 + blk), device)
        kb = torch.randn(batch, n_kv_heads, BLK, D, generator=g, device=device, dtype=torch.float32)
        vb = torch.randn(batch, n_kv_heads, BLK, D, generator=g, device=device, dtype=torch.float32)
        ks.append(kb[:, :, lo:lo + n])
        vs.append(vb[:, :, lo:lo + n])
        t += n
    k = torch.cat(ks, dim=2) * sk[None, :, None, :]
    v = torch.cat(vs, dim=2) * sv[None, :, None, :]
    return k.to(dt).contiguous(), v.to(dt).contiguous()


def chunk_queries(w: dict, layer: int, batch: int, n_q_heads: int, T: int, device="cpu",
                  dtype=None) -> torch.Tensor:
    """Queries of a T-token prefill chunk [B][Hq][T][128], N(0, 1), in one draw."""
    dt = dtype or (torch.float32 if w["in_dtype"] == "f32" else torch.bfloat16)
    g = _gen(layer_seed(w, layer, 60000), device)
    return torch.randn(batch, n_q_heads, T, D, generator=g, device=device,
                       dtype=torch.float32).to(dt).contiguous()


def queries(w: dict, layer: int, batch: int, n_q_heads: int, step: int = 0, device="cpu",
            dtype=None) -> torch.Tensor:
    """Decode queries [B][Hq][128], N(0, 1)."""
    dt = dtype or (torch.float32 if w["in_dtype"] == "f32" else torch.bfloat16)
    g = _gen(layer_seed(w, layer, 50000 + step), device)
    return torch.randn(batch, n_q_heads, D, generator=g, device=device,
                       dtype=torch.float32).to(dt).contiguous()
