"""Shared test plumbing: build a GPU cache and the oracle cache from the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

from kv_cache_quantization_append_gb300 import QuantKVCache, lib, synth
from oracle import attention

from . import layout

FMT = dict(lib.K_FORMATS)
OFMT = {"q4g32": attention.Q4G32, "tq3_qjl": attention.TQ3_QJL, "q8g32": attention.Q8G32}


def make_pair(n_layers, n_kv, n_q, max_batch, max_seq_len, window=128, k_format="q4g32",
              sinkhorn=False, in_dtype="bf16", seed=0, n_pages=0, block_table=None, qjl_seed=None):
    """(gpu QuantKVCache, oracle cache, projection or None) for one configuration."""
    proj = synth.qjl_projection(qjl_seed if qjl_seed is not None else 4242) if k_format == "tq3_qjl" else None
    cfg = lib.make_config(n_layers, n_kv, n_q, max_batch, max_seq_len, window=window, n_pages=n_pages,
                          k_format=FMT[k_format], sinkhorn=sinkhorn,
                          in_dtype=lib.KVQ_IN_BF16 if in_dtype == "bf16" else lib.KVQ_IN_F32, seed=seed)
    bt = None if block_table is None else torch.as_tensor(block_table, dtype=torch.int32, device="cuda").contiguous()
    gpu = QuantKVCache(cfg, "cuda", bt, proj)
    ocfg = attention.OracleConfig(n_layers=n_layers, n_kv_heads=n_kv, n_q_heads=n_q, max_batch=max_batch,
                                  max_seq_len=max_seq_len, window=window, k_format=OFMT[k_format],
                                  sinkhorn=sinkhorn, seed=seed)
    ora = attention.OracleCache(ocfg, proj)
    return gpu, ora, proj


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def compare_codes(gpu: QuantKVCache, ora: attention.OracleCache, layer: int, b: int, h: int, n: int,
                  block_table=None):
    """Bit-exact comparison of every stored field of positions [0, n)."""
    got = layout.read_unit(gpu.buffer, gpu.cfg, layer, b, h, n, block_table)
    if ora.cfg.k_format == attention.TQ3_QJL:
        want = {"k_code": ora.k["code"], "k_bits": ora.k["bits"], "k_norm": ora.k["norm"], "k_gamma": ora.k["gamma"]}
    elif ora.cfg.k_format == attention.Q8G32:
        want = {"k_code": ora.k["code"], "k_scale": ora.k["scale"]}
    else:
        want = {"k_code": ora.k["code"], "k_scale": ora.k["scale"], "k_zero": ora.k["zero"]}
    want.update({"v_code": ora.v["code"], "v_scale": ora.v["scale"], "v_zero": ora.v["zero"]})
    for name, arr in want.items():
        w = arr[layer, b, h, :n]
        g = got[name]
        if w.dtype == np.float16:
            w, g = w.view(np.uint16), g.view(np.uint16)
        bad = np.argwhere(w != g)
        assert bad.size == 0, f"{name} differs at {bad[:5].tolist()} (layer {layer}, seq {b}, head {h})"


def compare_ring(gpu, ora, layer, b, h, L):
    W = ora.cfg.window
    if W == 0 or L == 0:
        return
    gk, gv = layout.read_ring(gpu.buffer, gpu.cfg, layer, b, h)
    slots = np.arange(max(0, L - W), L) % W
    assert np.array_equal(gk[slots].view(np.uint32), ora.ring_k[layer, b, h, slots].view(np.uint32))
    assert np.array_equal(gv[slots].view(np.uint32), ora.ring_v[layer, b, h, slots].view(np.uint32))


def assert_attention_close(out_gpu: np.ndarray, out_ora: np.ndarray, tol: float = 2e-3):
    """max |gpu - oracle| <= tol * max |oracle| (the float64 oracle on the same dequantised values)."""
    ref = np.max(np.abs(out_ora))
    err = np.max(np.abs(out_gpu.astype(np.float64) - out_ora))
    assert err <= tol * ref + 1e-30, f"max abs err {err:.3e} > {tol} * {ref:.3e}"
    return err / max(ref, 1e-30)
