"""Quantized KV cache for GB300: append (rotate, balance, 4-bit / 3-bit+QJL pack) and decode
attention over the compressed cache, as hand-written sm_103a CUDA behind a C ABI (include/kvq.h).

``lib`` is the thin ctypes binding (same names as the C entry points).  ``QuantKVCache`` only
owns the torch allocations a caller needs (cache buffer, block table, scratch) and forwards to it.
"""

from __future__ import annotations

import torch

from . import lib
from .lib import (KVQ_IN_BF16, KVQ_IN_F32, KVQ_Q4G32, KVQ_Q8G32, KVQ_TQ3_QJL, kv_cache_bytes,  # noqa: F401
                  kv_cache_init,
                  kv_calibrate, kv_calibrate_scratch_bytes, kv_decode_attention,
                  kv_decode_scratch_bytes, kv_quant_append, kv_status, kv_strerror, make_config)


class QuantKVCache:
    """Device buffers of one cache, allocated with torch; all work runs in libkvq's kernels."""

    def __init__(self, cfg: lib.kvq_config, device="cuda", block_table: torch.Tensor | None = None,
                 qjl_proj=None):
        self.cfg = cfg
        nbytes = kv_cache_bytes(cfg)
        if nbytes == 0:
            raise lib.KVQError("unsupported cache configuration")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.block_table = block_table
        self.handle = kv_cache_init(cfg, self.buffer, block_table, qjl_proj)
        self._scratch = {}

    def scratch(self, layer: int, batch: int) -> torch.Tensor:
        """Decode scratch (uninitialised), kept per (layer-mode, batch) and reused across calls."""
        key = (layer == -1, batch)
        need = kv_decode_scratch_bytes(self.handle, layer, batch)
        t = self._scratch.get(key)
        if t is None or t.numel() < need:
            t = torch.empty(need, dtype=torch.uint8, device=self.buffer.device)
            self._scratch[key] = t
        return t

    def append(self, layer: int, k: torch.Tensor, v: torch.Tensor, pos: torch.Tensor, stream=None):
        kv_quant_append(self.handle, layer, k, v, pos, stream)

    def calibrate(self, layer: int, k_calib: torch.Tensor, v_calib: torch.Tensor, stream=None):
        need = kv_calibrate_scratch_bytes(self.handle, layer, k_calib.shape[-2])
        work = torch.empty(need, dtype=torch.uint8, device=self.buffer.device)
        kv_calibrate(self.handle, layer, k_calib, v_calib, work, stream)

    def decode(self, layer: int, q: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        kv_decode_attention(self.handle, layer, q, out, seq_lens, self.scratch(layer, q.shape[-3]), stream)
        return out

    def prefill(self, layer: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor, pos: torch.Tensor,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Append the chunk (k, v at pos) and return its queries' attention [L?][B][Hq][T][128]."""
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        need = lib.kv_prefill_scratch_bytes(self.handle, layer, q.shape[-4])
        key = ("prefill", layer == -1, q.shape[-4])
        t = self._scratch.get(key)
        if t is None or t.numel() < need:
            t = torch.empty(need, dtype=torch.uint8, device=self.buffer.device)
            self._scratch[key] = t
        lib.kv_prefill_attention(self.handle, layer, k, v, q, out, pos, t, stream)
        return out

    def status(self) -> int:
        return kv_status(self.handle)
