"""ctypes binding of libkvq (the C ABI in include/kvq.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does nothing but check tensor
properties, take ``data_ptr()`` and the current CUDA stream, and translate status codes into
exceptions.  All computation happens in the library's CUDA kernels; there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libkvq.so")

KVQ_Q4G32 = 1
KVQ_TQ3_QJL = 3
KVQ_Q8G32 = 4
# the key formats by the names the workloads and the oracle use
K_FORMATS = {"q4g32": KVQ_Q4G32, "tq3_qjl": KVQ_TQ3_QJL, "q8g32": KVQ_Q8G32}
KVQ_IN_F32 = 0
KVQ_IN_BF16 = 1

DEV_BAD_PAGE = 1
DEV_POS_RANGE = 2
DEV_SEQLEN_RANGE = 4
DEV_TIMEOUT = 8

EXPORTS = ("kv_cache_bytes", "kv_cache_init", "kv_calibrate_scratch_bytes", "kv_calibrate",
           "kv_quant_append", "kv_decode_scratch_bytes", "kv_decode_attention",
           "kv_decode_attention_noalloc", "kv_prefill_scratch_bytes", "kv_prefill_attention",
           "kv_tbq_block_bytes", "kv_tbq_encode", "kv_tbq_decode", "kv_split_record_bytes",
           "kv_split_outliers", "kv_split_encode", "kv_split_decode", "kv_status", "kv_set_wait_limit_ns",
           "kv_strerror")
NOALLOC_SCRATCH_MAX = 32 * 1024 * 1024


class kvq_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("window", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("n_pages", ctypes.c_int32), ("k_format", ctypes.c_int32),
                ("v_format", ctypes.c_int32), ("sinkhorn", ctypes.c_int32),
                ("group", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("seed", ctypes.c_uint64)]


class kvq_cache(ctypes.Structure):
    _fields_ = [("cfg", kvq_config), ("dev", ctypes.c_void_p), ("bytes", ctypes.c_uint64),
                ("block_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int32),
                ("n_pages", ctypes.c_int32), ("device", ctypes.c_int32), ("magic", ctypes.c_uint32)]


class KVQError(RuntimeError):
    pass


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so; raises if it has not been built (there is no CPU fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise KVQError(f"libkvq.so not built ({path}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I32, SZ, U32P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
    cfgp, cachep = ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_cache)
    sig = {
        "kv_cache_bytes": (SZ, [cfgp]),
        "kv_cache_init": (ctypes.c_int, [cachep, cfgp, P, SZ, P, P, P]),
        "kv_calibrate_scratch_bytes": (SZ, [cachep, I32, I32]),
        "kv_calibrate": (ctypes.c_int, [cachep, I32, P, P, I32, P, SZ, P]),
        "kv_quant_append": (ctypes.c_int, [cachep, I32, P, P, P, I32, I32, P]),
        "kv_decode_scratch_bytes": (SZ, [cachep, I32, I32]),
        "kv_decode_attention": (ctypes.c_int, [cachep, I32, P, P, P, I32, P, SZ, P]),
        "kv_decode_attention_noalloc": (ctypes.c_int, [cachep, I32, P, P, P, I32, P]),
        "kv_prefill_scratch_bytes": (SZ, [cachep, I32, I32]),
        "kv_prefill_attention": (ctypes.c_int, [cachep, I32, P, P, P, P, P, I32, I32, P, SZ, P]),
        "kv_tbq_block_bytes": (SZ, [I32]),
        "kv_tbq_encode": (ctypes.c_int, [I32, ctypes.c_uint64, P, I32, ctypes.c_int64, P, P]),
        "kv_tbq_decode": (ctypes.c_int, [I32, ctypes.c_uint64, P, ctypes.c_int64, P, P]),
        "kv_split_record_bytes": (SZ, [I32]),
        "kv_split_outliers": (ctypes.c_int, [P, I32, I32, I32, P, P]),
        "kv_split_encode": (ctypes.c_int, [I32, ctypes.c_uint64, P, I32, P, I32, ctypes.c_int64, P, P]),
        "kv_split_decode": (ctypes.c_int, [I32, ctypes.c_uint64, P, I32, P, ctypes.c_int64, P, P]),
        "kv_status": (ctypes.c_int, [cachep, U32P, P]),
        "kv_set_wait_limit_ns": (ctypes.c_int, [ctypes.c_uint64]),
        "kv_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        raise KVQError(f"libkvq: {load().kv_strerror(rc).decode()} (code {rc})")


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise KVQError("device tensor expected")
    if not t.is_contiguous():
        raise KVQError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _check_in_dtype(cache: kvq_cache, *tensors: torch.Tensor):
    """k, v, q and calibration blocks must have the cache's input dtype (cfg.in_dtype)."""
    want = torch.bfloat16 if cache.cfg.in_dtype == KVQ_IN_BF16 else torch.float32
    for t in tensors:
        if t.dtype != want:
            raise KVQError(f"input dtype {t.dtype} does not match the cache's in_dtype ({want})")


def _layers_in_call(cache: kvq_cache, layer: int) -> int:
    return cache.cfg.n_layers if layer == -1 else 1


def _check_shape(name: str, t: torch.Tensor, want: tuple):
    """The library reads and writes whole rows of these shapes from the bare pointer; a tensor of
    another size would be read or written past its end, which the C ABI cannot see."""
    if tuple(t.shape) != tuple(want):
        raise KVQError(f"{name} has shape {tuple(t.shape)}, expected {tuple(want)}")


def _check_decode_shapes(cache: kvq_cache, layer: int, q: torch.Tensor, out: torch.Tensor,
                         seq_lens: torch.Tensor) -> int:
    """q and out [L?][B][Hq][128] (the layer axis present iff layer == -1), seq_lens [B]; returns B."""
    if q.dim() not in (3, 4) or q.dim() != (4 if layer == -1 else 3):
        raise KVQError(f"q must be {'[L][B][Hq][128]' if layer == -1 else '[B][Hq][128]'}, got {tuple(q.shape)}")
    B = q.shape[-3]
    lead = (_layers_in_call(cache, layer),) if layer == -1 else ()
    _check_shape("q", q, lead + (B, cache.cfg.n_q_heads, 128))
    _check_shape("out", out, tuple(q.shape))
    _check_shape("seq_lens", seq_lens, (B,))
    return B


def _check_append_shapes(cache: kvq_cache, layer: int, k: torch.Tensor, v: torch.Tensor,
                         pos: torch.Tensor) -> tuple:
    """k and v [L?][B][Hkv][T][128] (the layer axis present iff layer == -1), pos [B]; returns (B, T)."""
    if k.dim() != (5 if layer == -1 else 4):
        raise KVQError(f"k must be {'[L][B][Hkv][T][128]' if layer == -1 else '[B][Hkv][T][128]'}, "
                       f"got {tuple(k.shape)}")
    B, T = k.shape[-4], k.shape[-2]
    lead = (_layers_in_call(cache, layer),) if layer == -1 else ()
    _check_shape("k", k, lead + (B, cache.cfg.n_kv_heads, T, 128))
    _check_shape("v", v, tuple(k.shape))
    _check_shape("pos", pos, (B,))
    return B, T


def make_config(n_layers, n_kv_heads, n_q_heads, max_batch, max_seq_len, window=128, n_pages=0,
                k_format=KVQ_Q4G32, v_format=KVQ_Q4G32, sinkhorn=False, in_dtype=KVQ_IN_BF16,
                seed=0) -> kvq_config:
    return kvq_config(n_layers, n_kv_heads, n_q_heads, 128, max_batch, max_seq_len, window, 64,
                      n_pages, k_format, v_format, int(bool(sinkhorn)), 32, in_dtype, seed)


def kv_cache_bytes(cfg: kvq_config) -> int:
    return int(load().kv_cache_bytes(ctypes.byref(cfg)))


def kv_cache_init(cfg: kvq_config, dev_mem: torch.Tensor, block_table: torch.Tensor | None = None,
                  qjl_proj: np.ndarray | None = None, stream=None) -> kvq_cache:
    cache = kvq_cache()
    proj = None
    if qjl_proj is not None:
        proj = np.ascontiguousarray(qjl_proj, dtype=np.float32)
    pp = ctypes.c_void_p(proj.ctypes.data) if proj is not None else ctypes.c_void_p(0)
    _check(load().kv_cache_init(ctypes.byref(cache), ctypes.byref(cfg), _ptr(dev_mem),
                                dev_mem.numel() * dev_mem.element_size(), _ptr(block_table), pp,
                                _stream(stream)))
    return cache


def kv_calibrate_scratch_bytes(cache: kvq_cache, layer: int, n_tokens: int) -> int:
    return int(load().kv_calibrate_scratch_bytes(ctypes.byref(cache), layer, n_tokens))


def kv_calibrate(cache: kvq_cache, layer: int, k_calib: torch.Tensor, v_calib: torch.Tensor,
                 scratch: torch.Tensor, stream=None):
    _check_in_dtype(cache, k_calib, v_calib)
    n_tokens = k_calib.shape[-2]
    lead = (_layers_in_call(cache, layer),) if layer == -1 else ()
    _check_shape("k_calib", k_calib, lead + (cache.cfg.n_kv_heads, n_tokens, 128))
    _check_shape("v_calib", v_calib, tuple(k_calib.shape))
    _check(load().kv_calibrate(ctypes.byref(cache), layer, _ptr(k_calib), _ptr(v_calib), n_tokens,
                               _ptr(scratch), scratch.numel() * scratch.element_size(),
                               _stream(stream)))


def kv_quant_append(cache: kvq_cache, layer: int, k: torch.Tensor, v: torch.Tensor,
                    pos: torch.Tensor, stream=None):
    """k, v: [L?][B][Hkv][T][128]; pos: int32 [B] on the device."""
    if pos.dtype != torch.int32:
        raise KVQError("pos must be int32")
    _check_in_dtype(cache, k, v)
    B, T = _check_append_shapes(cache, layer, k, v, pos)
    _check(load().kv_quant_append(ctypes.byref(cache), layer, _ptr(k), _ptr(v), _ptr(pos), B, T,
                                  _stream(stream)))


def kv_decode_scratch_bytes(cache: kvq_cache, layer: int, batch: int) -> int:
    return int(load().kv_decode_scratch_bytes(ctypes.byref(cache), layer, batch))


def kv_decode_attention(cache: kvq_cache, layer: int, q: torch.Tensor, out: torch.Tensor,
                        seq_lens: torch.Tensor, scratch: torch.Tensor, stream=None):
    """q: [L?][B][Hq][128]; out: float32 like q; seq_lens: int32 [B]; scratch: device bytes (any
    contents), at least kv_decode_scratch_bytes."""
    if seq_lens.dtype != torch.int32 or out.dtype != torch.float32:
        raise KVQError("seq_lens must be int32 and out float32")
    _check_in_dtype(cache, q)
    B = _check_decode_shapes(cache, layer, q, out, seq_lens)
    _check(load().kv_decode_attention(ctypes.byref(cache), layer, _ptr(q), _ptr(out), _ptr(seq_lens),
                                      B, _ptr(scratch), scratch.numel() * scratch.element_size(),
                                      _stream(stream)))


def kv_decode_attention_noalloc(cache: kvq_cache, layer: int, q: torch.Tensor, out: torch.Tensor,
                                seq_lens: torch.Tensor, stream=None):
    """Decode without a caller scratch buffer: the library's own fixed device array is used (for
    callers that cannot allocate).  Same shapes as kv_decode_attention."""
    if seq_lens.dtype != torch.int32 or out.dtype != torch.float32:
        raise KVQError("seq_lens must be int32 and out float32")
    _check_in_dtype(cache, q)
    B = _check_decode_shapes(cache, layer, q, out, seq_lens)
    _check(load().kv_decode_attention_noalloc(ctypes.byref(cache), layer, _ptr(q), _ptr(out),
                                              _ptr(seq_lens), B, _stream(stream)))


def kv_prefill_scratch_bytes(cache: kvq_cache, layer: int, batch: int) -> int:
    return int(load().kv_prefill_scratch_bytes(ctypes.byref(cache), layer, batch))


def kv_prefill_attention(cache: kvq_cache, layer: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                         out: torch.Tensor, pos: torch.Tensor, scratch: torch.Tensor, stream=None):
    """Append a chunk and attend its queries.  k, v: [L?][B][Hkv][T][128]; q: [L?][B][Hq][T][128];
    out: float32 like q; pos: int32 [B]; scratch: device bytes, at least kv_prefill_scratch_bytes."""
    if pos.dtype != torch.int32 or out.dtype != torch.float32:
        raise KVQError("pos must be int32 and out float32")
    _check_in_dtype(cache, k, v, q)
    B, T = _check_append_shapes(cache, layer, k, v, pos)
    lead = (_layers_in_call(cache, layer),) if layer == -1 else ()
    _check_shape("q", q, lead + (B, cache.cfg.n_q_heads, T, 128))
    _check_shape("out", out, tuple(q.shape))
    _check(load().kv_prefill_attention(ctypes.byref(cache), layer, _ptr(k), _ptr(v), _ptr(q), _ptr(out),
                                       _ptr(pos), B, T, _ptr(scratch), scratch.numel() * scratch.element_size(),
                                       _stream(stream)))


def _in_dtype_of(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KVQ_IN_BF16
    if t.dtype == torch.float32:
        return KVQ_IN_F32
    raise KVQError(f"float32 or bfloat16 input expected, got {t.dtype}")


def kv_tbq_block_bytes(bits: int) -> int:
    return int(load().kv_tbq_block_bytes(bits))


def kv_tbq_encode(bits: int, seed: int, x: torch.Tensor, blocks: torch.Tensor, stream=None):
    """x: [..., 256] float32/bf16 (n_blocks = numel / 256); blocks: uint8 [n_blocks][98 or 130]."""
    nb = x.numel() // 256
    if x.shape[-1] != 256 or blocks.dtype != torch.uint8 or blocks.numel() != nb * kv_tbq_block_bytes(bits):
        raise KVQError("x must be [..., 256] and blocks uint8 of n_blocks * kv_tbq_block_bytes(bits) bytes")
    _check(load().kv_tbq_encode(bits, seed, _ptr(x), _in_dtype_of(x), nb, _ptr(blocks), _stream(stream)))


def kv_tbq_decode(bits: int, seed: int, blocks: torch.Tensor, out: torch.Tensor, stream=None):
    """blocks: uint8 [n_blocks][98 or 130]; out: float32 [..., 256] with n_blocks * 256 values."""
    nb = out.numel() // 256
    if out.dtype != torch.float32 or out.shape[-1] != 256 or blocks.numel() != nb * kv_tbq_block_bytes(bits):
        raise KVQError("out must be float32 [..., 256] and blocks n_blocks * kv_tbq_block_bytes(bits) bytes")
    _check(load().kv_tbq_decode(bits, seed, _ptr(blocks), nb, _ptr(out), _stream(stream)))


def kv_split_record_bytes(hi_bits: int) -> int:
    return int(load().kv_split_record_bytes(hi_bits))


def kv_split_outliers(calib: torch.Tensor, outliers: torch.Tensor, stream=None):
    """calib: [n_sets][n_tokens][128] float32/bf16; outliers: int16 [n_sets][64] (written)."""
    if calib.dim() != 3 or calib.shape[-1] != 128 or outliers.dtype != torch.int16:
        raise KVQError("calib must be [n_sets][n_tokens][128] and outliers int16")
    _check_shape("outliers", outliers, (calib.shape[0], 64))
    _check(load().kv_split_outliers(_ptr(calib), _in_dtype_of(calib), calib.shape[0], calib.shape[1],
                                    _ptr(outliers), _stream(stream)))


def kv_split_encode(hi_bits: int, seed: int, outliers: torch.Tensor, x: torch.Tensor, records: torch.Tensor,
                    stream=None):
    """x: [n_sets][...][128]; records: uint8 [n_vectors][44 or 60]; outliers: int16 [n_sets][64]."""
    n_sets = outliers.shape[0]
    nv = x.numel() // 128
    if x.shape[0] != n_sets or x.shape[-1] != 128 or records.numel() != nv * kv_split_record_bytes(hi_bits):
        raise KVQError("x must be [n_sets][...][128] and records n_vectors * kv_split_record_bytes bytes")
    _check(load().kv_split_encode(hi_bits, seed, _ptr(outliers), n_sets, _ptr(x), _in_dtype_of(x), nv,
                                  _ptr(records), _stream(stream)))


def kv_split_decode(hi_bits: int, seed: int, outliers: torch.Tensor, records: torch.Tensor, out: torch.Tensor,
                    stream=None):
    n_sets = outliers.shape[0]
    nv = out.numel() // 128
    if out.dtype != torch.float32 or out.shape[0] != n_sets or records.numel() != nv * kv_split_record_bytes(hi_bits):
        raise KVQError("out must be float32 [n_sets][...][128] and records n_vectors * kv_split_record_bytes bytes")
    _check(load().kv_split_decode(hi_bits, seed, _ptr(outliers), n_sets, _ptr(records), nv, _ptr(out),
                                  _stream(stream)))


def kv_status(cache: kvq_cache, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(load().kv_status(ctypes.byref(cache), ctypes.byref(v), _stream(stream)))
    return int(v.value)


def kv_set_wait_limit_ns(ns: int) -> None:
    """Stall limit (ns, 1..1e10) of later decode calls' producer waits; the default is 1e9."""
    _check(load().kv_set_wait_limit_ns(int(ns)))


def kv_strerror(code: int) -> str:
    return load().kv_strerror(code).decode()
