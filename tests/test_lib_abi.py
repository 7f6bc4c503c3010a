"""The C ABI library: builds, loads without a GPU, exports every declared symbol, sizes caches."""

import os
import re

import pytest

from kv_cache_quantization_append_gb300 import lib, synth
from oracle import attention

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    if not os.path.exists(lib.LIB_PATH):
        from kv_cache_quantization_append_gb300 import build

        build.build()
    return lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(kvq):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(kvq, n), n
    assert set(names) == set(lib.EXPORTS)


def test_strerror(kvq):
    assert lib.kv_strerror(0) == "ok"
    assert "unknown" in lib.kv_strerror(99)


def _cfg(w, layers=None):
    return lib.make_config(layers or w.get("alloc_layers", w["n_layers"]), w["n_kv_heads"], w["n_q_heads"],
                           w["batch"], w.get("ctx", w.get("ctx_range", (0, 0))[1]), window=w["window"],
                           k_format=lib.K_FORMATS[w["k_format"]],
                           sinkhorn=w["sinkhorn"])


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_cache_bytes_closed_form(kvq, name):
    """Library size = oracle payload (records + window ring) + page rounding + a small header."""
    w = synth.WORKLOADS[name]
    cfg = _cfg(w)
    got = lib.kv_cache_bytes(cfg)
    ocfg = attention.OracleConfig(n_layers=cfg.n_layers, n_kv_heads=cfg.n_kv_heads, n_q_heads=cfg.n_q_heads,
                                  max_batch=cfg.max_batch, max_seq_len=cfg.max_seq_len, window=cfg.window,
                                  k_format=w["k_format"], v_format=w["v_format"])
    pages = -(-cfg.max_seq_len // 64) * 64
    payload = (cfg.n_layers * cfg.max_batch * cfg.n_kv_heads * pages *
               attention.payload_bytes_per_token_head(ocfg) + attention.window_bytes(ocfg))
    header = got - payload
    assert 0 < header <= 64 * 1024 + 128 * 128 * 4 + 4 * cfg.max_batch * pages // 64 + \
        4 * cfg.n_layers * cfg.n_kv_heads * 256 + 4096


def test_invalid_configs_have_no_size(kvq):
    good = lib.make_config(2, 8, 24, 1, 1024)
    assert lib.kv_cache_bytes(good) > 0
    for field, bad in (("head_dim", 64), ("n_q_heads", 23), ("n_q_heads", 48), ("window", 102),
                       ("page_tokens", 32), ("k_format", 7), ("max_batch", 0)):
        c = lib.make_config(2, 8, 24, 1, 1024)
        setattr(c, field, bad)
        assert lib.kv_cache_bytes(c) == 0, field
    c = lib.make_config(2, 8, 24, 1, 1024, k_format=lib.KVQ_TQ3_QJL, sinkhorn=True)
    assert lib.kv_cache_bytes(c) == 0


def test_llama_3b_32k_quantised_store_is_6_4x_smaller_than_fp32(kvq):
    """[QC]: 6.4x KV compression; FP32 KV of Llama-3.2-3B at 32K is 7.17 GB."""
    flat = lib.make_config(28, 8, 24, 1, 32768, window=0)
    b = lib.kv_cache_bytes(flat)
    fp32 = attention.fp32_kv_bytes(28, 8, 32768)
    assert abs(fp32 / b - 6.4) < 0.01


# ------------------------------------------------------------------ host-side argument checks
# Only inputs that the library rejects before its first CUDA call: no device is touched, and the
# fake device addresses below are never dereferenced.
KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_ALIGN = 0, 1, 2, 3
KVQ_ERR_CAPACITY, KVQ_ERR_CUDA, KVQ_ERR_NOT_INIT = 4, 5, 6
FAKE_DEV = 0x7F0000000000          # 16-byte aligned, never dereferenced


def test_strerror_names_every_status_code(kvq):
    msgs = [lib.kv_strerror(c) for c in range(7)]
    assert len(set(msgs)) == 7 and not any("unknown" in m for m in msgs)
    assert "align" in msgs[KVQ_ERR_ALIGN] and "initialised" in msgs[KVQ_ERR_NOT_INIT]


def test_cache_init_rejects_bad_arguments_before_any_device_work(kvq):
    import ctypes

    cfg = lib.make_config(2, 8, 24, 1, 1024)
    need = lib.kv_cache_bytes(cfg)
    cache = lib.kvq_cache()
    init = kvq.kv_cache_init
    P = ctypes.c_void_p
    assert init(None, ctypes.byref(cfg), P(FAKE_DEV), need, None, None, None) == KVQ_ERR_INVALID_ARG
    assert init(ctypes.byref(cache), None, P(FAKE_DEV), need, None, None, None) == KVQ_ERR_INVALID_ARG
    assert init(ctypes.byref(cache), ctypes.byref(cfg), None, need, None, None, None) == KVQ_ERR_INVALID_ARG
    bad = lib.make_config(2, 8, 24, 1, 1024, window=102)
    assert init(ctypes.byref(cache), ctypes.byref(bad), P(FAKE_DEV), need, None, None, None) == KVQ_ERR_UNSUPPORTED
    assert init(ctypes.byref(cache), ctypes.byref(cfg), P(FAKE_DEV), need - 1, None, None, None) == KVQ_ERR_CAPACITY
    assert init(ctypes.byref(cache), ctypes.byref(cfg), P(FAKE_DEV + 8), need, None, None, None) == KVQ_ERR_ALIGN
    assert init(ctypes.byref(cache), ctypes.byref(cfg), P(FAKE_DEV), need, P(FAKE_DEV + 4), None,
                None) == KVQ_ERR_ALIGN
    tq = lib.make_config(2, 8, 24, 1, 1024, k_format=lib.KVQ_TQ3_QJL)
    assert init(ctypes.byref(cache), ctypes.byref(tq), P(FAKE_DEV), lib.kv_cache_bytes(tq), None, None,
                None) == KVQ_ERR_INVALID_ARG          # TurboQuant keys need the projection matrix
    assert cache.magic == 0                          # nothing was initialised


def test_uninitialised_cache_is_refused_by_every_entry_point(kvq):
    import ctypes

    cache = lib.kvq_cache()                           # zeroed: never passed through kv_cache_init
    cache.cfg = lib.make_config(2, 8, 24, 1, 1024)
    c = ctypes.byref(cache)
    P = ctypes.c_void_p
    d = P(FAKE_DEV)
    flags = ctypes.c_uint32(0)
    assert kvq.kv_calibrate(c, 0, d, d, 64, d, 1 << 20, None) == KVQ_ERR_NOT_INIT
    assert kvq.kv_quant_append(c, 0, d, d, d, 1, 1, None) == KVQ_ERR_NOT_INIT
    assert kvq.kv_decode_attention(c, 0, d, d, d, 1, d, 1 << 20, None) == KVQ_ERR_NOT_INIT
    assert kvq.kv_decode_attention_noalloc(c, 0, d, d, d, 1, None) == KVQ_ERR_NOT_INIT
    assert kvq.kv_status(c, ctypes.byref(flags), None) == KVQ_ERR_NOT_INIT
    assert kvq.kv_calibrate_scratch_bytes(c, 0, 64) == 0
    assert kvq.kv_decode_scratch_bytes(c, 0, 1) == 0
    # and a NULL cache
    assert kvq.kv_quant_append(None, 0, d, d, d, 1, 1, None) == KVQ_ERR_INVALID_ARG
    assert kvq.kv_decode_attention_noalloc(None, 0, d, d, d, 1, None) == KVQ_ERR_INVALID_ARG


def test_cache_bytes_null_config(kvq):
    assert kvq.kv_cache_bytes(None) == 0


def test_block_codec_sizes_and_refusals(kvq):
    """Record sizes are the pages' bit widths; unsupported widths and bad arguments are refused
    before any device work."""
    import ctypes

    assert lib.kv_tbq_block_bytes(3) == 98 and lib.kv_tbq_block_bytes(4) == 130
    assert lib.kv_tbq_block_bytes(2) == 0 and lib.kv_tbq_block_bytes(5) == 0
    assert lib.kv_split_record_bytes(3) == 44 and lib.kv_split_record_bytes(4) == 60
    assert lib.kv_split_record_bytes(2) == 0
    P = ctypes.c_void_p
    d = P(FAKE_DEV)
    assert kvq.kv_tbq_encode(5, 0, d, 1, 4, d, None) == KVQ_ERR_UNSUPPORTED
    assert kvq.kv_tbq_encode(3, 0, d, 7, 4, d, None) == KVQ_ERR_UNSUPPORTED
    assert kvq.kv_tbq_encode(3, 0, None, 1, 4, d, None) == KVQ_ERR_INVALID_ARG
    assert kvq.kv_tbq_encode(3, 0, P(FAKE_DEV + 4), 1, 4, d, None) == KVQ_ERR_ALIGN
    assert kvq.kv_tbq_decode(4, 0, d, -1, d, None) == KVQ_ERR_INVALID_ARG
    assert kvq.kv_split_encode(3, 0, d, 3, d, 1, 10, d, None) == KVQ_ERR_INVALID_ARG     # 10 vectors, 3 sets
    assert kvq.kv_split_encode(5, 0, d, 1, d, 1, 10, d, None) == KVQ_ERR_UNSUPPORTED
    assert kvq.kv_split_decode(4, 0, None, 1, d, 10, d, None) == KVQ_ERR_INVALID_ARG
    assert kvq.kv_split_outliers(d, 1, 0, 10, d, None) == KVQ_ERR_INVALID_ARG


# ------------------------------------------------------------------ the header from plain C
C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvq.h"

int main(void) {
  kvq_config c;
  kvq_cache cache;
  size_t good, bad;
  int rc;
  memset(&c, 0, sizeof c);
  c.n_layers = 28; c.n_kv_heads = 8; c.n_q_heads = 24; c.head_dim = 128; c.max_batch = 1;
  c.max_seq_len = 32768; c.window = 128; c.page_tokens = 64; c.n_pages = 0;
  c.k_format = KVQ_Q4G32; c.v_format = KVQ_Q4G32; c.sinkhorn = 0; c.group = 32;
  c.in_dtype = KVQ_IN_BF16; c.seed = 0;
  good = kv_cache_bytes(&c);
  c.head_dim = 64;
  bad = kv_cache_bytes(&c);
  memset(&cache, 0, sizeof cache);
  rc = kv_quant_append(&cache, 0, NULL, NULL, NULL, 1, 1, NULL);
  printf("%zu %zu %d %s\n", good, bad, rc, kv_strerror(rc));
  return 0;
}
"""


def test_header_is_plain_c_and_links(kvq):
    """include/kvq.h compiles as strict C99 and as C++; a C program links against libkvq.so and
    calls it (size query, refusal of an uninitialised cache) with no GPU."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    out_dir = os.path.dirname(lib.LIB_PATH)
    src = os.path.join(out_dir, "abi_check.c")
    exe = os.path.join(out_dir, "abi_check")
    with open(src, "w") as f:
        f.write(C_PROGRAM)
    inc = os.path.join(ROOT, "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, src,
                    "-L", out_dir, "-lkvq", f"-Wl,-rpath,{out_dir}", "-o", exe], check=True)
    gxx = shutil.which("g++")
    if gxx is not None:
        subprocess.run([gxx, "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++",
                        os.path.join(inc, "kvq.h")], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, check=True)
    good, bad, rc, msg = res.stdout.strip().split(" ", 3)
    cfg = lib.make_config(28, 8, 24, 1, 32768, window=128)
    assert int(good) == lib.kv_cache_bytes(cfg) > 0
    assert int(bad) == 0
    assert int(rc) == 6 and msg == "cache not initialised"


# ------------------------------------------------------------------ the binding's shape checks
# The library reads q, k, v and writes out through bare pointers; a tensor of the wrong size would
# be read or written past its end, which the C ABI cannot see.  The binding refuses such tensors
# before any library call (so these checks run on CPU tensors, with no device touched).
def _fake_cache(layers=2, hkv=2, hq=6, batch=3):
    cache = lib.kvq_cache()
    cache.cfg = lib.make_config(layers, hkv, hq, batch, 256)
    return cache


def test_decode_binding_refuses_mismatched_shapes():
    import torch

    c = _fake_cache()
    bf = torch.bfloat16
    sl = torch.zeros(3, dtype=torch.int32)
    cases = [
        (-1, torch.zeros(3, 6, 128, dtype=bf), torch.zeros(3, 6, 128)),          # no layer axis
        (-1, torch.zeros(1, 3, 6, 128, dtype=bf), torch.zeros(1, 3, 6, 128)),    # one layer of two
        (0, torch.zeros(2, 3, 6, 128, dtype=bf), torch.zeros(2, 3, 6, 128)),     # layer axis on a layer call
        (0, torch.zeros(3, 4, 128, dtype=bf), torch.zeros(3, 4, 128)),           # wrong head count
        (0, torch.zeros(3, 6, 128, dtype=bf), torch.zeros(2, 6, 128)),           # out smaller than q
        (0, torch.zeros(3, 6, 64, dtype=bf), torch.zeros(3, 6, 64)),             # head_dim 64
    ]
    for layer, q, out in cases:
        for fn in (lambda: lib.kv_decode_attention(c, layer, q, out, sl, torch.zeros(16, dtype=torch.uint8)),
                   lambda: lib.kv_decode_attention_noalloc(c, layer, q, out, sl)):
            with pytest.raises(lib.KVQError, match="shape|must be"):
                fn()
    q = torch.zeros(3, 6, 128, dtype=bf)
    with pytest.raises(lib.KVQError, match="seq_lens"):
        lib.kv_decode_attention_noalloc(c, 0, q, torch.zeros(3, 6, 128), torch.zeros(2, dtype=torch.int32))


def test_append_binding_refuses_mismatched_shapes():
    import torch

    c = _fake_cache()
    bf = torch.bfloat16
    pos = torch.zeros(3, dtype=torch.int32)
    cases = [
        (-1, torch.zeros(3, 2, 5, 128, dtype=bf), torch.zeros(3, 2, 5, 128, dtype=bf), pos),
        (-1, torch.zeros(1, 3, 2, 5, 128, dtype=bf), torch.zeros(1, 3, 2, 5, 128, dtype=bf), pos),
        (0, torch.zeros(3, 1, 5, 128, dtype=bf), torch.zeros(3, 1, 5, 128, dtype=bf), pos),
        (0, torch.zeros(3, 2, 5, 128, dtype=bf), torch.zeros(3, 2, 4, 128, dtype=bf), pos),
        (0, torch.zeros(3, 2, 5, 128, dtype=bf), torch.zeros(3, 2, 5, 128, dtype=bf), pos[:2]),
    ]
    for layer, k, v, p in cases:
        with pytest.raises(lib.KVQError, match="shape|must be"):
            lib.kv_quant_append(c, layer, k, v, p)


def test_wait_limit_range_is_checked(kvq):
    """kv_set_wait_limit_ns refuses 0 and limits above 10 s (no device work either way)."""
    assert kvq.kv_set_wait_limit_ns(0) == 1                 # KVQ_ERR_INVALID_ARG
    assert kvq.kv_set_wait_limit_ns(10**10 + 1) == 1
    assert kvq.kv_set_wait_limit_ns(10**9) == 0             # the default, restored
