"""The allocation-free decode entry point (for callers that cannot allocate device memory).

kv_decode_attention_noalloc takes its scratch from a fixed array inside the library instead of a
caller buffer.  Its results must match kv_decode_attention's on the same cache, call after call
(the shared array keeps the previous call's contents, so a second call checks that nothing depends
on them), and a
call that needs more scratch than the array holds must be refused without launching anything.
This file is collected last so that a run stopping at its first failure has run everything else.
"""

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import QuantKVCache, lib, synth

pytestmark = pytest.mark.gpu


def _cache_and_inputs():
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, H, Hq, B = 2, 2, 6, 3
    lens = np.array([1500, 37, 900], np.int32)
    cache = QuantKVCache(lib.make_config(Lyr, H, Hq, B, 1600, window=128), "cuda")
    for layer in range(Lyr):
        k, v = synth.kv_tokens(w, layer, B, H, 0, int(lens.max()), device="cuda")
        cache.append(layer, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    q = torch.stack([synth.queries(w, layer, B, Hq, device="cuda") for layer in range(Lyr)]).contiguous()
    return cache, q, torch.as_tensor(lens, device="cuda")


def test_noalloc_matches_scratch_entry_point_on_consecutive_calls():
    torch.cuda.set_device(0)
    cache, q, seq = _cache_and_inputs()
    ref = cache.decode(-1, q, seq).clone()
    torch.cuda.synchronize()
    scale = ref.abs().max().item()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lib.kv_decode_attention_noalloc(cache.handle, -1, q, out, seq)
        torch.cuda.synchronize()
        assert cache.status() == 0
        err = (out - ref).abs().max().item()
        assert err <= 2e-3 * scale, f"call {call}: max abs err {err:.3e} vs {scale:.3e}"
    # a per-layer call reuses the same array with a different layout of record ranges and records
    one = torch.empty(q.shape[1:], dtype=torch.float32, device="cuda")
    lib.kv_decode_attention_noalloc(cache.handle, 1, q[1].contiguous(), one, seq)
    torch.cuda.synchronize()
    assert (one - ref[1]).abs().max().item() <= 2e-3 * scale


def test_noalloc_refuses_calls_beyond_its_array():
    torch.cuda.set_device(0)
    cfg = lib.make_config(4, 8, 8, 256, 64, window=0)
    cache = QuantKVCache(cfg, "cuda")
    assert lib.kv_decode_scratch_bytes(cache.handle, -1, 256) > lib.NOALLOC_SCRATCH_MAX
    q = torch.zeros(4, 256, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(4, 256, 8, 128, dtype=torch.float32, device="cuda")
    seq = torch.ones(256, dtype=torch.int32, device="cuda")
    with pytest.raises(lib.KVQError, match="code 4"):
        lib.kv_decode_attention_noalloc(cache.handle, -1, q, out, seq)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
