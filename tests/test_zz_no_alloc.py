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
    """Both entry points launch the same deterministic kernels with the same split of the work (the
    scratch only holds partial records, merged in a fixed order), so the outputs are bit-identical;
    the tolerance of the other tests (2e-3 of max |out|) would hide a dependence on stale contents."""
    torch.cuda.set_device(0)
    cache, q, seq = _cache_and_inputs()
    ref = cache.decode(-1, q, seq).clone()
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lib.kv_decode_attention_noalloc(cache.handle, -1, q, out, seq)
        torch.cuda.synchronize()
        assert cache.status() == 0
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"call {call} differs"
    # a per-layer call reuses the same array with a different layout of record ranges and records
    ref1 = cache.decode(1, q[1].contiguous(), seq).clone()
    one = torch.full_like(ref1, float("nan"))
    lib.kv_decode_attention_noalloc(cache.handle, 1, q[1].contiguous(), one, seq)
    torch.cuda.synchronize()
    assert torch.equal(one.view(torch.int32), ref1.view(torch.int32))


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
