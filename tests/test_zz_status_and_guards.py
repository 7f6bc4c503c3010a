"""Device-side checks and buffer bounds of the CUDA path (through the C ABI).

* Guard canaries: every kernel writes only inside the buffers it is given (cache, decode scratch,
  output); the bytes just before and after each buffer keep their fill pattern.
* Status word: a sequence length outside [0, max_seq_len] and a block-table entry outside the
  cache's pages are flagged in the device status word (read and cleared by kv_status); the
  affected sequence attends to nothing / the bad page is skipped, and nothing else changes.
"""

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import lib, synth

from . import harness, layout

pytestmark = pytest.mark.gpu

GUARD = 4096                                   # bytes of canary on each side (keeps 16-B alignment)
FILL = 0xA5


def _guarded_bytes(nbytes):
    buf = torch.full((nbytes + 2 * GUARD,), FILL, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def _guards_intact(buf, nbytes):
    return bool((buf[:GUARD] == FILL).all()) and bool((buf[GUARD + nbytes:] == FILL).all())


def test_kernels_write_only_inside_their_buffers(gpu_lib):
    """Ragged appends (bulk and per-token kernels) and decode (all-layer and per-layer calls,
    both merge kernels) into buffers with canaries on both sides."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, H, Hq, B, cap = 2, 2, 6, 3, 768
    lens = np.array([700, 129, 1], np.int32)
    cfg = lib.make_config(Lyr, H, Hq, B, cap, window=128)
    nbytes = lib.kv_cache_bytes(cfg)
    cbuf, cview = _guarded_bytes(nbytes)
    cache = lib.kv_cache_init(cfg, cview)
    for layer in range(Lyr):
        for b in range(B):
            T = int(lens[b])
            k, v = synth.kv_tokens(w, layer, B, H, 0, T, device="cuda")
            pos = torch.full((B,), -1, dtype=torch.int32, device="cuda")
            pos[b] = 0
            lib.kv_quant_append(cache, layer, k, v, pos)
    torch.cuda.synchronize()
    assert lib.kv_status(cache) == 0

    q = torch.stack([synth.queries(w, layer, B, Hq, device="cuda") for layer in range(Lyr)])
    sl = torch.as_tensor(lens, device="cuda")
    n_out = Lyr * B * Hq * 128
    obuf = torch.full((n_out + 2 * GUARD // 4,), float("nan"), dtype=torch.float32, device="cuda")
    nan_bits = obuf[:1].view(torch.int32).clone()
    out = obuf[GUARD // 4:GUARD // 4 + n_out].view(Lyr, B, Hq, 128)
    need = lib.kv_decode_scratch_bytes(cache, -1, B)
    sbuf, sview = _guarded_bytes(need)
    lib.kv_decode_attention(cache, -1, q, out, sl, sview)
    torch.cuda.synchronize()
    all_layers = out.clone()
    per_layer = torch.empty_like(out)
    for layer in range(Lyr):
        need1 = lib.kv_decode_scratch_bytes(cache, layer, B)
        s1buf, s1view = _guarded_bytes(need1)
        o1buf = torch.full((B * Hq * 128 + 2 * GUARD // 4,), float("nan"), dtype=torch.float32, device="cuda")
        o1 = o1buf[GUARD // 4:GUARD // 4 + B * Hq * 128].view(B, Hq, 128)
        lib.kv_decode_attention(cache, layer, q[layer].contiguous(), o1, sl, s1view)
        torch.cuda.synchronize()
        assert _guards_intact(s1buf, need1)
        head = o1buf[:GUARD // 4].view(torch.int32)
        tail = o1buf[GUARD // 4 + B * Hq * 128:].view(torch.int32)
        assert bool((head == nan_bits).all()) and bool((tail == nan_bits).all())
        per_layer[layer] = o1
    assert lib.kv_status(cache) == 0
    assert _guards_intact(cbuf, nbytes)
    assert _guards_intact(sbuf, need)
    head = obuf[:GUARD // 4].view(torch.int32)
    tail = obuf[GUARD // 4 + n_out:].view(torch.int32)
    assert bool((head == nan_bits).all()) and bool((tail == nan_bits).all())
    assert bool(torch.isfinite(all_layers).all()) and bool(torch.isfinite(per_layer).all())
    scale = float(all_layers.abs().max())
    assert float((all_layers - per_layer).abs().max()) <= 1e-4 * scale


def test_seq_len_out_of_range_is_flagged_and_attends_nothing(gpu_lib):
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    gpu, ora, _ = harness.make_pair(1, 1, 2, 3, 256, window=128)
    k, v = synth.kv_tokens(w, 0, 3, 1, 0, 40, device="cuda")
    gpu.append(0, k, v, torch.zeros(3, dtype=torch.int32, device="cuda"))
    ora.append(0, harness.to_np(k), harness.to_np(v), np.zeros(3, np.int64))
    torch.cuda.synchronize()
    assert gpu.status() == 0
    q = synth.queries(w, 0, 3, 2, device="cuda")
    lens = np.array([300, 40, -7], np.int32)
    out = gpu.decode(0, q, torch.as_tensor(lens, device="cuda"))
    torch.cuda.synchronize()
    assert gpu.status() == 4                       # KVQ_DEV_SEQLEN_RANGE
    assert gpu.status() == 0                       # read-and-clear
    o = harness.to_np(out)
    assert not o[0].any() and not o[2].any()       # treated as empty
    want = ora.decode(0, harness.to_np(q), np.array([0, 40, 0]))
    harness.assert_attention_close(o[1], want[1])


def test_bad_block_table_entry_is_flagged_and_skipped(gpu_lib):
    """A block-table entry outside the cache's pages: decode flags it and skips that page (the
    other sequences are unaffected); an append through it flags it and writes no page."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    B, H, Hq, cap = 2, 1, 2, 512
    maxpps = cap // 64
    n_pages = B * maxpps
    bt = np.random.default_rng(7).permutation(n_pages).astype(np.int32).reshape(B, maxpps)
    gpu, ora, _ = harness.make_pair(1, H, Hq, B, cap, window=128, n_pages=n_pages, block_table=bt)
    T = 400
    k, v = synth.kv_tokens(w, 0, B, H, 0, T, device="cuda")
    gpu.append(0, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    ora.append(0, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    torch.cuda.synchronize()
    assert gpu.status() == 0

    gpu.block_table[0, 1] = n_pages                # sequence 0, tokens 64..127: past the last page
    q = synth.queries(w, 0, B, Hq, device="cuda")
    lens = np.array([T, T], np.int32)
    out = gpu.decode(0, q, torch.as_tensor(lens, device="cuda"))
    torch.cuda.synchronize()
    assert gpu.status() == 1                       # KVQ_DEV_BAD_PAGE
    o = harness.to_np(out)
    assert np.all(np.isfinite(o[0]))
    want = ora.decode(0, harness.to_np(q), lens)
    harness.assert_attention_close(o[1], want[1])

    gpu.block_table[1, 7] = -3                     # sequence 1, tokens 448..511: not written yet
    before = gpu.buffer.clone()
    for n in (40, 1):                              # the bulk and the per-token append kernels
        kk, vv = synth.kv_tokens(w, 0, B, H, T, n, device="cuda")
        gpu.append(0, kk, vv, torch.tensor([-1, 448], dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        assert gpu.status() == 1
    off = layout.regions(gpu.cfg, gpu.buffer.numel())["off_pages"]
    assert torch.equal(before[off:], gpu.buffer[off:])  # no page byte changed (the ring may)


def test_calls_with_another_device_current_are_refused(gpu_lib):
    """The cache's pointers belong to the device current at kv_cache_init; a handle that names
    another device (as if that device were current now) is refused before anything launches."""
    import ctypes

    w = synth.WORKLOADS["qwen3-4b-kvarn-128k"]
    gpu, _, _ = harness.make_pair(1, 1, 2, 1, 256, window=128, sinkhorn=True)
    other = lib.kvq_cache.from_buffer_copy(gpu.handle)
    other.device = gpu.handle.device + 1
    k, v = synth.kv_tokens(w, 0, 1, 1, 0, 8, device="cuda")
    q = synth.queries(w, 0, 1, 2, device="cuda")
    out = torch.zeros(1, 2, 128, dtype=torch.float32, device="cuda")
    sl = torch.tensor([8], dtype=torch.int32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = gpu.scratch(0, 1)
    before = gpu.buffer.clone()
    for call in (lambda: lib.kv_quant_append(other, 0, k, v, pos),
                 lambda: lib.kv_decode_attention(other, 0, q, out, sl, scratch),
                 lambda: lib.kv_decode_attention_noalloc(other, 0, q, out, sl),
                 lambda: lib.kv_calibrate(other, 0, k[0].contiguous(), v[0].contiguous(),
                                          torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))):
        with pytest.raises(lib.KVQError, match="code 1"):
            call()
    torch.cuda.synchronize()
    assert torch.equal(before, gpu.buffer) and torch.count_nonzero(out).item() == 0
    assert ctypes.sizeof(other) == ctypes.sizeof(gpu.handle)
