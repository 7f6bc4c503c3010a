"""GPU parity of the chunked prefill (append a chunk, attend its queries) against the CPU oracle.

The oracle's prefill is its definition written out: T single-token steps (append token t, decode at
length pos + t + 1).  Checked: every stored field of the appended chunk bit-exact, and every query's
attention within 2e-3 of the oracle's max |out|, for each key format, windows 0 / partial /
covering the whole context, ragged and skipped sequences, Sinkhorn balancing, an all-layer call.
"""

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import synth
from oracle import attention

from . import harness, layout

pytestmark = pytest.mark.gpu

WL = {"q4g32": "llama3.2-3b-32k", "q8g32": "llama3.2-3b-32k-k8v4", "tq3_qjl": "llama3.1-8b-tq-b8-32k"}


def _queries(w, layer, B, Hq, T):
    """[B][Hq][T][128]: one decode-step query set per position of the chunk."""
    return torch.stack([synth.queries(w, layer, B, Hq, step=t, device="cuda") for t in range(T)], dim=2).contiguous()


def _run(k_format, window, H, Hq, prefix, T, sinkhorn=False, layers=1, all_layers=False, in_dtype="bf16"):
    """Prefix appends (positions [0, prefix[b])), then one prefill chunk of T tokens at pos = prefix
    (a negative prefix: the sequence takes no part)."""
    prefix = np.asarray(prefix)
    B = len(prefix)
    cap = int(max(prefix.max(), 0) + T + 64)
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k" if sinkhorn else WL[k_format]]
    dt = torch.float32 if in_dtype == "f32" else None
    gpu, ora, _ = harness.make_pair(layers, H, Hq, B, cap, window=window, k_format=k_format, sinkhorn=sinkhorn,
                                    in_dtype=in_dtype)
    for l in range(layers):
        if sinkhorn:
            kc, vc = synth.kv_tokens(w, l, 1, H, 5000, 300, device="cuda")
            gpu.calibrate(l, kc[0].contiguous(), vc[0].contiguous())
            ora.calibrate(l, harness.to_np(kc[0]), harness.to_np(vc[0]))
        pmax = int(max(prefix.max(), 0))
        if pmax > 0:
            k, v = synth.kv_tokens(w, l, B, H, 0, pmax, device="cuda", dtype=dt)
            for b in range(B):
                if prefix[b] > 0:
                    p = np.where(np.arange(B) == b, 0, -1).astype(np.int32)
                    kk = k[:, :, :prefix[b]].contiguous()
                    vv = v[:, :, :prefix[b]].contiguous()
                    gpu.append(l, kk, vv, torch.as_tensor(p, device="cuda"))
                    ora.append(l, harness.to_np(kk), harness.to_np(vv), p)
    pos = prefix.astype(np.int32)
    chunks = [synth.kv_tokens(w, l, B, H, 20000, T, device="cuda", dtype=dt) for l in range(layers)]
    qs = [_queries(w, l, B, Hq, T) for l in range(layers)]
    if dt is not None:
        qs = [q.float() for q in qs]
    want = []
    for l in range(layers):
        k, v = chunks[l]
        want.append(attention.prefill(ora, l, harness.to_np(k), harness.to_np(v), harness.to_np(qs[l]), pos))
    pos_d = torch.as_tensor(pos, device="cuda")
    if all_layers:
        k = torch.stack([c[0] for c in chunks]).contiguous()
        v = torch.stack([c[1] for c in chunks]).contiguous()
        got = gpu.prefill(-1, k, v, torch.stack(qs).contiguous(), pos_d)
        got = [got[l] for l in range(layers)]
    else:
        got = [gpu.prefill(l, chunks[l][0], chunks[l][1], qs[l], pos_d) for l in range(layers)]
    torch.cuda.synchronize()
    assert gpu.status() == 0
    for l in range(layers):
        g = harness.to_np(got[l])
        for b in range(B):
            if pos[b] < 0:
                assert not g[b].any()
                continue
            harness.assert_attention_close(g[b], want[l][b])
            for h in range(H):
                harness.compare_codes(gpu, ora, l, b, h, int(pos[b]) + T)
                harness.compare_ring(gpu, ora, l, b, h, int(pos[b]) + T)
    return got, want


@pytest.mark.parametrize("window", [128, 64, 0])
def test_prefill_q4_windows(gpu_lib, window):
    """GQA 3 (63 of 64 rows per block): sequences with no prefix (the window covers the first
    queries' whole context), a prefix of 150, and one that takes no part."""
    _run("q4g32", window, 2, 6, [0, 150, -1], 90)


def test_prefill_q8_keys(gpu_lib):
    _run("q8g32", 128, 2, 4, [200, 31], 80)


def test_prefill_tq3_keys(gpu_lib):
    """GQA 4: [q~, S q~] against [n c, n sqrt(pi/2)/128 gamma (2b - 1)]."""
    _run("tq3_qjl", 128, 2, 8, [100, 0], 75)


def test_prefill_sinkhorn(gpu_lib):
    _run("q4g32", 128, 2, 8, [300, 10], 65, sinkhorn=True)


def test_prefill_all_layers_call(gpu_lib):
    """One call over two layers (leading layer axis), GQA 2, the chunk longer than a block's 32
    queries and than the window."""
    _run("q4g32", 128, 2, 4, [40, 257], 140, layers=2, all_layers=True)


def test_prefill_fp32_inputs_and_mha(gpu_lib):
    """fp32 inputs, one query head per kv-head (64 queries a block), chunk start inside a page."""
    _run("q4g32", 128, 1, 1, [77], 100, in_dtype="f32")


def test_prefill_matches_token_steps_on_the_gpu(gpu_lib):
    """The GPU's own prefill against T single-token GPU steps (append, then decode at pos + t + 1):
    within the tolerance (different splits and precision paths), same stored bytes."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    H, Hq, B, T, cap = 2, 6, 2, 40, 512
    a, _, _ = harness.make_pair(1, H, Hq, B, cap, window=64)
    c, _, _ = harness.make_pair(1, H, Hq, B, cap, window=64)
    k0, v0 = synth.kv_tokens(w, 0, B, H, 0, 200, device="cuda")
    for x in (a, c):
        x.append(0, k0, v0, torch.zeros(B, dtype=torch.int32, device="cuda"))
    k, v = synth.kv_tokens(w, 0, B, H, 9000, T, device="cuda")
    q = _queries(w, 0, B, Hq, T)
    got = a.prefill(0, k, v, q, torch.full((B,), 200, dtype=torch.int32, device="cuda"))
    steps = []
    for t in range(T):
        c.append(0, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(),
                 torch.full((B,), 200 + t, dtype=torch.int32, device="cuda"))
        steps.append(c.decode(0, q[:, :, t].contiguous(), torch.full((B,), 201 + t, dtype=torch.int32,
                                                                        device="cuda")).clone())
    torch.cuda.synchronize()
    ref = torch.stack(steps, dim=2)
    assert (got - ref).abs().max().item() <= 2e-3 * ref.abs().max().item()
    for b in range(B):
        for h in range(H):
            ua = layout.read_unit(a.buffer, a.cfg, 0, b, h, 200 + T)
            uc = layout.read_unit(c.buffer, c.cfg, 0, b, h, 200 + T)
            for name in ua:
                assert np.array_equal(ua[name].view(np.uint8), uc[name].view(np.uint8)), name
