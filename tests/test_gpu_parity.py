"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Codes, scales, zeros, norms, sign bits, Sinkhorn scales and ring contents must match bit for bit;
attention outputs within 2e-3 of max |out| of the float64 oracle, per layer.
"""

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import synth
from oracle import codec

from . import harness, layout

pytestmark = pytest.mark.gpu


def _inputs(w, layer, B, H, Hq, T, t0=0, dtype=None):
    k, v = synth.kv_tokens(w, layer, B, H, t0, T, device="cuda", dtype=dtype)
    return k, v


def _decode_both(gpu, ora, layer, q, seq_lens_np):
    sl = torch.as_tensor(seq_lens_np, dtype=torch.int32, device="cuda")
    out = gpu.decode(layer, q, sl)
    torch.cuda.synchronize()
    assert gpu.status() == 0
    want = ora.decode(layer, harness.to_np(q), seq_lens_np)
    return harness.to_np(out), want


def test_tiny_reference_workload(gpu_lib):
    """1 layer, 4 query heads on 1 kv head, 512 tokens, fp32, K channels 0-3 x10, window 128."""
    w = synth.WORKLOADS["tiny"]
    gpu, ora, _ = harness.make_pair(1, 1, 4, 1, 512, window=128, in_dtype="f32", seed=0)
    k, v = _inputs(w, 0, 1, 1, 4, 512)
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu.append(0, k, v, pos)
    ora.append(0, harness.to_np(k), harness.to_np(v), np.array([0]))
    harness.compare_codes(gpu, ora, 0, 0, 0, 512)
    harness.compare_ring(gpu, ora, 0, 0, 0, 512)
    q = synth.queries(w, 0, 1, 4, device="cuda")
    got, want = _decode_both(gpu, ora, 0, q, np.array([512]))
    harness.assert_attention_close(got, want)


def test_bulk_append_equals_token_by_token(gpu_lib):
    """[QC] v3.2: a T-token append writes exactly the bytes of T single-token appends."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    a, _, _ = harness.make_pair(1, 2, 6, 2, 400, window=128)
    b, _, _ = harness.make_pair(1, 2, 6, 2, 400, window=128)
    k, v = _inputs(w, 0, 2, 2, 6, 300)
    a.append(0, k, v, torch.tensor([5, 50], dtype=torch.int32, device="cuda"))
    for t in range(300):
        b.append(0, k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(),
                 torch.tensor([5 + t, 50 + t], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    R = layout.regions(a.cfg, a.buffer.numel())
    # pages and ring of positions actually written must be identical; compare via the readers
    for s, p0 in ((0, 5), (1, 50)):
        for h in range(2):
            ua = layout.read_unit(a.buffer, a.cfg, 0, s, h, p0 + 300)
            ub = layout.read_unit(b.buffer, b.cfg, 0, s, h, p0 + 300)
            for name in ua:
                assert np.array_equal(ua[name][p0:].view(np.uint8), ub[name][p0:].view(np.uint8)), name
            ka, va = layout.read_ring(a.buffer, a.cfg, 0, s, h)
            kb, vb = layout.read_ring(b.buffer, b.cfg, 0, s, h)
            assert np.array_equal(ka.view(np.uint32), kb.view(np.uint32))
            assert np.array_equal(va.view(np.uint32), vb.view(np.uint32))
    assert R["page_bytes"] == 10240 and R["half_bytes"] == 5120


@pytest.mark.parametrize("window", [128, 0, 64])
def test_ragged_edge_lengths(gpu_lib, window):
    lens = np.array([0, 1, 7, 63, 64, 65, 127, 128, 129, 191, 192, 200, 700, 1100], dtype=np.int32)
    B = len(lens)
    w = synth.WORKLOADS["dense27b-ragged-b32"]
    gpu, ora, _ = harness.make_pair(1, 2, 4, B, 1152, window=window)
    T = int(lens.max())
    k, v = _inputs(w, 0, B, 2, 4, T)
    gpu.append(0, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    ora.append(0, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    q = synth.queries(w, 0, B, 4, device="cuda")
    got, want = _decode_both(gpu, ora, 0, q, lens)
    for b in range(B):
        if lens[b] == 0:
            assert np.all(got[b] == 0)
        else:
            harness.assert_attention_close(got[b], want[b])


def test_multilayer_gqa3_all_layers_call(gpu_lib):
    """Llama-3.2-3B-shaped (GQA 3) at small size: one launch over all layers and per-layer calls."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, H, Hq, L = 3, 2, 6, 1500
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, 1, 2048, window=128)
    ks, vs = zip(*[_inputs(w, l, 1, H, Hq, L) for l in range(Lyr)])
    k, v = torch.stack(ks), torch.stack(vs)
    gpu.append(-1, k, v, torch.zeros(1, dtype=torch.int32, device="cuda"))
    for l in range(Lyr):
        ora.append(l, harness.to_np(ks[l]), harness.to_np(vs[l]), np.array([0]))
        for h in range(H):
            harness.compare_codes(gpu, ora, l, 0, h, L)
            harness.compare_ring(gpu, ora, l, 0, h, L)
    q = torch.stack([synth.queries(w, l, 1, Hq, device="cuda") for l in range(Lyr)])
    sl = np.array([L], dtype=np.int32)
    out = gpu.decode(-1, q, torch.as_tensor(sl, device="cuda"))
    torch.cuda.synchronize()
    for l in range(Lyr):
        want = ora.decode(l, harness.to_np(q[l]), sl)
        harness.assert_attention_close(harness.to_np(out[l]), want)
        one = gpu.decode(l, q[l].contiguous(), torch.as_tensor(sl, device="cuda"))
        torch.cuda.synchronize()
        harness.assert_attention_close(harness.to_np(one), want)


def test_decode_is_deterministic(gpu_lib):
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    gpu, _, _ = harness.make_pair(2, 2, 6, 3, 3000, window=128)
    for l in range(2):
        k, v = _inputs(w, l, 3, 2, 6, 2900)
        gpu.append(l, k, v, torch.zeros(3, dtype=torch.int32, device="cuda"))
    q = torch.stack([synth.queries(w, l, 3, 6, device="cuda") for l in range(2)])
    sl = torch.tensor([2900, 1234, 77], dtype=torch.int32, device="cuda")
    a = gpu.decode(-1, q, sl).clone()
    b = gpu.decode(-1, q, sl).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_output_independent_of_the_split(gpu_lib):
    """The same decode as one all-layer call (64 units over the grid's warps: one-warp merges of a
    few records each) and as per-layer calls (16 units: each unit spread over ~140 warps and merged
    by a CTA per head) splits the work differently; the outputs agree far inside the oracle
    tolerance (1e-4 of max |out| here, against 2e-3)."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, H, Hq, B = 4, 2, 6, 8
    lens = np.array([2000, 1500, 777, 64, 1999, 1234, 3, 1800], np.int32)
    gpu, _, _ = harness.make_pair(Lyr, H, Hq, B, 2048, window=128)
    for b in range(B):
        # sequence b alone (the others' positions are negative: untouched), exactly lens[b] tokens
        pos = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        pos[b] = 0
        for l in range(Lyr):
            k, v = _inputs(w, l, B, H, Hq, int(lens[b]))
            gpu.append(l, k, v, pos)
    q = torch.stack([synth.queries(w, l, B, Hq, device="cuda") for l in range(Lyr)]).contiguous()
    sl = torch.as_tensor(lens, device="cuda")
    whole = gpu.decode(-1, q, sl).clone()
    per = torch.stack([gpu.decode(l, q[l].contiguous(), sl).clone() for l in range(Lyr)])
    torch.cuda.synchronize()
    assert gpu.status() == 0
    scale = whole.abs().max().item()
    assert scale > 0
    err = (whole - per).abs().max().item()
    assert err <= 1e-4 * scale, f"all-layer vs per-layer calls: max |diff| {err:.3e} vs max |out| {scale:.3e}"


def test_sinkhorn_kvarn(gpu_lib):
    """Qwen3-4B KVarN-shaped (GQA 4) at small size: calibrate, append, decode."""
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k"]
    Lyr, H, Hq, L, n_cal = 2, 2, 8, 1300, 1024
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, 1, 1408, window=128, sinkhorn=True)
    for l in range(Lyr):
        k, v = _inputs(w, l, 1, H, Hq, L)
        kc, vc = k[0, :, :n_cal].contiguous(), v[0, :, :n_cal].contiguous()
        gpu.calibrate(l, kc, vc)
        ora.calibrate(l, harness.to_np(kc), harness.to_np(vc))
        gpu.append(l, k, v, torch.zeros(1, dtype=torch.int32, device="cuda"))
        ora.append(l, harness.to_np(k), harness.to_np(v), np.array([0]))
    torch.cuda.synchronize()
    sk, sv = layout.read_sigma(gpu.buffer, gpu.cfg)
    assert np.array_equal(sk.view(np.uint16), ora.sigma_k.view(np.uint16))
    assert np.array_equal(sv.view(np.uint16), ora.sigma_v.view(np.uint16))
    for l in range(Lyr):
        for h in range(H):
            harness.compare_codes(gpu, ora, l, 0, h, L)
        q = synth.queries(w, l, 1, Hq, device="cuda")
        got, want = _decode_both(gpu, ora, l, q, np.array([L]))
        harness.assert_attention_close(got, want)


def test_turboquant_keys(gpu_lib):
    """Llama-3.1-8B TurboQuant-shaped (GQA 4, B=2) at small size: TQ3+QJL keys, Q4 values."""
    w = synth.WORKLOADS["llama3.1-8b-tq-b8-32k"]
    Lyr, H, Hq, B, L = 2, 2, 8, 2, 900
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, B, 1024, window=128, k_format="tq3_qjl")
    for l in range(Lyr):
        k, v = _inputs(w, l, B, H, Hq, L)
        gpu.append(l, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
        ora.append(l, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    torch.cuda.synchronize()
    for l in range(Lyr):
        for b in range(B):
            for h in range(H):
                harness.compare_codes(gpu, ora, l, b, h, L)
        q = synth.queries(w, l, B, Hq, device="cuda")
        got, want = _decode_both(gpu, ora, l, q, np.array([L, L - 321]))
        harness.assert_attention_close(got, want)


@pytest.mark.parametrize("sinkhorn", [False, True])
def test_8bit_keys(gpu_lib, sinkhorn):
    """[TQ] "when to use what": K kept at 8 bits, V at 4 bits (GQA 3, B = 2, different lengths), plain
    and Sinkhorn-balanced: codes and scales bit-exact, attention within 2e-3."""
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k" if sinkhorn else "llama3.2-3b-32k-k8v4"]
    Lyr, H, Hq, B, L = 2, 2, 6, 2, 900
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, B, 1024, window=128, k_format="q8g32", sinkhorn=sinkhorn)
    for l in range(Lyr):
        k, v = _inputs(w, l, B, H, Hq, L)
        if sinkhorn:
            kc, vc = k[0, :, :512].contiguous(), v[0, :, :512].contiguous()
            gpu.calibrate(l, kc, vc)
            ora.calibrate(l, harness.to_np(kc), harness.to_np(vc))
        gpu.append(l, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
        ora.append(l, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    torch.cuda.synchronize()
    for l in range(Lyr):
        for b in range(B):
            for h in range(H):
                harness.compare_codes(gpu, ora, l, b, h, L)
        q = synth.queries(w, l, B, Hq, device="cuda")
        got, want = _decode_both(gpu, ora, l, q, np.array([L, L - 321]))
        harness.assert_attention_close(got, want)


@pytest.mark.parametrize("window", [128, 0])
def test_8bit_keys_ragged_edge_lengths(gpu_lib, window):
    """Q8 keys at the edge lengths of the step list (half-page tails, window boundaries, empty)."""
    lens = np.array([0, 1, 31, 32, 33, 127, 128, 129, 160, 191, 192, 700], dtype=np.int32)
    B = len(lens)
    w = synth.WORKLOADS["llama3.2-3b-32k-k8v4"]
    gpu, ora, _ = harness.make_pair(1, 2, 4, B, 768, window=window, k_format="q8g32")
    T = int(lens.max())
    k, v = _inputs(w, 0, B, 2, 4, T)
    gpu.append(0, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
    ora.append(0, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    torch.cuda.synchronize()
    q = synth.queries(w, 0, B, 4, device="cuda")
    got, want = _decode_both(gpu, ora, 0, q, lens)
    for b in range(B):
        if lens[b] == 0:
            assert not got[b].any()
        else:
            harness.assert_attention_close(got[b], want[b])


def test_paged_ragged_batch(gpu_lib):
    """dense-27B-shaped (GQA 2) paged cache: shuffled block table, chunked ragged prefill."""
    w = synth.WORKLOADS["dense27b-ragged-b32"]
    rng = np.random.default_rng(3)
    B, H, Hq, cap, chunk = 5, 2, 4, 2048, 256
    lens = rng.integers(100, 2000, B).astype(np.int32)
    maxpps = cap // 64
    need = [int(-(-L // 64)) for L in lens]
    n_pages = sum(need) + 3
    perm = rng.permutation(n_pages)
    bt = np.full((B, maxpps), -1, np.int32)
    o = 0
    for b in range(B):
        bt[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    gpu, ora, _ = harness.make_pair(1, H, Hq, B, cap, window=128, n_pages=n_pages, block_table=bt)
    T = int(lens.max())
    k, v = _inputs(w, 0, B, H, Hq, T)

    def app(t0, n, live):
        pos = np.array([t0 if b in live else -1 for b in range(B)], np.int32)
        kk, vv = k[:, :, t0:t0 + n].contiguous(), v[:, :, t0:t0 + n].contiguous()
        gpu.append(0, kk, vv, torch.as_tensor(pos, device="cuda"))
        ora.append(0, harness.to_np(kk), harness.to_np(vv), pos)

    for t0 in range(0, T, chunk):                      # full chunks, all sequences that have them
        live = {b for b in range(B) if lens[b] >= t0 + chunk}
        if live:
            app(t0, chunk, live)
    for b in range(B):                                  # each sequence's remainder on its own
        r0 = (int(lens[b]) // chunk) * chunk
        if lens[b] > r0:
            app(r0, int(lens[b]) - r0, {b})
    torch.cuda.synchronize()
    assert gpu.status() == 0
    for b in range(B):
        for h in range(H):
            harness.compare_codes(gpu, ora, 0, b, h, int(lens[b]), bt)
            harness.compare_ring(gpu, ora, 0, b, h, int(lens[b]))
    q = synth.queries(w, 0, B, Hq, device="cuda")
    got, want = _decode_both(gpu, ora, 0, q, lens)
    harness.assert_attention_close(got, want)


def test_out_of_range_append_is_flagged_and_skipped(gpu_lib):
    gpu, _, _ = harness.make_pair(1, 1, 2, 2, 256, window=128)
    before = gpu.buffer.clone()
    k = torch.ones(2, 1, 10, 128, dtype=torch.bfloat16, device="cuda")
    gpu.append(0, k, k, torch.tensor([250, -1], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert gpu.status() == 2                        # KVQ_DEV_POS_RANGE
    assert torch.equal(before, gpu.buffer)
    assert gpu.status() == 0                        # read-and-clear


@pytest.mark.parametrize("variant", ["bf16", "f32", "sinkhorn", "tq3_keys", "paged", "q8_keys", "q8_sinkhorn"])
def test_chunked_appends_at_odd_offsets(gpu_lib, variant):
    """Appends of 1..257 tokens starting at odd, even, half-page and page offsets, with sequences
    skipped (pos = -1) in some calls: every stored field of every written position and the window
    ring bit-exact with the oracle (covers both append kernels and the split between them)."""
    balanced = variant in ("sinkhorn", "q8_sinkhorn")
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k" if balanced else "llama3.2-3b-32k"]
    B, H, Hq, cap, W = 4, 2, 4, 1024, 64
    starts = np.array([0, 1, 31, 63], np.int32)
    chunks = [16, 1, 17, 31, 5, 32, 33, 100, 15, 257]
    bt, n_pages = None, 0
    if variant == "paged":
        maxpps = cap // 64
        n_pages = B * maxpps + 5
        perm = np.random.default_rng(5).permutation(n_pages)
        bt = perm[:B * maxpps].reshape(B, maxpps).astype(np.int32)
    gpu, ora, _ = harness.make_pair(1, H, Hq, B, cap, window=W, in_dtype="f32" if variant == "f32" else "bf16",
                                    sinkhorn=balanced,
                                    k_format={"tq3_keys": "tq3_qjl", "q8_keys": "q8g32",
                                              "q8_sinkhorn": "q8g32"}.get(variant, "q4g32"),
                                    n_pages=n_pages, block_table=bt)
    if balanced:
        kc, vc = _inputs(w, 0, 1, H, Hq, 256, t0=4096)
        gpu.calibrate(0, kc[0].contiguous(), vc[0].contiguous())
        ora.calibrate(0, harness.to_np(kc[0]), harness.to_np(vc[0]))
    pos = starts.copy()
    last_T = np.zeros(B, np.int64)
    t_in = 0
    for i, T in enumerate(chunks):
        k, v = _inputs(w, 0, B, H, Hq, T, t0=t_in, dtype=torch.float32 if variant == "f32" else None)
        t_in += T
        p = pos.copy()
        if i % 3 == 1:
            p[(i // 3) % B] = -1
        gpu.append(0, k, v, torch.as_tensor(p, device="cuda"))
        ora.append(0, harness.to_np(k), harness.to_np(v), p)
        live = p >= 0
        pos[live] += T
        last_T[live] = T
    torch.cuda.synchronize()
    assert gpu.status() == 0
    names = {"tq3_keys": (("k_code", "code"), ("k_bits", "bits"), ("k_norm", "norm"), ("k_gamma", "gamma")),
             "q8_keys": (("k_code", "code"), ("k_scale", "scale")),
             "q8_sinkhorn": (("k_code", "code"), ("k_scale", "scale"))}.get(
        variant, (("k_code", "code"), ("k_scale", "scale"), ("k_zero", "zero")))
    for b in range(B):
        s0, s1 = int(starts[b]), int(pos[b])
        for h in range(H):
            got = layout.read_unit(gpu.buffer, gpu.cfg, 0, b, h, s1, bt)
            for gname, oname in names:
                assert np.array_equal(got[gname][s0:s1].view(np.uint8),
                                      ora.k[oname][0, b, h, s0:s1].view(np.uint8)), (gname, b, h)
            for oname in ("code", "scale", "zero"):
                assert np.array_equal(got["v_" + oname][s0:s1].view(np.uint8),
                                      ora.v[oname][0, b, h, s0:s1].view(np.uint8)), ("v_" + oname, b, h)
            rk, rv = layout.read_ring(gpu.buffer, gpu.cfg, 0, b, h)
            slots = np.arange(s1 - min(W, int(last_T[b])), s1) % W
            assert np.array_equal(rk[slots].view(np.uint32), ora.ring_k[0, b, h, slots].view(np.uint32))
            assert np.array_equal(rv[slots].view(np.uint32), ora.ring_v[0, b, h, slots].view(np.uint32))


@pytest.mark.parametrize("k_format", ["q4g32", "q8g32"])
def test_bulk_append_degenerate_groups(gpu_lib, k_format):
    """Rotated groups whose codes clamp, whose zero overflows fp16, that are exactly zero, or that
    span many decades, through the bulk kernel (bf16 inputs, starts inside a block): codes, scales
    and zeros of K and V bit-exact with the oracle.

    With s the rotation's signs and e_j the unit vectors, x = beta * s (.) (e_0 + e_32 + e_64 + e_96)
    + gamma * s (.) e_1 rotates exactly to c (4 beta +- gamma) on channels 0..31 and c (+-gamma) on
    the rest: group 0 holds two values 2 c gamma apart around 4 c beta, so its fp16 zero misses its
    minimum by far more than its step when beta >> gamma (clamped codes), and overflows fp16 when
    |4 c beta| > 65504.  x = alpha * s rotates to one non-zero channel: groups 1..3 are all zero."""
    B, H, Hq, T = 2, 2, 4, 300
    gpu, ora, _ = harness.make_pair(1, H, Hq, B, 512, window=64, k_format=k_format)
    rng = np.random.default_rng(11)
    sg = ora.signs.astype(np.float64)
    xs = []
    for _ in range(2):  # K, then V
        x = rng.standard_normal((B, H, T, 128))
        for t in range(T):
            kind = t % 5
            if kind in (1, 2):
                beta = rng.uniform(100.0, 5000.0) if kind == 1 else -2.0e5
                gamma = float(rng.choice([0.5, 1.0, 2.0]))
                e = np.zeros(128)
                e[[0, 32, 64, 96]] = beta
                e[1] = gamma
                x[:, :, t] = sg * e
            elif kind == 3:
                x[:, :, t] *= np.exp(rng.uniform(-12.0, 12.0, (B, H, 128)))
            elif kind == 4:
                x[:, :, t] = 0.375 * sg
        xs.append(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16).cuda())
    k, v = xs
    p0 = np.array([3, 64], np.int64)
    gpu.append(0, k, v, torch.as_tensor(p0.astype(np.int32), device="cuda"))
    ora.append(0, harness.to_np(k), harness.to_np(v), p0)
    torch.cuda.synchronize()
    assert gpu.status() == 0
    names = (("k_code", "code"), ("k_scale", "scale")) + ((("k_zero", "zero"),) if k_format == "q4g32" else ())
    for b in range(B):
        s0 = int(p0[b])
        for h in range(H):
            got = layout.read_unit(gpu.buffer, gpu.cfg, 0, b, h, s0 + T)
            for gname, oname in names:
                assert np.array_equal(got[gname][s0:].view(np.uint8),
                                      ora.k[oname][0, b, h, s0:s0 + T].view(np.uint8)), (gname, b, h)
            for oname in ("code", "scale", "zero"):
                assert np.array_equal(got["v_" + oname][s0:].view(np.uint8),
                                      ora.v[oname][0, b, h, s0:s0 + T].view(np.uint8)), ("v_" + oname, b, h)
            harness.compare_ring(gpu, ora, 0, b, h, s0 + T)


def test_many_tiny_units(gpu_lib):
    """4096 (layer, sequence, kv-head) units of 0..5 tokens, a sixth of them empty: far more units
    than warps, so warps stream dozens of units each and most units have a single record."""
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, H, Hq, B = 2, 4, 12, 512
    lens = (np.arange(B) % 6).astype(np.int32)          # 0..5 tokens, window 4 (ring only for most)
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, B, 64, window=4)
    for l in range(Lyr):
        k, v = _inputs(w, l, B, H, Hq, 5)
        gpu.append(l, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
        ora.append(l, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    torch.cuda.synchronize()
    q = torch.stack([synth.queries(w, l, B, Hq, device="cuda") for l in range(Lyr)]).contiguous()
    sl = torch.as_tensor(lens, device="cuda")
    out = gpu.decode(-1, q, sl)
    torch.cuda.synchronize()
    assert gpu.status() == 0
    for l in range(Lyr):
        want = ora.decode(l, harness.to_np(q[l]), lens)
        harness.assert_attention_close(harness.to_np(out[l]), want)
    # a second call on the same, now used, scratch, then one on a scratch full of NaN patterns:
    # every call writes what it reads, so the results are identical
    out2 = gpu.decode(-1, q, sl)
    scratch = gpu.scratch(-1, B)
    scratch.fill_(0xFF)
    out3 = gpu.decode(-1, q, sl)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
    assert torch.equal(out.view(torch.int32), out3.view(torch.int32))
