"""Full-size parity of the chunked prefill on sampled queries, in the configuration the benchmark times.

Each workload's cache is built exactly as bench.py builds it, then the bench's prefill call runs:
layer 0, the last T positions of every sequence rewritten by one chunk (the bench's T), every query
of the chunk attending over the whole context.  For a few (sequence, kv-head) units the CPU oracle
replays the definition: the unit's prefix positions from the same seeded inputs, then the chunk's
tokens appended in order, and at each sampled query t the single-token decode at length
pos + t + 1.  The GPU's outputs for those queries must be within 2e-3 of the oracle's max |out|, and
after the last sampled query (the chunk's last) every stored record of the unit must match bit for
bit.
"""

import numpy as np
import pytest
import torch

import bench
from kv_cache_quantization_append_gb300 import synth
from oracle import attention

from . import harness, layout

pytestmark = pytest.mark.gpu

# (sequence, kv-head) units and the chunk's query indices sampled, per workload
SAMPLES = {
    "llama3.1-8b-tq-b8-32k": ([(7, 7), (3, 2)], "first, middle, last"),
    "llama3.2-3b-32k": ([(0, 5)], "first, middle, last"),
    "dense27b-ragged-b32": ([(17, 9)], "first, last"),
}


def _query_indices(T, which):
    idx = {"first": 0, "middle": T // 2, "last": T - 1}
    return sorted({idx[s.strip()] for s in which.split(",")})


def _unit_tokens(w, layer, B, H, b, h, n):
    """Positions [0, n) of sequence b, kv-head h, as the cache build generated them (4096 at a time)."""
    ks, vs = [], []
    for t0 in range(0, n, 4096):
        k, v = synth.kv_tokens(w, layer, B, H, t0, min(4096, n - t0), device="cuda")
        ks.append(k[b, h].clone())
        vs.append(v[b, h].clone())
        del k, v
    return torch.cat(ks)[None, None], torch.cat(vs)[None, None]


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_prefill_sampled_queries(gpu_lib, name):
    torch.cuda.empty_cache()
    cache, w, layers, lens = bench.build_cache(name, "cuda")
    B, H, Hq = w["batch"], w["n_kv_heads"], w["n_q_heads"]
    g = Hq // H
    # the bench's prefill call (time_prefill): layer 0, chunk of T at pos = len - T.  The cache was
    # built through position len - 2, so its window ring holds the positions just before len - 1;
    # the definition wants the ring of the state "positions [0, pos) written": the W positions
    # before pos are appended again (identical records, the ring restored).
    T = min(bench.PREFILL_CHUNK.get(name, 1024), int(lens.min()))
    pos = (lens - T).astype(np.int32)
    W = w["window"]
    starts = sorted(set(int(max(0, p - W)) for p in pos))
    for s0 in starts:
        sel = [b for b in range(B) if max(0, int(pos[b]) - W) == s0]
        n = max(int(pos[b]) - s0 for b in sel)
        if n == 0:
            continue
        kk, vv = synth.kv_tokens(w, 0, B, H, s0, n, device="cuda")
        # sequences of this start needing all n positions in one call, the others one call each
        pa = np.full(B, -1, np.int32)
        for b in sel:
            if int(pos[b]) - s0 == n:
                pa[b] = s0
        cache.append(0, kk, vv, torch.as_tensor(pa, device="cuda"))
        for b in sel:
            m = int(pos[b]) - s0
            if m != n and m > 0:
                pb = np.full(B, -1, np.int32)
                pb[b] = s0
                cache.append(0, kk[:, :, :m].contiguous(), vv[:, :, :m].contiguous(), torch.as_tensor(pb, device="cuda"))
        del kk, vv
    torch.cuda.synchronize()
    assert cache.status() == 0
    k, v = synth.kv_tokens(w, 0, B, H, 0, T, device="cuda")
    q = synth.chunk_queries(w, 0, B, Hq, T, device="cuda")
    out = cache.prefill(0, k, v, q, torch.as_tensor(pos, device="cuda"))
    torch.cuda.synchronize()
    assert cache.status() == 0
    bt = None if cache.block_table is None else cache.block_table.cpu().numpy()
    proj = synth.qjl_projection(w["qjl_seed"]) if w["k_format"] == "tq3_qjl" else None
    units, which = SAMPLES[name]
    ts = _query_indices(T, which)
    for (b, h) in units:
        P = int(pos[b])
        ocfg = attention.OracleConfig(n_layers=1, n_kv_heads=1, n_q_heads=g, max_batch=1, max_seq_len=P + T,
                                      window=w["window"], k_format=harness.OFMT[w["k_format"]],
                                      sinkhorn=w["sinkhorn"], seed=w["wht_seed"])
        ora = attention.OracleCache(ocfg, proj)
        if w["sinkhorn"]:
            kc, vc = synth.kv_tokens(w, 0, 1, H, 0, w.get("calib_tokens", 1024), device="cuda")
            ora.calibrate(0, harness.to_np(kc[0, h:h + 1]), harness.to_np(vc[0, h:h + 1]))
        if P > 0:
            kp, vp = _unit_tokens(w, 0, B, H, b, h, P)
            ora.append(0, harness.to_np(kp), harness.to_np(vp), np.array([0]))
            del kp, vp
        kc_u = harness.to_np(k[b:b + 1, h:h + 1])
        vc_u = harness.to_np(v[b:b + 1, h:h + 1])
        done = 0  # chunk tokens appended to the oracle so far
        for t in ts:
            ora.append(0, kc_u[:, :, done:t + 1], vc_u[:, :, done:t + 1], np.array([P + done]))
            done = t + 1
            qg = harness.to_np(q[b, h * g:(h + 1) * g, t])
            want = ora.decode_unit(0, 0, 0, qg, P + t + 1)
            rel = harness.assert_attention_close(harness.to_np(out[b, h * g:(h + 1) * g, t]), want)
            print(f"{name} unit ({b}, {h}) query {t} of {T} at position {P + t}: max|err| / max|out| = {rel:.2e}")
        assert done == T
        # every stored record of the unit after the whole chunk
        L = P + T
        got = layout.read_unit(cache.buffer, cache.cfg, 0, b, h, L, bt)
        names = {"tq3_qjl": ("code", "bits", "norm", "gamma"), "q8g32": ("code", "scale")}.get(
            w["k_format"], ("code", "scale", "zero"))
        for n in names:
            assert np.array_equal(ora.k[n][0, 0, 0, :L].view(np.uint8), got["k_" + n].view(np.uint8)), f"k_{n}"
        for n in ("code", "scale", "zero"):
            assert np.array_equal(ora.v[n][0, 0, 0, :L].view(np.uint8), got["v_" + n].view(np.uint8)), f"v_{n}"
    del cache
    torch.cuda.empty_cache()
