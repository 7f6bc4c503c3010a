"""Full-size parity on sampled units, in the launch configuration the benchmark times.

Each workload's cache is built exactly as bench.py builds it (all layers, full context, the same
seeded inputs, the same block table for the paged workload), the newest token of every layer is
appended and one decode launch covers all layers.  A few (layer, sequence, kv-head) units are then
recomputed by the CPU oracle from the same inputs: every stored code, scale, zero, norm, sign bit,
Sinkhorn scale and ring value of the unit must match bit for bit, and its attention outputs must be
within 2e-3 of the oracle's max |out|, from the all-layer call and from a per-layer call alike.
"""

import numpy as np
import pytest
import torch

import bench
from kv_cache_quantization_append_gb300 import synth
from oracle import attention

from . import harness, layout

pytestmark = pytest.mark.gpu

SAMPLES = {
    "llama3.2-3b-32k": [(0, 0, 0), (27, 0, 7), (13, 0, 3)],
    "qwen3-4b-kvarn-128k": [(35, 0, 5), (0, 0, 0)],
    "llama3.1-8b-tq-b8-32k": [(31, 7, 7), (4, 3, 2)],
    "dense27b-ragged-b32": [(0, 0, 0), (0, 17, 9), (0, 31, 15)],
    "llama3.2-3b-32k-k8v4": [(0, 0, 0), (27, 0, 7)],
}


def _unit_tokens(w, layer, B, H, b, h, n):
    """Positions [0, n) of sequence b, kv-head h, generated a 4096-token block at a time (the
    generator draws whole blocks, so this equals slicing one large call)."""
    ks, vs = [], []
    for t0 in range(0, n, 4096):
        k, v = synth.kv_tokens(w, layer, B, H, t0, min(4096, n - t0), device="cuda")
        ks.append(k[b, h].clone())
        vs.append(v[b, h].clone())
        del k, v
    return torch.cat(ks)[None, None], torch.cat(vs)[None, None]


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_size_sampled_units(gpu_lib, name):
    torch.cuda.empty_cache()
    cache, w, layers, lens = bench.build_cache(name, "cuda")
    B, H, Hq = w["batch"], w["n_kv_heads"], w["n_q_heads"]
    g = Hq // H
    # the benchmark's step: newest token of every layer, then one decode launch over all layers
    kvs = [synth.kv_tokens(w, l, B, H, int(lens.max()) - 1, 1, device="cuda") for l in range(layers)]
    knew = torch.stack([k for k, _ in kvs]).contiguous()
    vnew = torch.stack([v for _, v in kvs]).contiguous()
    pos = torch.as_tensor((lens - 1).astype(np.int32), device="cuda")
    cache.append(-1, knew, vnew, pos)
    q = torch.stack([synth.queries(w, l, B, Hq, device="cuda") for l in range(layers)]).contiguous()
    out = cache.decode(-1, q, torch.as_tensor(lens.astype(np.int32), device="cuda"))
    torch.cuda.synchronize()
    assert cache.status() == 0
    bt = None if cache.block_table is None else cache.block_table.cpu().numpy()
    proj = synth.qjl_projection(w["qjl_seed"]) if w["k_format"] == "tq3_qjl" else None
    lens_t = torch.as_tensor(lens.astype(np.int32), device="cuda")
    per_layer = {}  # layer -> output of a per-layer decode call
    for (layer, b, h) in SAMPLES[name]:
        L = int(lens[b])
        ocfg = attention.OracleConfig(n_layers=1, n_kv_heads=1, n_q_heads=g, max_batch=1, max_seq_len=L,
                                      window=w["window"], k_format=harness.OFMT[w["k_format"]],
                                      sinkhorn=w["sinkhorn"],
                                      seed=w["wht_seed"])
        ora = attention.OracleCache(ocfg, proj)
        if w["sinkhorn"]:
            kc, vc = synth.kv_tokens(w, layer, 1, H, 0, w.get("calib_tokens", 1024), device="cuda")
            ora.calibrate(0, harness.to_np(kc[0, h:h + 1]), harness.to_np(vc[0, h:h + 1]))
            sk, sv = layout.read_sigma(cache.buffer, cache.cfg)
            assert np.array_equal(sk[layer, h].view(np.uint16), ora.sigma_k[0, 0].view(np.uint16))
            assert np.array_equal(sv[layer, h].view(np.uint16), ora.sigma_v[0, 0].view(np.uint16))
        # the unit's inputs: prefill positions [0, L-1) from the blocks of 4096, plus the newest token
        k, v = _unit_tokens(w, layer, B, H, b, h, L - 1)
        ku = torch.cat([k, knew[layer, b:b + 1, h:h + 1]], dim=2)
        vu = torch.cat([v, vnew[layer, b:b + 1, h:h + 1]], dim=2)
        del k, v
        ora.append(0, harness.to_np(ku), harness.to_np(vu), np.array([0]))
        got = layout.read_unit(cache.buffer, cache.cfg, layer, b, h, L, bt)
        names = {"tq3_qjl": ("code", "bits", "norm", "gamma"), "q8g32": ("code", "scale")}.get(
            w["k_format"], ("code", "scale", "zero"))
        for n in names:
            wv, gv = ora.k[n][0, 0, 0, :L], got["k_" + n]
            assert np.array_equal(wv.view(np.uint8), gv.view(np.uint8)), f"{name} {layer},{b},{h} k_{n}"
        for n in ("code", "scale", "zero"):
            wv, gv = ora.v[n][0, 0, 0, :L], got["v_" + n]
            assert np.array_equal(wv.view(np.uint8), gv.view(np.uint8)), f"{name} {layer},{b},{h} v_{n}"
        rk, rv = layout.read_ring(cache.buffer, cache.cfg, layer, b, h)
        W = w["window"]
        slots = np.arange(max(0, L - W), L) % W
        assert np.array_equal(rk[slots].view(np.uint32), ora.ring_k[0, 0, 0, slots].view(np.uint32))
        assert np.array_equal(rv[slots].view(np.uint32), ora.ring_v[0, 0, 0, slots].view(np.uint32))
        qg = harness.to_np(q[layer, b, h * g:(h + 1) * g])
        want = ora.decode_unit(0, 0, 0, qg, L)
        rel = harness.assert_attention_close(harness.to_np(out[layer, b, h * g:(h + 1) * g]), want)
        # the same unit through a per-layer call (one layer's units spread over the whole grid: the
        # CTA-per-head merge for the single-sequence workloads)
        if layer not in per_layer:
            per_layer[layer] = cache.decode(layer, q[layer].contiguous(), lens_t)
            torch.cuda.synchronize()
            assert cache.status() == 0
        rel_l = harness.assert_attention_close(harness.to_np(per_layer[layer][b, h * g:(h + 1) * g]), want)
        print(f"{name} unit ({layer}, {b}, {h}) L={L}: max|err| / max|out| = {rel:.2e} "
              f"(per-layer call {rel_l:.2e})")
    del cache
    torch.cuda.empty_cache()
