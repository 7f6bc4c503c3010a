"""The seeded input generators shared by the GPU tests, the bench and the oracle's callers (CPU).

Parity tests regenerate any slice of a workload's context on both sides, so the draws must be
deterministic and slice-consistent; the workload recipe's stated figures are checked here too.
"""

import numpy as np
import torch

from kv_cache_quantization_append_gb300 import synth


def test_draws_are_deterministic():
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    a = synth.kv_tokens(w, 3, 2, 2, 0, 300)
    b = synth.kv_tokens(w, 3, 2, 2, 0, 300)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(synth.queries(w, 3, 2, 6, step=4), synth.queries(w, 3, 2, 6, step=4))
    assert not torch.equal(synth.queries(w, 3, 2, 6, step=4), synth.queries(w, 3, 2, 6, step=5))
    assert not torch.equal(a[0], synth.kv_tokens(w, 4, 2, 2, 0, 300)[0])      # per layer


def test_any_slice_regenerates_across_block_boundaries():
    w = synth.WORKLOADS["dense27b-ragged-b32"]
    k, v = synth.kv_tokens(w, 0, 2, 2, 0, 9000)
    for t0, T in ((0, 1), (4000, 200), (4095, 2), (8190, 810), (100, 8800)):
        ks, vs = synth.kv_tokens(w, 0, 2, 2, t0, T)
        assert torch.equal(ks, k[:, :, t0:t0 + T]) and torch.equal(vs, v[:, :, t0:t0 + T])


def test_dtypes_and_shapes():
    tiny = synth.WORKLOADS["tiny"]
    k, v = synth.kv_tokens(tiny, 0, 1, 1, 0, 512)
    assert k.dtype == torch.float32 and k.shape == (1, 1, 512, 128) and v.shape == k.shape
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    k, _ = synth.kv_tokens(w, 0, 1, 8, 0, 16)
    assert k.dtype == torch.bfloat16 and k.is_contiguous()
    assert synth.queries(w, 0, 1, 24).shape == (1, 24, 128)


def test_ragged_length_recipe():
    """numpy default_rng(7).integers(1024, 65537, 32): sum 1,135,994, from 1,363 to 64,921."""
    lens = synth.ragged_lengths(*synth.WORKLOADS["dense27b-ragged-b32"]["ctx_range"], n=32, seed=7)
    assert lens.dtype == np.int32 and len(lens) == 32
    assert int(lens.sum()) == 1_135_994 and int(lens.min()) == 1_363 and int(lens.max()) == 64_921


def test_outlier_channels():
    """x % of the 128 channels = round(x * 128) per (layer, kv-head), scaled in K (and V where the
    recipe says so); the tiny workload scales K channels 0-3 by 10 and leaves V alone."""
    assert synth.n_outliers(synth.WORKLOADS["llama3.2-3b-32k"]) == 3
    assert synth.n_outliers(synth.WORKLOADS["dense27b-ragged-b32"]) == 1
    assert synth.n_outliers(synth.WORKLOADS["llama3.1-8b-tq-b8-32k"]) == 4
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    for which in ("k", "v"):
        sc = synth.channel_scales(w, 5, 8, which)
        assert sc.shape == (8, 128)
        assert torch.all((sc == 8.0).sum(1) == 3) and torch.all((sc == 1.0).sum(1) == 125)
    tiny = synth.WORKLOADS["tiny"]
    sk = synth.channel_scales(tiny, 0, 1, "k")
    assert torch.equal(torch.nonzero(sk[0] == 10.0).flatten(), torch.arange(4))
    assert torch.all(synth.channel_scales(tiny, 0, 1, "v") == 1.0)
    q = synth.WORKLOADS["qwen3-4b-kvarn-128k"]
    sq = synth.channel_scales(q, 2, 8, "k")
    assert float(sq.min()) >= 0.1 and float(sq.max()) <= 10.0 and float(sq.std()) > 1.0


def test_qjl_projection_is_standard_gaussian():
    s = synth.qjl_projection(4242)
    assert s.dtype == np.float32 and s.shape == (128, 128)
    assert np.array_equal(s, synth.qjl_projection(4242))
    assert abs(float(s.mean())) < 0.02 and abs(float(s.std()) - 1.0) < 0.02
