"""GPU parity of the block codecs (TBQ blocks, outlier-channel split) against the CPU oracle:
records (norms and code streams) and decoded values bit for bit, the outlier channels exactly."""

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import lib, synth
from oracle import blocks

pytestmark = pytest.mark.gpu


def _kv_rows(name, n_tokens, layer=0, dtype=None):
    """K rows of a workload's first kv-heads as [tokens][...], with its outlier channels."""
    w = synth.WORKLOADS[name]
    k, _ = synth.kv_tokens(w, layer, 1, w["n_kv_heads"], 0, n_tokens, device="cuda", dtype=dtype)
    return k[0]  # [H][T][128]


@pytest.mark.parametrize("bits", [3, 4])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_tbq_blocks_match_oracle(gpu_lib, bits, dtype):
    k = _kv_rows("llama3.2-3b-32k", 333, dtype=dtype)            # [8][333][128]
    rows = k.permute(1, 0, 2).reshape(-1, 256).contiguous()     # a token row = 8 heads: 4 blocks of 256
    nb = rows.shape[0]
    rec = torch.empty(nb, lib.kv_tbq_block_bytes(bits), dtype=torch.uint8, device="cuda")
    lib.kv_tbq_encode(bits, 11, rows, rec)
    out = torch.empty(nb, 256, dtype=torch.float32, device="cuda")
    lib.kv_tbq_decode(bits, 11, rec, out)
    torch.cuda.synchronize()
    x = rows.float().cpu().numpy()
    want = blocks.tbq_encode(x, bits, 11)
    got = rec.cpu().numpy()
    assert np.array_equal(got, want)
    dec = blocks.tbq_decode(want, bits, 11)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), dec.view(np.uint32))


def test_tbq_edge_blocks(gpu_lib):
    """A zero block, a constant block, tiny and large magnitudes, and a single block."""
    x = np.zeros((5, 256), np.float32)
    x[1] = 3.0
    x[2] = np.random.default_rng(0).standard_normal(256) * 1e-20
    x[3] = np.random.default_rng(1).standard_normal(256) * 1e3
    x[4, 17] = -2.5
    t = torch.as_tensor(x, device="cuda")
    for bits in (3, 4):
        rec = torch.empty(5, lib.kv_tbq_block_bytes(bits), dtype=torch.uint8, device="cuda")
        lib.kv_tbq_encode(bits, 0, t, rec)
        out = torch.empty(5, 256, dtype=torch.float32, device="cuda")
        lib.kv_tbq_decode(bits, 0, rec, out)
        torch.cuda.synchronize()
        want = blocks.tbq_encode(x, bits, 0)
        assert np.array_equal(rec.cpu().numpy(), want)
        assert np.array_equal(out.cpu().numpy().view(np.uint32), blocks.tbq_decode(want, bits, 0).view(np.uint32))


def test_split_outliers_match_oracle(gpu_lib):
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k"]                   # per-channel std log-uniform [0.1, 10]
    k, _ = synth.kv_tokens(w, 2, 1, 8, 0, 700, device="cuda")
    calib = k[0].contiguous()                                   # [8 sets][700][128] bf16
    got = torch.empty(8, 64, dtype=torch.int16, device="cuda")
    lib.kv_split_outliers(calib, got)
    torch.cuda.synchronize()
    c = calib.float().cpu().numpy()
    for s in range(8):
        assert np.array_equal(got[s].cpu().numpy(), blocks.split_outliers(c[s]))
    flat = torch.ones(1, 16, 128, dtype=torch.float32, device="cuda")   # all equal: the lowest 64
    lo = torch.empty(1, 64, dtype=torch.int16, device="cuda")
    lib.kv_split_outliers(flat, lo)
    torch.cuda.synchronize()
    assert np.array_equal(lo[0].cpu().numpy(), np.arange(64))


@pytest.mark.parametrize("hi_bits", [3, 4])
def test_split_records_match_oracle(gpu_lib, hi_bits):
    w = synth.WORKLOADS["qwen3-4b-kvarn-128k"]
    k, _ = synth.kv_tokens(w, 1, 1, 4, 0, 1000, device="cuda")
    x = k[0].contiguous()                                       # [4 sets][1000][128]
    outl = torch.empty(4, 64, dtype=torch.int16, device="cuda")
    lib.kv_split_outliers(x[:, :512].contiguous(), outl)
    rec = torch.empty(4 * 1000, lib.kv_split_record_bytes(hi_bits), dtype=torch.uint8, device="cuda")
    lib.kv_split_encode(hi_bits, 3, outl, x, rec)
    out = torch.empty(4, 1000, 128, dtype=torch.float32, device="cuda")
    lib.kv_split_decode(hi_bits, 3, outl, rec, out)
    torch.cuda.synchronize()
    xn = x.float().cpu().numpy()
    on = outl.cpu().numpy()
    got = rec.cpu().numpy().reshape(4, 1000, -1)
    dec = out.cpu().numpy()
    for s in range(4):
        want = blocks.split_encode(xn[s], on[s], hi_bits, 3)
        assert np.array_equal(got[s], want), f"set {s}"
        assert np.array_equal(dec[s].view(np.uint32), blocks.split_decode(want, on[s], hi_bits, 3).view(np.uint32))
