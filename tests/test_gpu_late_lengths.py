"""Sequence lengths written by the kernel just before a decode call, while the decode's blocks are
already resident.

For Q4G32 and Q8G32 keys the decode computes its split of the work from the lengths before its
dependency wait and reads them again after it.  A helper kernel (tests/helpers/late_lengths.cu,
compiled here with nvcc) lets its programmatic dependents start at once and writes new lengths
2 ms later (longer than the host takes to launch the decode), so the decode launched right after
it sees the old lengths first.  Its output must
equal, bit for bit, a decode of the new lengths from a quiet start (same kernels, same split), and
match the oracle.
"""

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from kv_cache_quantization_append_gb300 import build, lib, synth

from . import harness

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("late_lengths") / "liblate_lengths.so")
    subprocess.run([build.nvcc(), *build.ARCH, "-O2", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "helpers", "late_lengths.cu"), "-o", so], check=True)
    h = ctypes.CDLL(so)
    h.launch_write_lengths_late.restype = ctypes.c_int
    h.launch_write_lengths_late.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong,
                                            ctypes.c_void_p]
    return h


@pytest.mark.parametrize("k_format", ["q4g32", "q8g32"])
def test_lengths_written_while_the_decode_starts(gpu_lib, helper, k_format):
    w = synth.WORKLOADS["llama3.2-3b-32k"]
    Lyr, B, H, Hq = 2, 3, 2, 6
    gpu, ora, _ = harness.make_pair(Lyr, H, Hq, B, 3072, window=128, k_format=k_format)
    for layer in range(Lyr):
        k, v = synth.kv_tokens(w, layer, B, H, 0, 3000, device="cuda")
        gpu.append(layer, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"))
        ora.append(layer, harness.to_np(k), harness.to_np(v), np.zeros(B, np.int64))
    q = torch.stack([synth.queries(w, layer, B, Hq, device="cuda") for layer in range(Lyr)]).contiguous()
    new = np.array([2900, 1234, 3000], np.int32)
    new_t = torch.as_tensor(new, device="cuda")
    ref = gpu.decode(-1, q, new_t.clone()).clone()
    torch.cuda.synchronize()
    assert gpu.status() == 0
    for old in ([100, 200, 300], [3000, 0, 17]):
        lens_t = torch.as_tensor(np.array(old, np.int32), device="cuda")
        out = torch.empty_like(ref)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream().cuda_stream
        assert helper.launch_write_lengths_late(lens_t.data_ptr(), new_t.data_ptr(), B, 2_000_000, stream) == 0
        gpu.decode(-1, q, lens_t, out)
        torch.cuda.synchronize()
        assert gpu.status() == 0
        assert torch.equal(lens_t.cpu(), new_t.cpu())
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), f"old lengths {old}"
    for layer in range(Lyr):
        want = ora.decode(layer, harness.to_np(q[layer]), new)
        harness.assert_attention_close(harness.to_np(ref[layer]), want)
