"""Benchmark of one decode step of quantized-KV attention plus the append of one token per layer.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Default workload: the largest single-GPU configuration, a Llama-3.1-8B-shaped TurboQuant cache
(32 layers, 32 query / 8 kv heads, 8 sequences of 32768 tokens, 3-bit Lloyd-Max keys with a 1-bit
QJL residual sketch, 4-bit group-32 values, 128-token FP32 window; 10.2 GB streamed per step).
One step = append the newest token of every layer (one launch over all layers) + decode attention
over every layer (one streaming launch over all layers, then a small launch that merges the
partial softmax states).  Every cache is larger than L2, so every step streams it from HBM.

Prints one JSON line.  ``value`` = cached tokens attended per second, device-timed with CUDA events
over K steps on resident inputs; ``e2e`` = the same through the public API with every step's inputs
copied from pinned host memory and its output copied back inside the timed region (the copies on
their own streams, overlapping the neighbouring steps' compute as a serving loop would).  ``roofline``
is the decode call alone, timed over at least one second of back-to-back calls.  ``workloads``
carries the same decode roofline, the per-layer call form and the bulk (prefill-sized) append for
the other large configurations (Llama-3.2-3B at 32K, Qwen3-4B KVarN at 128K, the ragged 27B-class
batch), each built and measured after the headline one.
With --impl reference the CPU oracle is timed instead (a bounded sample of each step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # the CPU oracle is timed on one core
os.environ.setdefault("OMP_NUM_THREADS", "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_quantization_append_gb300 import QuantKVCache, lib, synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
# the largest configuration that fits one GPU (10.2 GB streamed per step) is the headline; the other
# large configurations are measured after it in the same run
HEADLINE_WORKLOAD = "llama3.1-8b-tq-b8-32k"
OTHER_WORKLOADS = ("llama3.2-3b-32k", "qwen3-4b-kvarn-128k", "dense27b-ragged-b32", "llama3.2-3b-32k-k8v4")
# bytes of one key record (a 128-value vector) per key format; a Q4G32 value record is 80 B
K_RECORD_BYTES = {"q4g32": 80, "tq3_qjl": 68, "q8g32": 136}
DTYPE_NAMES = {"q4g32": "q4/fp16-mma,f32-accum", "tq3_qjl": "tq3+qjl/q4,f32-accum", "q8g32": "q8/q4,fp16-mma,f32-accum"}
PROFILES = os.path.join(ROOT, "profiles")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    for f in ("decode.cu", "kvq_internal.cuh"):
        with open(os.path.join(ROOT, "kv_cache_quantization_append_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for key in ("hbm_gbs", "hbm_GBps", "hbm_bandwidth_gbs"):
                if key in d:
                    return float(d[key]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_traffic(workload: str):
    """dram read+write bytes per decode launch from the committed ncu summary, if the kernel
    source is unchanged since that capture (else None)."""
    p = os.path.join(PROFILES, "decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except ValueError:
        return None
    e = d.get(workload)
    if not e or e.get("kernel_source_sha") != kernel_source_sha():
        return None
    return e.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling (200 ms) during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ------------------------------------------------------------------ workload set-up
def workload_cfg(name: str, batch=None):
    w = synth.WORKLOADS[name]
    layers = w.get("alloc_layers", w["n_layers"])
    if "ctx_range" in w:
        lens = synth.ragged_lengths(*w["ctx_range"], n=w["batch"], seed=w["len_seed"])
    else:
        lens = np.full(w["batch"], w["ctx"], np.int32)
    if batch is not None and batch < w["batch"]:
        w = dict(w, batch=batch)
        lens = lens[:batch]
    return w, layers, lens


def build_cache(name: str, device="cuda", batch=None):
    """Allocate and prefill the cache of a workload; returns (cache, w, layers, lens).  ``batch``
    keeps only the first sequences of the workload (a smaller case for profiler captures)."""
    w, layers, lens = workload_cfg(name, batch)
    B, H, Hq = w["batch"], w["n_kv_heads"], w["n_q_heads"]
    cap = int(-(-(int(lens.max()) + 64) // 64) * 64)
    kf = lib.K_FORMATS[w["k_format"]]
    bt = None
    n_pages = 0
    if w.get("page_tokens"):
        # paged pool sized to the real lengths (+ one prefill chunk per sequence), shuffled
        extra = w.get("prefill_chunk", 0)
        cap = int(-(-(int(lens.max()) + extra + 64) // 64) * 64)
        maxpps = cap // 64
        need = [int(-(-(int(L) + extra) // 64)) for L in lens]
        n_pages = sum(need)
        perm = np.random.default_rng(11).permutation(n_pages)
        table = np.full((B, maxpps), 0, np.int32)
        o = 0
        for b in range(B):
            table[b, :need[b]] = perm[o:o + need[b]]
            o += need[b]
        bt = torch.as_tensor(table, device=device).contiguous()
    proj = synth.qjl_projection(w["qjl_seed"]) if kf == lib.KVQ_TQ3_QJL else None
    cfg = lib.make_config(layers, H, Hq, B, cap, window=w["window"], n_pages=n_pages, k_format=kf,
                          sinkhorn=w["sinkhorn"], in_dtype=lib.KVQ_IN_BF16 if w["in_dtype"] == "bf16" else lib.KVQ_IN_F32,
                          seed=w["wht_seed"])
    cache = QuantKVCache(cfg, device, bt, proj)
    # prefill positions [0, L_b - 1) in chunks; the newest token is written by every step
    T_pre = lens - 1
    chunk = 4096
    for layer in range(layers):
        if w["sinkhorn"]:
            n_cal = w.get("calib_tokens", 1024)
            kc, vc = synth.kv_tokens(w, layer, 1, H, 0, n_cal, device=device)
            cache.calibrate(layer, kc[0].contiguous(), vc[0].contiguous())
        for t0 in range(0, int(T_pre.max()), chunk):
            n = min(chunk, int(T_pre.max()) - t0)
            full = T_pre >= t0 + n
            k, v = synth.kv_tokens(w, layer, B, H, t0, n, device=device)
            if full.any():
                pos = torch.as_tensor(np.where(full, t0, -1).astype(np.int32), device=device)
                cache.append(layer, k, v, pos)
            for b in np.nonzero(~full & (T_pre > t0))[0]:
                m = int(T_pre[b]) - t0
                pos = torch.as_tensor(np.where(np.arange(B) == b, t0, -1).astype(np.int32), device=device)
                cache.append(layer, k[:, :, :m].contiguous(), v[:, :, :m].contiguous(), pos)
    torch.cuda.synchronize()
    if cache.status() != 0:
        raise RuntimeError("device status set during prefill")
    return cache, w, layers, lens


def bulk_append_bytes(w, layers, T) -> int:
    """Bytes an append of T tokens per sequence must move: the K and V inputs, the packed records
    (K 80 B or 68 B for TQ3 keys, V 80 B per token and kv-head) and the FP32 window copy of the
    last min(window, T) tokens (512 B each of K and V)."""
    inb = 2 if w["in_dtype"] == "bf16" else 4
    rec = K_RECORD_BYTES[w["k_format"]] + 80
    per_seq_head = T * (2 * 128 * inb + rec) + min(w["window"], T) * 1024
    return layers * w["batch"] * w["n_kv_heads"] * per_seq_head


def launches_per_step(w):
    """Kernels one timed step launches: the append (TurboQuant keys: a keys kernel and a values
    kernel; otherwise one kernel for both), then the decode kernel and its merge kernel."""
    return (2 if w["k_format"] == "tq3_qjl" else 1) + 2


def bench_config(name, w, layers, lens, world) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    cfg = {"workload": name, "layers": layers, "batch": int(w["batch"]),
           "n_q_heads": w["n_q_heads"], "n_kv_heads": w["n_kv_heads"], "seq_len_sum": int(lens.sum()),
           "window": w["window"], "k_format": w["k_format"], "v_format": w["v_format"],
           "sinkhorn": bool(w["sinkhorn"]), "parallelism": f"replicas x{world}",
           "l2": f"{algorithmic_bytes(w, layers, lens) / 1e9:.2f} GB of cache streamed each step (> 126 MB L2)"}
    if layers < w["n_layers"]:
        # only `layers` of the model's layers are allocated and timed; the whole-model step repeats
        # the same per-layer work
        cfg["timed_layers"] = layers
        cfg["model_layers"] = w["n_layers"]
    return cfg


def algorithmic_bytes(w, layers, lens) -> int:
    """Bytes the decode step must move: packed records of the quantised tokens, the FP32 window,
    q and out (per launch over all layers)."""
    W = w["window"]
    rec = K_RECORD_BYTES[w["k_format"]] + 80
    H, Hq = w["n_kv_heads"], w["n_q_heads"]
    per_layer = 0
    for L in lens:
        L = int(L)
        Lq = max(0, L - W) if W > 0 else L
        per_layer += H * (Lq * rec + (L - Lq) * 1024)
    per_layer += len(lens) * Hq * 128 * (2 + 4)
    return per_layer * layers


# ------------------------------------------------------------------ ranks
def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group (x itself without one):
    every rank's timed region ends when the slowest rank's does."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_step_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: the cached tokens every rank's replica attends per step, summed over
    the ranks, over the slowest rank's time per step."""
    return tokens_per_step_per_rank * world / (ms_per_step_max / 1e3)


# ------------------------------------------------------------------ GPU arm
DECODE_ROOFLINE_MIN_S = 1.0   # the decode-only pass runs at least this long, whatever --steps is
BULK_APPEND_REPS = 10
# FP32 rate of interleaved packed multiplies and adds (mul.rn.f32x2 / add.rn.f32x2, each half rounded
# like the scalar operation), measured on a GB300 with independent chains: 236.5 results per SM
# clock, 74.4 Tops/s over 152 SMs at 2070 MHz (scalar adds alone: 120 per clock)
FP32_PAIR_PEAK_TOPS = 74.4


def step_inputs(w, layers, lens, dev, nbuf=8):
    """Per-step inputs of a workload: ``nbuf`` rotating query sets [L][B][Hq][128], the newest token
    of every layer and sequence [L][B][Hkv][1][128] (K and V), its positions and the lengths."""
    B, H, Hq = w["batch"], w["n_kv_heads"], w["n_q_heads"]
    qs = [torch.stack([synth.queries(w, l, B, Hq, step=i, device=dev) for l in range(layers)]) for i in range(nbuf)]
    kvs = [synth.kv_tokens(w, l, B, H, int(lens.max()) - 1, 1, device=dev) for l in range(layers)]
    knew = torch.stack([k for k, _ in kvs]).contiguous()
    vnew = torch.stack([v for _, v in kvs]).contiguous()
    pos = torch.as_tensor((lens - 1).astype(np.int32), device=dev)
    seq = torch.as_tensor(lens.astype(np.int32), device=dev)
    return qs, knew, vnew, pos, seq


def time_decode_only(cache, qs, seq, out, steps, warmup, stream, min_s=DECODE_ROOFLINE_MIN_S):
    """Average duration of one all-layer decode call (the streaming launch and its merge launch),
    from CUDA events around at least DECODE_ROOFLINE_MIN_S seconds of back-to-back calls (and at
    least ``steps`` calls).  Returns (microseconds per call, calls timed)."""
    nbuf = len(qs)
    for i in range(warmup):
        cache.decode(-1, qs[i % nbuf], seq, out)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(3):
        cache.decode(-1, qs[i % nbuf], seq, out)
    e1.record(stream)
    torch.cuda.synchronize()
    est_s = e0.elapsed_time(e1) / 3 / 1e3
    n = max(steps, int(np.ceil(min_s / max(est_s, 1e-6))))
    e0.record(stream)
    for i in range(n):
        cache.decode(-1, qs[i % nbuf], seq, out)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n * 1e3, n


def time_per_layer_graph(cache, qs, seq, out, layers, steps, warmup, stream):
    """The second form of the decode step: one decode call per layer (two launches each), the calls
    of a step captured in one CUDA graph and replayed.  The first calls, outside the capture,
    allocate the per-layer scratch and set the kernels' attributes.  Seconds per step."""
    q0 = qs[0].contiguous()
    ql = [q0[l] for l in range(layers)]
    ol = [out[l] for l in range(layers)]
    for l in range(layers):
        cache.decode(l, ql[l], seq, ol[l])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for l in range(layers):
            cache.decode(l, ql[l], seq, ol[l])
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    del graph
    return g0.elapsed_time(g1) / steps / 1e3


def time_bulk_append(cache, w, layers, lens, dev, stream, peak, peak_src):
    """Bulk (prefill-sized) append: the workload's prefill chunk written at the end of every sequence
    where the workload names one (the cache has room for it), else a rewrite of positions
    [0, 4096) of every layer from the same seeded inputs (identical page bytes; the window ring then
    holds those positions, so nothing decodes after it)."""
    B, H = w["batch"], w["n_kv_heads"]
    Tc = int(w.get("prefill_chunk", 4096))
    if w.get("prefill_chunk"):
        kc, vc = synth.kv_tokens(w, 0, B, H, 0, Tc, device=dev)
        kc = torch.stack([kc] * layers) if layers > 1 else kc
        vc = torch.stack([vc] * layers) if layers > 1 else vc
        pos_c = torch.as_tensor(lens.astype(np.int32), device=dev)
    else:
        kl = [synth.kv_tokens(w, l, B, H, 0, Tc, device=dev) for l in range(layers)]
        kc = torch.stack([k for k, _ in kl]).contiguous()
        vc = torch.stack([v for _, v in kl]).contiguous()
        del kl
        pos_c = torch.zeros(B, dtype=torch.int32, device=dev)
    lay = -1 if layers > 1 else 0
    for _ in range(3):
        cache.append(lay, kc, vc, pos_c)
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(BULK_APPEND_REPS):
        cache.append(lay, kc, vc, pos_c)
    a1.record(stream)
    torch.cuda.synchronize()
    if cache.status() != 0:
        raise RuntimeError("device status set during the bulk append")
    a_s = a0.elapsed_time(a1) / BULK_APPEND_REPS / 1e3
    a_bytes = bulk_append_bytes(w, layers, Tc)
    bulk = "append_bulk_bf16_kernel" if w["in_dtype"] == "bf16" else "append_bulk_kernel"
    res = {"tokens_per_sequence": Tc, "us": a_s * 1e6, "algorithmic_bytes": a_bytes,
           "achieved_gbs": a_bytes / a_s / 1e9, "tokens_per_s": layers * B * Tc / a_s,
           "kernel": f"append_tq_keys_kernel + {bulk} (values)" if w["k_format"] == "tq3_qjl" else bulk}
    res["roofline"] = {"bound": "hbm", "achieved": res["achieved_gbs"], "peak": peak, "unit": "GB/s",
                       "frac": res["achieved_gbs"] / peak, "peak_source": peak_src}
    if w["k_format"] == "tq3_qjl":
        # TurboQuant keys: the QJL projection (128 x 128 separately rounded products and sums per key,
        # in the codec's order) bounds the keys kernel on the FP32 pipes, not on HBM
        ops = float(layers * B * H * Tc) * 2 * 128 * 128
        res["roofline_keys"] = {
            "bound": "alu", "achieved": ops / a_s / 1e12, "peak": FP32_PAIR_PEAK_TOPS, "unit": "Tops/s",
            "frac": ops / a_s / 1e12 / FP32_PAIR_PEAK_TOPS, "peak_source": "measured (packed fp32 multiply/add)",
            "note": "projection operations over the whole append call (keys and values kernels): a lower "
                    "bound for the keys kernel's own rate"}
    return res


PREFILL_CHUNK = {"llama3.1-8b-tq-b8-32k": 1024, "llama3.2-3b-32k": 2048, "llama3.2-3b-32k-k8v4": 2048,
                 "qwen3-4b-kvarn-128k": 1024, "dense27b-ragged-b32": 1024}
PREFILL_REPS = 2


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            if "bf16_tflops" in d:
                return float(d["bf16_tflops"]), "measured"
        except (OSError, ValueError):
            pass
    return 1900.0, "fallback"


def time_prefill(name, cache, w, layers, lens, dev, stream):
    """Chunked prefill of layer 0: the last T positions of every sequence rewritten by one
    kv_prefill_attention call (append + attention of the chunk's T queries over the whole context).
    Reported with the method's multiply-adds per (query head, attended position): key width
    (128; 256 for TQ3 keys, codes and QJL signs) for the logits + 128 for P.V; the tensor-core
    work executed is three times that (fp16 hi/lo products)."""
    B, H, Hq = w["batch"], w["n_kv_heads"], w["n_q_heads"]
    T = min(PREFILL_CHUNK.get(name, 1024), int(lens.min()))
    pos_np = (lens - T).astype(np.int32)
    k, v = synth.kv_tokens(w, 0, B, H, 0, T, device=dev)
    q = synth.chunk_queries(w, 0, B, Hq, T, device=dev)
    pos = torch.as_tensor(pos_np, device=dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    lay = 0
    cache.prefill(lay, k, v, q, pos, out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(PREFILL_REPS):
        cache.prefill(lay, k, v, q, pos, out)
    e1.record(stream)
    torch.cuda.synchronize()
    if cache.status() != 0:
        raise RuntimeError("device status set during the prefill timing")
    s = e0.elapsed_time(e1) / PREFILL_REPS / 1e3
    kd = 256 if w["k_format"] == "tq3_qjl" else 128
    attended = float(sum(int(T) * int(p) + T * (T + 1) / 2 for p in pos_np))   # per (query head): sum over t of pos + t + 1
    flops = 2.0 * (kd + 128) * attended * Hq
    # products executed per method multiply-add: 3 (hi/lo splits), except TQ3 keys' centroid half,
    # whose fp16 centroids are exact (2: the query's hi and lo)
    exec_macs = (2 * 128 + 3 * 128 + 3 * 128) if w["k_format"] == "tq3_qjl" else 3 * (kd + 128)
    peak, src = bf16_peak()
    achieved = 2.0 * exec_macs * attended * Hq / s / 1e12
    return {"layers": 1, "tokens_per_sequence": int(T), "us": s * 1e6, "tokens_per_s": B * T / s,
            "algorithmic_tflops": flops / s / 1e12,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": src,
                         "note": "executed fp16 tcgen05 products (hi/lo splits: 3 per method multiply-add, 2 "
                                 "for TQ3 keys' exact centroids) against the measured dense bf16 GEMM rate"},
            "kernels": "snapshot_kernel + append kernels + prefill_kernel"}


CODEC_BLOCKS = 1 << 21        # 256-value TBQ blocks timed (2^29 bf16 values: 1 GiB in)
CODEC_REPS = 5


def time_block_codecs(dev, stream):
    """Encode and decode throughput of the block codecs on seeded bf16 N(0,1) data (1 GiB in): TBQ3 /
    TBQ4 blocks and the 2.5 / 3.5-bit outlier split (64 sets, outliers from each set's first 1024
    vectors).  Algorithmic bytes = the input read + the output written."""
    g = torch.Generator(device=dev)
    g.manual_seed(424242)
    x = torch.randn(CODEC_BLOCKS, 256, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    peak, src = hbm_peak()
    res = {}

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(CODEC_REPS):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / CODEC_REPS / 1e3

    def entry(nbytes, s):
        gbs = nbytes / s / 1e9
        return {"us": s * 1e6, "achieved_gbs": gbs, "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak,
                                                                  "unit": "GB/s", "frac": gbs / peak, "peak_source": src}}

    for bits in (3, 4):
        rb = lib.kv_tbq_block_bytes(bits)
        blk = torch.empty(CODEC_BLOCKS, rb, dtype=torch.uint8, device=dev)
        out = torch.empty(CODEC_BLOCKS, 256, dtype=torch.float32, device=dev)
        se = timed(lambda: lib.kv_tbq_encode(bits, 0, x, blk))
        sd = timed(lambda: lib.kv_tbq_decode(bits, 0, blk, out))
        res[f"tbq{bits}_encode"] = entry(CODEC_BLOCKS * (512 + rb), se)
        res[f"tbq{bits}_decode"] = entry(CODEC_BLOCKS * (rb + 1024), sd)
        del blk, out
    xv = x.view(64, -1, 128)
    nv = xv.shape[0] * xv.shape[1]
    outl = torch.empty(64, 64, dtype=torch.int16, device=dev)
    lib.kv_split_outliers(xv[:, :1024].contiguous(), outl)
    for hi in (3, 4):
        rb = lib.kv_split_record_bytes(hi)
        rec = torch.empty(nv, rb, dtype=torch.uint8, device=dev)
        out = torch.empty(xv.shape, dtype=torch.float32, device=dev)
        se = timed(lambda: lib.kv_split_encode(hi, 0, outl, xv, rec))
        sd = timed(lambda: lib.kv_split_decode(hi, 0, outl, rec, out))
        res[f"split{hi - 0.5:g}bit_encode"] = entry(nv * (256 + rb), se)
        res[f"split{hi - 0.5:g}bit_decode"] = entry(nv * (rb + 512), sd)
        del rec, out
    del x
    torch.cuda.empty_cache()
    return res


def decode_roofline(name, w, layers, lens, dec_us, calls):
    peak, peak_src = hbm_peak()
    alg = algorithmic_bytes(w, layers, lens)
    achieved = alg / (dec_us / 1e6) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": peak_src, "traffic": measured_traffic(name), "algorithmic_bytes_per_launch": alg,
            "kernel": "decode call: decode_kernel (all layers) + merge_kernel", "decode_us_avg": dec_us,
            "calls_timed": calls}


def measure_other_workload(name, args, dev, stream):
    """Decode roofline, per-layer call form and bulk append of one more workload (built, measured
    and freed here)."""
    cache, w, layers, lens = build_cache(name, dev)
    qs, _, _, _, seq = step_inputs(w, layers, lens, dev)
    out = torch.empty(layers, w["batch"], w["n_q_heads"], 128, dtype=torch.float32, device=dev)
    dec_us, calls = time_decode_only(cache, qs, seq, out, args.steps, args.warmup, stream, args.decode_min_s)
    if cache.status() != 0:
        raise RuntimeError(f"device status set during the decode timing of {name}")
    res = {"config": bench_config(name, w, layers, lens, 1),
           "roofline": decode_roofline(name, w, layers, lens, dec_us, calls),
           "tokens_per_s_decode": float(lens.sum()) / (dec_us / 1e6)}
    if layers > 1:
        g_s = time_per_layer_graph(cache, qs, seq, out, layers, args.steps, args.warmup, stream)
        res["decode_per_layer_graph"] = {"form": "per-layer decode calls captured in one CUDA graph",
                                         "decode_us_per_step": g_s * 1e6, "launches_per_step": 2 * layers,
                                         "vs_all_layer_call": g_s * 1e6 / dec_us}
    peak, peak_src = hbm_peak()
    res["bulk_append"] = time_bulk_append(cache, w, layers, lens, dev, stream, peak, peak_src)
    res["prefill"] = time_prefill(name, cache, w, layers, lens, dev, stream)
    del cache, qs, out
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    cache, w, layers, lens = build_cache(args.workload, dev, batch=args.batch)
    B, Hq = w["batch"], w["n_q_heads"]
    qs, knew, vnew, pos, seq = step_inputs(w, layers, lens, dev)
    nbuf = len(qs)
    out = torch.empty(layers, B, Hq, 128, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        cache.append(-1, knew, vnew, pos)
        cache.decode(-1, qs[i % nbuf], seq, out)
    torch.cuda.synchronize()
    # device-timed region: events around the whole loop of K steps (nothing between the append
    # and the decode of a step, so the decode's programmatic launch can overlap the append's end)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            cache.append(-1, knew, vnew, pos)
            cache.decode(-1, qs[i % nbuf], seq, out)
        t1.record(stream)
        torch.cuda.synchronize()
        # the decode call alone, for its roofline: back-to-back calls for at least a second
        dec_us, dec_calls = time_decode_only(cache, qs, seq, out, args.steps, 0, stream, args.decode_min_s)
    total_ms = max_over_ranks(t0.elapsed_time(t1), dev)
    if cache.status() != 0:
        raise RuntimeError("device status set during the timed region")

    per_layer = None
    if layers > 1:
        g_s = max_over_ranks(time_per_layer_graph(cache, qs, seq, out, layers, args.steps, args.warmup, stream), dev)
        if cache.status() != 0:
            raise RuntimeError("device status set during the per-layer graph timing")
        per_layer = {"form": "per-layer decode calls captured in one CUDA graph", "decode_us_per_step": g_s * 1e6,
                     "launches_per_step": 2 * layers, "vs_all_layer_call": g_s * 1e6 / dec_us,
                     "tokens_per_s": weak_scaling_value(float(lens.sum()), world, g_s * 1e3)}

    # end-to-end through the public API: host inputs in, host output out, every step.  The copies
    # run on their own streams (one per direction, double-buffered device inputs and outputs), so
    # that step i+1's inputs land and step i's output leaves while the GPU computes: the pipeline a
    # serving loop runs.  Every step's copies are inside the timed region.
    q_h = [q.cpu().pin_memory() for q in qs]
    k_h, v_h = knew.cpu().pin_memory(), vnew.cpu().pin_memory()
    out_h = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    q_d = [torch.empty_like(qs[0]) for _ in range(2)]
    k_d, v_d = [torch.empty_like(knew) for _ in range(2)], [torch.empty_like(vnew) for _ in range(2)]
    out_d = [torch.empty_like(out) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # buffer j's inputs landed
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step using buffer j finished computing
    ev_out = [torch.cuda.Event() for _ in range(2)]   # buffer j's output copied out

    def run_e2e(n, start_event=None):
        def h2d(i):
            j = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(ev_done[j])       # the step that used buffer j has read it
                q_d[j].copy_(q_h[i % nbuf], non_blocking=True)
                k_d[j].copy_(k_h, non_blocking=True)
                v_d[j].copy_(v_h, non_blocking=True)
                ev_in[j].record(h2d_s)
        if start_event is not None:
            h2d_s.wait_event(start_event)
        h2d(0)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])           # out_d[j] of step i-2 has been copied out
            cache.append(-1, k_d[j], v_d[j], pos)
            cache.decode(-1, q_d[j], seq, out_d[j])
            ev_done[j].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[j])
                out_h[j].copy_(out_d[j], non_blocking=True)
                ev_out[j].record(d2h_s)
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)

    run_e2e(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_e2e(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    # for comparison, the same copies serialised with the compute on one stream
    e0.record(stream)
    for i in range(args.steps):
        q_d[0].copy_(q_h[i % nbuf], non_blocking=True)
        k_d[0].copy_(k_h, non_blocking=True)
        v_d[0].copy_(v_h, non_blocking=True)
        cache.append(-1, k_d[0], v_d[0], pos)
        cache.decode(-1, q_d[0], seq, out_d[0])
        out_h[0].copy_(out_d[0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = max_over_ranks(e0.elapsed_time(e1), dev)

    h2d_bytes = int(q_h[0].numel() * q_h[0].element_size() + 2 * knew.numel() * knew.element_size())
    d2h_bytes = int(out_h[0].numel() * 4)
    peak, peak_src = hbm_peak()
    append_res = time_bulk_append(cache, w, layers, lens, dev, stream, peak, peak_src)
    prefill_res = time_prefill(args.workload, cache, w, layers, lens, dev, stream)
    del cache, qs, out, q_h, q_d, k_d, v_d
    torch.cuda.empty_cache()

    tokens_per_rank = float(lens.sum())  # sequence lengths summed; every layer attends them
    ms_step = total_ms / args.steps
    value = weak_scaling_value(tokens_per_rank, world, ms_step)
    roof = decode_roofline(args.workload, w, layers, lens, dec_us, dec_calls)
    result = None
    if rank == 0:
        result = {
            "metric": "quantized-KV decode attention: cached tokens/s (decode of all layers + append of one token per layer)",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "us_per_step": ms_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAMES[w["k_format"]],
            "data": "synthetic (seeded N(0,1) with outlier channels, shapes of the workload; no weights)",
            "config": bench_config(args.workload, w, layers, lens, world),
            "hbm_gbs": roof["achieved"],
            "roofline": roof,
            "e2e": {"value": weak_scaling_value(tokens_per_rank, world, e2e_ms / args.steps), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": e2e_ms / args.steps,
                    "copies": "on their own streams (one per direction), double-buffered, overlapping the "
                              "neighbouring steps' compute",
                    "serialised": {"value": weak_scaling_value(tokens_per_rank, world, e2e_serial_ms / args.steps),
                                   "ms_per_step": e2e_serial_ms / args.steps,
                                   "copies": "on the compute stream, before and after each step"}},
            "gpu_launches": launches_per_step(w) * args.steps,
            "decode_per_layer_graph": per_layer,
            "clocks": clk.summary(),
            "bulk_append": append_res,
            "prefill": prefill_res,
            "block_codecs": time_block_codecs(dev, stream),
        }
        if layers < w["n_layers"]:
            # only `layers` of the model's layers are allocated and timed; the whole-model step
            # repeats the same per-layer work
            f = w["n_layers"] / layers
            result["value"] = value / f
            result["ms_per_step"] = ms_step * f
            result["us_per_step"] = ms_step * f * 1e3
            result["ms_per_step_timed_layers"] = ms_step
            result["e2e"]["value"] /= f
            result["e2e"]["serialised"]["value"] /= f
    others = [n for n in (args.also or []) if n != args.workload]
    if others and world == 1 and args.batch is None:
        with Clocks(local) as clk2:
            res_o = {n: measure_other_workload(n, args, dev, stream) for n in others}
        if result is not None:
            result["workloads"] = res_o
            result["workloads_clocks"] = clk2.summary()
    return result, w, layers, lens


# ------------------------------------------------------------------ CPU oracle
ORACLE_CPU_WORK_S = 24.0      # CPU-seconds of oracle decode per baseline sample (all workers)
REFERENCE_WALL_S = 60.0       # wall seconds of timed oracle work in a whole --impl reference run


def _oracle_units(w, layers, lens, n):
    """``n`` (layer, sequence) units spread over the workload: their seeded K/V, q and length."""
    H, Hq = w["n_kv_heads"], w["n_q_heads"]
    g = Hq // H
    seqs = np.linspace(0, len(lens) - 1, n).round().astype(int)
    units = []
    for i in range(n):
        layer, b = i % layers, int(seqs[i])
        L = int(lens[b])
        k, v = synth.kv_tokens(w, layer, 1, 1, 0, L, device="cpu")
        q = synth.queries(w, layer, 1, g, device="cpu").float().numpy()
        units.append((L, k.float().numpy(), v.float().numpy(), q))
    return units


def _oracle_cache(w, unit, proj):
    from oracle import attention

    L, k, v, q = unit
    ocfg = attention.OracleConfig(n_layers=1, n_kv_heads=1, n_q_heads=q.shape[1], max_batch=1,
                                  max_seq_len=L, window=w["window"], k_format=w["k_format"],
                                  sinkhorn=w["sinkhorn"], seed=w["wht_seed"])
    ora = attention.OracleCache(ocfg, proj)
    ora.append(0, k, v, np.array([0]))      # encode: not timed
    return ora


def _time_decode(ora, q, L, budget_s):
    """Repeat the oracle's decode of one unit until ``budget_s`` seconds of it have run."""
    spent, tokens, n = 0.0, 0, 0
    while spent < budget_s or n < 1:
        t = time.perf_counter()
        ora.decode(0, q, np.array([L]))
        spent += time.perf_counter() - t
        tokens += L
        n += 1
    return tokens, spent, n


def _oracle_worker(conn, w, unit, proj):
    """Spawned process, one BLAS thread: encode one unit, then time its decode once per budget
    received on ``conn`` and send back (tokens, seconds, calls); ``None`` ends the process."""
    try:
        ora = _oracle_cache(w, unit, proj)
        L, _, _, q = unit
        ora.decode(0, q, np.array([L]))     # warm-up call
        conn.send("ready")
        while True:
            budget = conn.recv()
            if budget is None:
                break
            conn.send(_time_decode(ora, q, L, budget))
    except Exception as e:                  # reported to the parent, which then gives up the pool
        conn.send(("error", repr(e)))
    finally:
        conn.close()


class OracleTimer:
    """One spawned worker process per host core, each holding one oracle unit of the workload.

    ``step(budget)`` has every worker time its unit's decode for ``budget`` seconds at the same
    time, so the sum of the workers' rates is the oracle's throughput on all cores.
    """

    def __init__(self, w, layers, lens, procs: int, timeout_s: float = 300.0):
        import multiprocessing as mp

        self.w, self.procs, self.timeout = w, procs, timeout_s
        proj = synth.qjl_projection(w["qjl_seed"]) if w["k_format"] == "tq3_qjl" else None
        units = _oracle_units(w, layers, lens, procs)
        ctx = mp.get_context("spawn")       # never fork a process that holds a CUDA context
        self.conns, self.workers = [], []
        for u in units:
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(b, w, u, proj), daemon=True)
            pr.start()
            b.close()
            self.conns.append(a)
            self.workers.append(pr)
        for c in self.conns:
            self._recv(c, "ready")

    def _recv(self, c, want=None):
        if not c.poll(self.timeout):
            raise RuntimeError("oracle worker timed out")
        m = c.recv()
        if isinstance(m, tuple) and m and m[0] == "error":
            raise RuntimeError(f"oracle worker failed: {m[1]}")
        if want is not None and m != want:
            raise RuntimeError(f"oracle worker sent {m!r}")
        return m

    def step(self, budget_s: float):
        for c in self.conns:
            c.send(budget_s)
        return [self._recv(c) for c in self.conns]

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for pr in self.workers:
            pr.join(timeout=30)
            if pr.is_alive():
                pr.terminate()
                pr.join(timeout=30)


def _baseline_record(w, layers, lens, results, procs, budget_s, all_cores: bool):
    """cpu_baseline object from per-unit (tokens, seconds, calls).  Rates add across workers that
    ran at the same time; units timed one after another in one thread give tokens / seconds.  One
    step attends every cached token once per (layer, kv-head), over the ``layers`` the GPU step
    covers."""
    H = w["n_kv_heads"]
    if all_cores:
        rates = [t / s for t, s, _ in results]          # token-heads per second, per worker
        rate, per_core_rate = sum(rates), sum(rates) / len(rates)
    else:
        rate = per_core_rate = sum(t for t, _, _ in results) / sum(s for _, s, _ in results)
    step_token_heads = float(lens.sum()) * H * layers
    value = float(lens.sum()) / (step_token_heads / rate)
    per_core = float(lens.sum()) / (step_token_heads / per_core_rate)
    calls = sum(n for _, _, n in results)
    how = (f"{procs} spawned processes, one BLAS thread each, each timing its own (layer, sequence, "
           f"kv-head) unit concurrently for {budget_s:.2f} s" if all_cores else
           "one thread in this process (the worker pool was not available)")
    return {"value": value, "unit": "tokens/s", "cores": procs if all_cores else 1, "kind": "oracle",
            "per_core_value": per_core,
            "sample": f"numpy oracle decode of {len(results)} units ({calls} timed calls) of the "
                      f"{layers * len(lens) * H} in one step, scaled by tokens attended to the "
                      f"whole step; not timed: the oracle's encode of each unit and the step's append of "
                      f"one token per layer (about 1/32000 of a step's tokens at these lengths); {how}"}


ORACLE_MAX_WORKERS = 64       # bounds the pool's start-up time and memory on very large hosts


def host_cores() -> int:
    """Oracle workers to start: the cores this process may run on, at most ORACLE_MAX_WORKERS."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(ORACLE_MAX_WORKERS, n))


def cpu_baseline(w, layers, lens, timer: OracleTimer | None = None, budget_s: float | None = None,
                 pool: bool = True):
    """The oracle's decode throughput on this host's cores (one worker per core); if the worker
    pool cannot be used (or ``pool`` is false), one thread in this process on three units."""
    own = timer is None
    try:
        if not pool:
            raise RuntimeError("worker pool not requested")
        if own:
            timer = OracleTimer(w, layers, lens, host_cores())
        budget = budget_s if budget_s is not None else max(1.0, ORACLE_CPU_WORK_S / timer.procs)
        return _baseline_record(w, layers, lens, timer.step(budget), timer.procs, budget, True)
    except Exception as e:  # noqa: BLE001 -- fall back to a one-thread sample and say so
        if pool:
            print(f"bench: oracle worker pool unavailable ({e}); timing one thread instead", file=sys.stderr)
        proj = synth.qjl_projection(w["qjl_seed"]) if w["k_format"] == "tq3_qjl" else None
        units = _oracle_units(w, layers, lens, 3)
        caches = [_oracle_cache(w, u, proj) for u in units]
        budget = budget_s if budget_s is not None else 12.0
        res = [_time_decode(c, u[3], u[0], budget / len(units)) for c, u in zip(caches, units)]
        return _baseline_record(w, layers, lens, res, 1, budget, False)
    finally:
        if own and timer is not None:
            timer.close()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    w, layers, lens = workload_cfg(args.workload)
    budget = max(0.5, REFERENCE_WALL_S / max(1, args.steps + args.warmup))   # wall seconds per step
    vals = []
    timer = None
    try:
        timer = OracleTimer(w, layers, lens, host_cores())
    except Exception as e:  # noqa: BLE001
        print(f"bench: oracle worker pool unavailable ({e}); timing one thread instead", file=sys.stderr)
        timer = None
    try:
        for i in range(args.warmup + args.steps):
            cb = cpu_baseline(w, layers, lens, timer=timer, budget_s=budget, pool=timer is not None)
            if i >= args.warmup:
                vals.append(cb["value"])
    finally:
        if timer is not None:
            timer.close()
    value = statistics.mean(vals)
    step_s = float(lens.sum()) / value
    cb["value"] = value
    return {"impl": "reference", "metric": "quantized-KV decode attention: cached tokens/s (decode of all layers + append of one token per layer)",
            "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64 attention, f32 codec", "data": "synthetic",
            "config": bench_config(args.workload, w, layers, lens, 1),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=HEADLINE_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--also", nargs="*", default=list(OTHER_WORKLOADS), choices=list(synth.WORKLOADS),
                    help="workloads measured after the headline one (decode roofline, per-layer form, "
                         "bulk append); none with --also alone")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep only the first B sequences of the workload (smaller profiler captures)")
    ap.add_argument("--decode-min-s", type=float, default=DECODE_ROOFLINE_MIN_S,
                    help="seconds of back-to-back decode calls timed for the roofline (0: --steps calls)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res))
        return
    res, w, layers, lens = run_gpu(args)
    if res is not None:
        if not args.no_cpu_baseline and res["n_gpus"] == 1:
            res["cpu_baseline"] = cpu_baseline(w, layers, lens)
        print(json.dumps(res))


if __name__ == "__main__":
    main()
