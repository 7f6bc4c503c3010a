"""CPU oracle for the quantized KV cache: test infrastructure, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library: it is a plain, slow numpy restatement of
what the method computes, written from the source pages:

* [QC] "Beyond RAG: load the whole document on your laptop" (molayo1419.me summary of the
  quant.cpp README) -- 128 most recent tokens kept in FP32, everything else 4-bit ("how it works"
  paragraph and the PPL / KV-memory table); batched prefill writes the quantized K cache
  bit-identically to per-token writes (v3.2 note); the ``1/max(sqrt(ss), eps)`` normalisation
  (v3.19 note); fixed floating-point reduction order for determinism (v3.18 note).
* [KV] "Running Bonsai ternary 27B at 120K context in under 10 GB of VRAM" (molayo1419.me repost
  of the KVarN port) -- Walsh-Hadamard transform plus Sinkhorn variance balancing before 4-bit
  ("TLDR" paragraph).
* [TQ] "LLM memory saving: weights vs KV-cache quantization (2026)" (conanssam.com) -- random
  rotation, per-coordinate optimal scalar quantiser, 1-bit QJL sketch of the residual for an
  unbiased inner product ("method comparison" table, "key idea" row); K kept at 8 bits while V
  is cut to low bits as the safe asymmetric setting ("when to use what" and "rules" lists).

Codec arithmetic is IEEE float32 in a fixed operation order with no fused multiply-add (every
numpy ufunc call below rounds once), because the codes it decides must match the GPU bit for bit.
Attention is evaluated in float64 on the exact dequantized values.

``blocks`` holds the two block codecs next to the cache (the outlier-channel split behind
TurboQuant's 2.5 / 3.5-bit results, and TBQ3_0 / TBQ4_0-style 256-value blocks), pinned by
``tests/test_oracle_blocks.py``.

Every function is pinned by ``tests/test_oracle_pins.py`` against facts the pages or mathematics
fix.  One reading has no outside pin beyond invariants: the Sinkhorn balancing statistic
(``sinkhorn_sigma``) -- "parity unpinned" beyond the invariants listed in its docstring.
"""

from . import codec, attention, blocks  # noqa: F401
