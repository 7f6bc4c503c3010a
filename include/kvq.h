/*
 * kvq.h -- C ABI of the GB300 (sm_103a) quantized KV cache: append and decode attention.
 *
 * What the library computes (sources named by page title and section):
 *   [QC] "Beyond RAG: load the whole document on your laptop" (quant.cpp summary):
 *        the 128 most recent tokens stay FP32, everything else is 4-bit ("how it works"
 *        paragraph; PPL / KV-memory table row "4-bit + progressive"); a batched write of the
 *        quantized K cache is bit-identical to per-token writes (v3.2 batched-prefill note).
 *   [KV] "Running Bonsai ternary 27B at 120K context in under 10 GB of VRAM" (KVarN port):
 *        Walsh-Hadamard transform plus Sinkhorn variance balancing before 4-bit ("TLDR"
 *        paragraph); separate K and V cache types (--cache-type-k / --cache-type-v).
 *   [TQ] "LLM memory saving: weights vs KV-cache quantization (2026)": random rotation, a
 *        per-coordinate optimal scalar quantiser and a 1-bit QJL sketch of the residual for an
 *        unbiased inner product ("method comparison" table, "key idea" row); attention logits
 *        computed directly on low-bit keys ("inference cost" row).
 *
 * Conventions for every entry point
 *   - All functions are host functions.  Pointers documented as "device" must point to memory of
 *     the CUDA device that was current at kv_cache_init, and that device must be current when an
 *     entry point that launches work is called (KVQ_ERR_INVALID_ARG otherwise).  The caller owns
 *     every buffer (the cache, inputs, outputs, scratch, the block table) with one exception:
 *     kv_decode_attention_noalloc takes its scratch from a fixed array of the library's own device
 *     memory.  No entry point allocates or frees memory.
 *   - Device pointers must be 16-byte aligned (KVQ_ERR_ALIGN otherwise).
 *   - Work is enqueued asynchronously on ``stream`` (a cudaStream_t; NULL = legacy default
 *     stream).  Entry points return after launching; none synchronises except kv_cache_init
 *     (its header copy) and kv_status.
 *   - Invalid arguments return a KVQ_ERR_* code and launch nothing.  Inconsistencies only the
 *     device can see (a block-table entry out of range, a position past capacity, a sequence
 *     length out of range, a pipeline wait that gave up) set bits in the cache's device status
 *     word, read with kv_status.
 *   - head_dim is 128; n_q_heads is a multiple of n_kv_heads with a GQA group of 1..4 query heads
 *     per kv-head; page_tokens is 64; window is 0 or a multiple of 4 up to 1024.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, layer or batch out of range */
  KVQ_ERR_UNSUPPORTED = 2,   /* config outside the supported shapes (see conventions above) */
  KVQ_ERR_ALIGN = 3,         /* a device pointer is not 16-byte aligned */
  KVQ_ERR_CAPACITY = 4,      /* buffer too small for the config (cache or scratch) */
  KVQ_ERR_CUDA = 5,          /* a CUDA runtime call failed (launch, attribute, copy) */
  KVQ_ERR_NOT_INIT = 6,      /* cache struct not initialised by kv_cache_init */
};

/* bits of the device status word (kv_status) */
enum {
  KVQ_DEV_BAD_PAGE = 1u,       /* block-table entry outside [0, n_pages): the token was skipped */
  KVQ_DEV_POS_RANGE = 2u,      /* pos + n_tokens > max_seq_len: the sequence was skipped */
  KVQ_DEV_SEQLEN_RANGE = 4u,   /* seq_lens[b] < 0 or > max_seq_len: treated as empty */
  KVQ_DEV_TIMEOUT = 8u,        /* a copy-pipeline wait gave up after ~1 s: output is incomplete */
};

/* ---------------------------------------------------------------- formats */
enum {
  KVQ_Q4G32 = 1,     /* 4-bit asymmetric codes, groups of 32 channels, fp16 scale and zero (K, V) */
  KVQ_TQ3_QJL = 3,   /* keys only: 3-bit Lloyd-Max codes of the unit vector, fp16 norm, 128 QJL
                        residual sign bits and fp16 residual norm */
  KVQ_Q8G32 = 4,     /* keys only: 8-bit symmetric codes, groups of 32 channels, fp16 scale */
};
enum { KVQ_IN_F32 = 0, KVQ_IN_BF16 = 1 };

typedef struct kvq_config {
  int32_t n_layers;      /* layers held by this cache */
  int32_t n_kv_heads;
  int32_t n_q_heads;     /* multiple of n_kv_heads; n_q_heads / n_kv_heads in 1..4 */
  int32_t head_dim;      /* 128 */
  int32_t max_batch;     /* sequences the cache holds */
  int32_t max_seq_len;   /* capacity per sequence (tokens) */
  int32_t window;        /* most recent tokens also kept in FP32; 0 = flat 4-bit ([QC]: 128) */
  int32_t page_tokens;   /* 64 */
  int32_t n_pages;       /* physical pages per layer; 0 = max_batch * ceil(max_seq_len / 64) */
  int32_t k_format;      /* KVQ_Q4G32, KVQ_TQ3_QJL or KVQ_Q8G32 */
  int32_t v_format;      /* KVQ_Q4G32 */
  int32_t sinkhorn;      /* 1 = per-channel balancing scales (not with KVQ_TQ3_QJL keys) */
  int32_t group;         /* 32 */
  int32_t in_dtype;      /* KVQ_IN_F32 or KVQ_IN_BF16: dtype of k, v, q and calibration inputs */
  uint64_t seed;         /* seed of the rotation's random signs (SplitMix64 stream) */
} kvq_config;

/* Host-side handle, filled by kv_cache_init; plain data, may be copied. */
typedef struct kvq_cache {
  kvq_config cfg;
  void* dev;                    /* the cache buffer (device), caller-owned */
  uint64_t bytes;               /* its size */
  const int32_t* block_table;   /* device int32 [max_batch][max_pages_per_seq] */
  int32_t max_pages_per_seq;    /* ceil(max_seq_len / page_tokens) */
  int32_t n_pages;              /* physical pages per layer actually used */
  int32_t device;               /* CUDA device ordinal at init */
  uint32_t magic;               /* set by kv_cache_init */
} kvq_cache;

/*
 * Memory layout of the cache buffer (offsets 256-byte aligned, in this order):
 *   header     status word, rotation signs (float[128] of +-1), TQ3 codebook and its decode table,
 *              QJL projection (transposed, float[128][128], TQ3 keys only), Sinkhorn scales
 *              sigma_k, sigma_v (fp16 [n_layers][n_kv_heads][128], 1.0 until calibrated),
 *              identity block table (used when kv_cache_init gets none)
 *   ring_k     float [n_layers][max_batch][n_kv_heads][window][128]   slot = position % window
 *   ring_v     same
 *   pages      [n_layers][n_pages][n_kv_heads][page_bytes]; one page = 64 tokens of one
 *              (layer, kv-head) stored as two 32-token halves (tokens 0-31, 32-63), each half
 *              contiguous with regions in order (t = token index within the half):
 *     K main   Q4G32 and TQ3_QJL: 64 B per token at 64t; Q8G32: 128 B per token at 128t
 *     V main   64 B per token at K + 64t, K = 2048 (Q4G32, TQ3_QJL) or 4096 (Q8G32)
 *     K meta   after V main: Q4G32 per token fp16 {scale[4], zero[4]} (512 B); TQ3_QJL fp16
 *              norm[32], gamma[32] (128 B); Q8G32 per token fp16 scale[4] (256 B)
 *     V meta   after K meta: fp16 scale[4][32] then fp16 zero[4][32] (group-major, 512 B)
 *   Half sizes: Q4G32 K + Q4G32 V = 5120 B, TQ3_QJL K + Q4G32 V = 4736 B, Q8G32 K + Q4G32 V =
 *   6912 B.
 *   Q4G32 K record (64 B per token): 32-bit word (i, G), i, G = 0..3, at byte 16i + 4G holds channels
 *     32G + 8i .. 32G + 8i + 7 of the rotated (and balanced) vector; byte k of the word holds
 *     channel 32G + 8i + 2k in its low nibble and the next channel in its high nibble.
 *   Q4G32 V region (64 B per token): tokens 2p and 2p+1 of a half share bytes [128p, 128p + 128);
 *     for r = 0..7, G = 0..3 the 4 bytes at 128p + 16*((r + 2*(p mod 4)) mod 8) + 4G are
 *     [token 2p byte0, token 2p+1 byte0, token 2p byte1, token 2p+1 byte1], where byte0 holds
 *     channels 32G + 4r (low nibble) and 32G + 4r + 1, byte1 channels 32G + 4r + 2 and + 3.
 *   Q8G32 K record (128 B per token t): codes are stored as unsigned bytes u = c + 128 (c in
 *     -127..127); sixteen-byte chunk m = 2i + h (i = 0..3, h = 0..1) sits at 16 * (m XOR (t mod 2))
 *     and its 32-bit word w holds, for k = 16 (4h + w), the channels k + 2i, k + 2i + 1, k + 2i + 8,
 *     k + 2i + 9 in bytes 0..3.  Scale d of group G (channels 32G .. 32G + 31) at K meta + 8t + 2G.
 *   TQ3_QJL K record (64 B per token): byte j holds the 3-bit codes of channels 2j (bits 0-2) and
 *     2j + 1 (bits 3-5) and the QJL sign bits (1 = (S r)_i >= 0) of projections i = 2j (bit 6) and
 *     2j + 1 (bit 7).
 */

/*
 * Closed-form size of the cache buffer for ``cfg``; 0 if the config is invalid or unsupported.
 * [QC] PPL / KV-memory table and the "6.4x KV compression" figure: a Q4G32 record is 4-bit codes
 * plus an fp16 scale and zero per 32 values, 80 B per 128-value vector against 512 B in FP32
 * (6.4x); the "4-bit + progressive" row adds the 128-token FP32 window on top of the 4-bit store
 * (2.33 vs 2.30 GB for Llama-3.2-3B at 32K), which is the ring counted here.  [TQ] "method
 * comparison" table, compression >= 4.5x: a TQ3_QJL key record is 68 B (3-bit codes, 128 sign bits,
 * fp16 norm and residual norm).  [TQ] "when to use what" and "rules" lists (keep K at Q8, cut only
 * V): a Q8G32 key record is 136 B (8-bit codes and four fp16 scales).  Total = header + 2 rings of n_layers * max_batch * n_kv_heads *
 * window * 512 B + n_layers * n_pages * n_kv_heads pages of 64 tokens x (K record + 80 B), each
 * region rounded up to 256 B.
 */
size_t kv_cache_bytes(const kvq_config* cfg);

/*
 * Lay out a cache in the caller's device buffer ``dev_mem`` (``bytes`` >= kv_cache_bytes(cfg)),
 * write the header (signs from cfg->seed, codebook, QJL projection, unit Sinkhorn scales,
 * identity block table) and clear the status word.  Page and ring contents are not cleared.
 * The header holds what the pages' codecs fix once per cache: the random +-1 signs of the
 * randomised Walsh-Hadamard rotation ([KV] TLDR; [TQ] "key idea" row, random rotation), the
 * per-coordinate optimal (Lloyd-Max) 3-bit codebook and the Gaussian projection of the 1-bit QJL
 * residual sketch ([TQ] "key idea" row), and the Sinkhorn scales of [KV] TLDR (1 until
 * kv_calibrate).  The window size follows [QC] "how it works" (the 128 most recent tokens in FP32).
 *   block_table      device int32 [max_batch][max_pages_per_seq] mapping (sequence, logical page)
 *                    to a physical page in [0, n_pages); NULL = contiguous identity table.  The
 *                    caller keeps it alive and may rewrite it between calls.
 *   qjl_proj_host    host float [128][128] row-major i.i.d. N(0,1) projection S of the QJL sketch;
 *                    required when k_format == KVQ_TQ3_QJL, ignored otherwise.
 * Synchronises ``stream`` before returning (the header copies are complete on return).
 * Saving and restoring: the buffer holds the whole state (header with signs, codebook, projection
 * and Sinkhorn scales; the identity block table; rings; pages), none of it tied to its address.
 * To restore a saved copy, call kv_cache_init with the same config on a buffer of the same size
 * (or reuse the struct of the original buffer), then copy the saved bytes over the whole buffer;
 * a caller-supplied block table is the caller's to save.  Re-initialising a live buffer resets
 * its Sinkhorn scales to 1.
 */
int kv_cache_init(kvq_cache* cache, const kvq_config* cfg, void* dev_mem, size_t bytes,
                  const int32_t* block_table, const float* qjl_proj_host, void* stream);

/*
 * KVarN calibration ([KV] TLDR): for each kv-head of ``layer`` (or every layer when layer == -1)
 * rotate the raw calibration block, run 8 Sinkhorn row/column RMS balancing iterations and store
 * the per-channel scale sigma (fp16) for K and for V.  Must precede the quantised appends of that
 * layer.  Inputs (device, cfg.in_dtype): k_calib, v_calib [L?][n_kv_heads][n_tokens][128] with the
 * leading layer axis present when layer == -1.  n_tokens in 1..4096.  ``scratch`` (device, at
 * least kv_calibrate_scratch_bytes) holds the float working copies.  Needs cfg.sinkhorn == 1.
 * sigma is relative (an overall factor is free) and stored as fp16: a channel whose scale falls
 * below fp16's smallest subnormal relative to the others (column RMS ratios beyond ~10^7) stores
 * sigma = 0, and values later appended in that channel are divided by zero.
 */
size_t kv_calibrate_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t n_tokens);
int kv_calibrate(kvq_cache* cache, int32_t layer, const void* k_calib, const void* v_calib,
                 int32_t n_tokens, void* scratch, size_t scratch_bytes, void* stream);

/*
 * Append ``n_tokens`` new K/V vectors to each of the first ``batch`` sequences at positions
 * pos[b] .. pos[b] + n_tokens - 1 ([QC] "how it works"; v3.2 note: one call with n_tokens = T
 * writes exactly the bytes of T calls with n_tokens = 1).  Every token is rotated, balanced
 * (if calibrated) and quantised into its page; the last min(n_tokens, window) tokens are also
 * written raw (float) into the window ring.
 *   layer      0..n_layers-1, or -1 for all layers (k, v then carry a leading layer axis)
 *   k, v       device, cfg.in_dtype, [L?][batch][n_kv_heads][n_tokens][128], contiguous
 *   pos        device int32 [batch]; pos[b] < 0 leaves sequence b untouched (lets a caller
 *              append ragged chunks to a subset of the batch)
 * Value range: scales, zeros, norms and sigma are stored as fp16, so each vector must be finite
 * with Euclidean norm below 65504 (after division by sigma when balanced; the rotation keeps the
 * norm).  TQ3 keys must also be zero or have some rotated element above 2^-75 in magnitude: when
 * every square underflows float32 the norm is 0, the 1/max(norm, FLT_MIN) guard scales the vector
 * by 2^126 and the stored residual norm is infinite (the key's logits are then NaN).  Outside
 * these ranges the stored metadata is infinite or NaN and the codes are undefined; nothing is
 * flagged.
 */
int kv_quant_append(kvq_cache* cache, int32_t layer, const void* k, const void* v,
                    const int32_t* pos, int32_t batch, int32_t n_tokens, void* stream);

/*
 * One decode step of attention for the first ``batch`` sequences over their cached tokens:
 * positions [0, L - window) through the quantised pages (logits in rotated space), positions
 * [L - window, L) through the FP32 ring, one softmax with scale 1/sqrt(128), L = seq_lens[b]
 * (tokens already appended, the current one included).  An empty sequence (L = 0) gives zeros.
 * Sources: [QC] "how it works" (attention over the 4-bit store plus the FP32 window of the most
 * recent 128 tokens; the PPL / KV-memory table's "4-bit + progressive" row is this read path);
 * [TQ] "method comparison" table, "inference cost" row (attention logits computed directly on the
 * low-bit keys, no dense FP16 copy) and "key idea" row (the QJL residual term makes the inner
 * product estimate unbiased); [KV] TLDR (the Sinkhorn scales are folded into q and the output).
 *   layer      0..n_layers-1, or -1 for all layers (q, out then carry a leading layer axis)
 *   q          device, cfg.in_dtype, [L?][batch][n_q_heads][128]; query head j uses kv-head
 *              j / (n_q_heads / n_kv_heads)
 *   out        device float [L?][batch][n_q_heads][128]
 *   seq_lens   device int32 [batch]
 *   scratch    device, >= kv_decode_scratch_bytes(cache, layer, batch) bytes, any contents
 *              (every call writes what it reads).  Calls that share a scratch buffer must not
 *              overlap on the GPU.
 * Splits the token axis over all SMs and runs a bulk-copy pipeline per SM (one launch); a second,
 * small launch on the same stream merges the partial softmax states.  Results do not depend on
 * timing (fixed merge order).  Calls may be captured in a CUDA graph once a call of the same or a
 * larger batch has run on the device outside capture (the first call sets the kernel's
 * shared-memory size, a host-side step that capture does not record).
 */
size_t kv_decode_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t batch);
int kv_decode_attention(kvq_cache* cache, int32_t layer, const void* q, float* out,
                        const int32_t* seq_lens, int32_t batch, void* scratch,
                        size_t scratch_bytes, void* stream);

/*
 * Allocation-free variant of kv_decode_attention (no counterpart on the pages: it exists for
 * callers that cannot allocate device memory -- hosts that own every device allocation
 * themselves, such as a serving engine that hands a plugin only pre-planned buffers, or a C caller
 * without an allocator of its own).  Same arguments and results as kv_decode_attention minus the
 * scratch buffer: the scratch comes from a fixed array of KVQ_NOALLOC_SCRATCH_MAX bytes inside the
 * library's device memory, held on every device that uses it until the process exits.
 *   - Calls needing more scratch than that (kv_decode_scratch_bytes > KVQ_NOALLOC_SCRATCH_MAX)
 *     return KVQ_ERR_CAPACITY and launch nothing.
 *   - The first call on a device looks up the array's device address (once per device, with that
 *     device current); make that first call before any stream capture.  The address is kept for
 *     the life of the process: after a cudaDeviceReset (or any teardown of the device's primary
 *     context) this entry point must not be called again on that device.
 *   - Every call shares the one array: calls that overlap on the GPU (other streams, other host
 *     threads) race on it and must be serialised by the caller.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define KVQ_NOALLOC_SCRATCH_MAX (32u * 1024u * 1024u)
int kv_decode_attention_noalloc(kvq_cache* cache, int32_t layer, const void* q, float* out,
                                const int32_t* seq_lens, int32_t batch, void* stream);

/*
 * Chunked prefill ([QC] v3.2 batched-prefill note: a batched prefill writes exactly what per-token
 * steps write; its attention is read the same way): append ``n_tokens`` new K/V vectors to each of
 * the first ``batch`` sequences at pos[b] .. pos[b] + n_tokens - 1 (exactly as kv_quant_append),
 * and compute the attention of their queries: query t of sequence b attends to positions
 * [0, pos[b] + t], the newest ``window`` of them through their raw values and the rest through
 * their quantised records -- what n_tokens single-token append + decode steps would compute.
 *   layer      0..n_layers-1, or -1 for all layers (k, v, q, out then carry a leading layer axis)
 *   k, v       device, cfg.in_dtype, [L?][batch][n_kv_heads][n_tokens][128]
 *   q          device, cfg.in_dtype, [L?][batch][n_q_heads][n_tokens][128]
 *   out        device float [L?][batch][n_q_heads][n_tokens][128]; rows of a sequence with
 *              pos[b] < 0 (not part of the call) or pos[b] + n_tokens > max_seq_len (flagged
 *              KVQ_DEV_POS_RANGE, nothing appended) are zeros
 *   pos        device int32 [batch]
 *   scratch    device, >= kv_prefill_scratch_bytes(cache, layer, batch) bytes, any contents: holds a
 *              copy of the window ring taken before the chunk's append (its raw values are read by
 *              the chunk's first queries after the append has overwritten their ring slots)
 * Three launches on ``stream``: the ring copy, the append, the attention (tensor-core logits and
 * P.V over tiles of 32 positions, 64 (query, head) rows per block).
 */
size_t kv_prefill_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t batch);
int kv_prefill_attention(kvq_cache* cache, int32_t layer, const void* k, const void* v, const void* q,
                         float* out, const int32_t* pos, int32_t batch, int32_t n_tokens, void* scratch,
                         size_t scratch_bytes, void* stream);

/*
 * Block codecs next to the cache: the TurboQuant MSE quantiser ([TQ] "key idea" row: random
 * rotation, per-coordinate optimal scalar quantiser of the unit vector, its norm) on other blocks.
 * Both rotate with randomized Walsh-Hadamard transforms whose signs are the SplitMix64 stream of
 * ``seed`` (its first 128 are a cache's rotation signs for the same seed), code each coordinate
 * with the 2^b-level Lloyd-Max codebook of N(0, 1/n) (fp16 centroids, fp32 midpoints, ties up) and
 * store the norm as fp16; codes are little-endian bit streams.  Asynchronous on ``stream``; device
 * pointers 16-byte aligned (``blocks`` of TBQ: any alignment).
 *
 * TBQ3_0 / TBQ4_0-style blocks ([TQ] "what the blogbot verified": the llama.cpp proposal adding
 * TBQ3_0 / TBQ4_0; "limits and counterpoints": about 3.0625 / 4.0625 bits per value): 256
 * consecutive values (e.g. two 128-value heads of a token row), 256-point rotation, record = fp16
 * norm + 256 codes of ``bits`` (3 or 4) bits = 98 / 130 bytes.
 *   x        device, in_dtype (KVQ_IN_F32 / KVQ_IN_BF16), [n_blocks][256]
 *   blocks   device bytes [n_blocks][kv_tbq_block_bytes(bits)]
 *   decode output: device float [n_blocks][256]
 */
size_t kv_tbq_block_bytes(int32_t bits);
int kv_tbq_encode(int32_t bits, uint64_t seed, const void* x, int32_t in_dtype, int64_t n_blocks, void* blocks,
                  void* stream);
int kv_tbq_decode(int32_t bits, uint64_t seed, const void* blocks, int64_t n_blocks, float* x, void* stream);

/*
 * Outlier-channel split ([TQ] "method comparison" table: LongBench at 2.5 and 3.5 bits; "what the
 * blogbot verified": non-integer widths come from splitting off outlier channels): per set (e.g. a
 * (layer, kv-head)), the 64 channels with the largest mean square over a calibration block are
 * coded at ``hi_bits`` (3 or 4) and the other 64 at hi_bits - 1 -- 2.5 or 3.5 bits a channel, norms
 * aside -- each set in ascending channel order, rotated by a 64-point transform (signs 0..63 and
 * 64..127).  Record = fp16 norm of the outlier set, of the others, then their code streams: 44 / 60
 * bytes per 128-value vector.
 *   kv_split_outliers: calib device, in_dtype, [n_sets][n_tokens][128]; outliers device int16
 *     [n_sets][64] (out), ascending; sums of squares in float64 over the tokens in order, ties to the
 *     lower channel.
 *   kv_split_encode / decode: vectors [n_vectors][128] in n_sets equal consecutive groups, group s
 *     coded with outliers[s]; records device [n_vectors][kv_split_record_bytes(hi_bits)]; decode
 *     output device float [n_vectors][128].
 */
size_t kv_split_record_bytes(int32_t hi_bits);
int kv_split_outliers(const void* calib, int32_t in_dtype, int32_t n_sets, int32_t n_tokens, int16_t* outliers,
                      void* stream);
int kv_split_encode(int32_t hi_bits, uint64_t seed, const int16_t* outliers, int32_t n_sets, const void* x,
                    int32_t in_dtype, int64_t n_vectors, void* records, void* stream);
int kv_split_decode(int32_t hi_bits, uint64_t seed, const int16_t* outliers, int32_t n_sets, const void* records,
                    int64_t n_vectors, float* x, void* stream);

/* Read and clear the device status word (synchronises ``stream``); *flags gets KVQ_DEV_* bits. */
int kv_status(kvq_cache* cache, uint32_t* flags, void* stream);

/* The stall limit, in nanoseconds, of the decode copy pipeline's producer wait (a producer warp
 * waiting for its consumers to release a stage) for every later kv_decode_attention / _noalloc
 * call of this process: a serving loop can tighten the ~1 s default to detect a stalled decode
 * sooner.  ns must lie in [1, 1e10], else KVQ_ERR_INVALID_ARG and the limit is unchanged.  A
 * producer whose wait runs out stops issuing copies and sets KVQ_DEV_TIMEOUT in the status word
 * (the call's output is then incomplete); its consumers give up on the stages that never come after
 * their own ~1 s limit, and the streaming kernel still waits for every copy it started before its
 * blocks exit.  The prefill and append kernels keep their own ~1 s limits.  Not thread-safe against
 * concurrent decode launches from other host threads. */
int kv_set_wait_limit_ns(uint64_t ns);

/* Static string for a KVQ_* status code. */
const char* kv_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
