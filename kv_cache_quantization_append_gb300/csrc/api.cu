// C ABI of libkvq: argument checking, cache layout and header set-up, kernel dispatch.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "kvq_internal.cuh"

namespace kvq {

static bool config_ok(const kvq_config& c) {
  if (c.n_layers < 1 || c.n_kv_heads < 1 || c.n_q_heads < 1) return false;
  if (c.head_dim != D || c.group != 32 || c.page_tokens != PAGE) return false;
  if (c.n_q_heads % c.n_kv_heads != 0) return false;
  const int g = c.n_q_heads / c.n_kv_heads;
  if (g < 1 || g > MAX_GQA) return false;
  if (c.max_batch < 1 || c.max_batch > MAX_BATCH || c.max_seq_len < 1) return false;
  if (c.window < 0 || c.window > MAX_WINDOW || c.window % WCHUNK != 0) return false;
  if (c.k_format != KVQ_Q4G32 && c.k_format != KVQ_TQ3_QJL && c.k_format != KVQ_Q8G32) return false;
  if (c.v_format != KVQ_Q4G32) return false;
  if (c.sinkhorn != 0 && c.sinkhorn != 1) return false;
  if (c.sinkhorn && c.k_format == KVQ_TQ3_QJL) return false;
  if (c.in_dtype != KVQ_IN_F32 && c.in_dtype != KVQ_IN_BF16) return false;
  if (c.n_pages < 0) return false;
  return true;
}

bool compute_layout(const kvq_config& c, Layout* L) {
  if (!config_ok(c)) return false;
  Layout l{};
  l.max_pages_per_seq = (c.max_seq_len + PAGE - 1) / PAGE;
  const long long contiguous = (long long)c.max_batch * l.max_pages_per_seq;
  if (contiguous > INT32_MAX) return false;
  l.n_pages = c.n_pages > 0 ? c.n_pages : (int)contiguous;
  // per token: K main 64 B (Q4G32, TQ3_QJL) or 128 B (Q8G32); K meta 16 B (Q4G32 scale and zero),
  // 4 B (TQ3_QJL norm and residual norm) or 8 B (Q8G32 scales)
  l.kmeta_bytes = c.k_format == KVQ_TQ3_QJL ? 4 : c.k_format == KVQ_Q8G32 ? 8 : 16;
  l.off_vmain = (c.k_format == KVQ_Q8G32 ? 128 : 64) * HALF;
  l.off_kmeta = l.off_vmain + 64 * HALF;
  l.off_vmeta = l.off_kmeta + l.kmeta_bytes * HALF;
  l.half_bytes = l.off_vmeta + 16 * HALF;
  l.page_bytes = 2 * l.half_bytes;
  size_t o = 0;
  l.off_status = o; o = align256(o + 16);
  l.off_signs = o;  o = align256(o + D * sizeof(float));
  l.off_cb = o;     o = align256(o + sizeof(CodebookDev));
  l.off_qjl = o;    o = align256(o + (c.k_format == KVQ_TQ3_QJL ? D * D * sizeof(float) : 0));
  const size_t sig = (size_t)c.n_layers * c.n_kv_heads * D * sizeof(__half);
  l.off_sigk = o;   o = align256(o + sig);
  l.off_sigv = o;   o = align256(o + sig);
  l.off_bt = o;     o = align256(o + (size_t)contiguous * sizeof(int32_t));
  const size_t ring = (size_t)c.n_layers * c.max_batch * c.n_kv_heads * c.window * D * sizeof(float);
  l.off_ringk = o;  o = align256(o + ring);
  l.off_ringv = o;  o = align256(o + ring);
  l.off_pages = o;
  o += (size_t)c.n_layers * l.n_pages * c.n_kv_heads * l.page_bytes;
  l.total = align256(o);
  *L = l;
  return true;
}

DevPtrs dev_ptrs(const kvq_cache& c, const Layout& L) {
  uint8_t* b = static_cast<uint8_t*>(c.dev);
  DevPtrs p;
  p.status = reinterpret_cast<unsigned*>(b + L.off_status);
  p.signs = reinterpret_cast<const float*>(b + L.off_signs);
  p.cb = reinterpret_cast<const CodebookDev*>(b + L.off_cb);
  p.qjl_t = reinterpret_cast<const float*>(b + L.off_qjl);
  p.sigk = reinterpret_cast<__half*>(b + L.off_sigk);
  p.sigv = reinterpret_cast<__half*>(b + L.off_sigv);
  p.ringk = reinterpret_cast<float*>(b + L.off_ringk);
  p.ringv = reinterpret_cast<float*>(b + L.off_ringv);
  p.pages = b + L.off_pages;
  return p;
}

// SplitMix64 (Steele, Lea & Flood 2014): sign j is -1 when bit 0 of output j+1 is set.
static void rotation_signs(uint64_t seed, float* out) {
  uint64_t state = seed;
  for (int j = 0; j < D; ++j) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    out[j] = (z & 1) ? -1.0f : 1.0f;
  }
}

// Lloyd-Max quantiser of a unit Gaussian, 8 levels, in double: alternate cell boundaries at
// centroid midpoints and centroids at the conditional means (phi(a) - phi(b)) / (Phi(b) - Phi(a)).
static void lloyd_max8(double* cent) {
  const double inv_sqrt2pi = 0.3989422804014327;
  for (int k = 0; k < 8; ++k) cent[k] = -2.0 + 4.0 * k / 7.0;
  for (int it = 0; it < 200000; ++it) {
    double edge[9];
    edge[0] = -INFINITY;
    edge[8] = INFINITY;
    for (int k = 1; k < 8; ++k) edge[k] = 0.5 * (cent[k - 1] + cent[k]);
    double change = 0.0;
    double next[8];
    for (int k = 0; k < 8; ++k) {
      const double a = edge[k], b = edge[k + 1];
      const double pa = std::isinf(a) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * a * a);
      const double pb = std::isinf(b) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * b * b);
      const double Fa = 0.5 * std::erfc(-a / std::sqrt(2.0));
      const double Fb = 0.5 * std::erfc(-b / std::sqrt(2.0));
      next[k] = (pa - pb) / (Fb - Fa);
      change = std::fmax(change, std::fabs(next[k] - cent[k]));
    }
    for (int k = 0; k < 8; ++k) cent[k] = next[k];
    if (change < 1e-15) break;
  }
}

static void build_codebook(CodebookDev* cb) {
  double c[8];
  lloyd_max8(c);
  const double s = 1.0 / std::sqrt(128.0);
  float cf[8];
  for (int k = 0; k < 8; ++k) {
    cb->cent[k] = __double2half(c[k] * s);
    cf[k] = __half2float(cb->cent[k]);
  }
  for (int k = 0; k < 7; ++k) cb->bnd[k] = (cf[k] + cf[k + 1]) / 2.0f;
  cb->bnd[7] = INFINITY;
  for (int v = 0; v < 256; ++v) {
    const __half lo = cb->cent[v & 7], hi = cb->cent[(v >> 3) & 7];
    uint16_t l, h;
    std::memcpy(&l, &lo, 2);
    std::memcpy(&h, &hi, 2);
    const uint32_t s0 = (v >> 6) & 1 ? 0x3C00u : 0xBC00u;  // fp16 +1 / -1
    const uint32_t s1 = (v >> 7) & 1 ? 0x3C00u : 0xBC00u;
    cb->lut8[v] = make_uint2((uint32_t)l | ((uint32_t)h << 16), s0 | (s1 << 16));
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static int cuda_err(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

static int check_cache(const kvq_cache* c, Layout* L) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->magic != MAGIC) return KVQ_ERR_NOT_INIT;
  if (!compute_layout(c->cfg, L)) return KVQ_ERR_NOT_INIT;
  return KVQ_OK;
}

static int layers_of_call(const kvq_cache* c, int32_t layer, int* l0, int* nl) {
  if (layer == -1) {
    *l0 = 0;
    *nl = c->cfg.n_layers;
    return KVQ_OK;
  }
  if (layer < 0 || layer >= c->cfg.n_layers) return KVQ_ERR_INVALID_ARG;
  *l0 = layer;
  *nl = 1;
  return KVQ_OK;
}

// The cache's pointers belong to the device that was current at kv_cache_init; a launch with
// another device current would hand that device foreign addresses, so such calls are refused.
static int check_device(const kvq_cache* c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  return dev == c->device ? KVQ_OK : KVQ_ERR_INVALID_ARG;
}

// give-up limit of the decode pipeline's waits (kv_set_wait_limit_ns)
std::atomic<unsigned long long> g_decode_wait_ns{1000000000ull};
unsigned long long decode_wait_ns() { return g_decode_wait_ns.load(); }

int decode_ctas(int device) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  return sms;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

size_t kv_cache_bytes(const kvq_config* cfg) {
  if (!cfg) return 0;
  Layout L;
  if (!compute_layout(*cfg, &L)) return 0;
  return L.total;
}

int kv_cache_init(kvq_cache* cache, const kvq_config* cfg, void* dev_mem, size_t bytes,
                  const int32_t* block_table, const float* qjl_proj_host, void* stream) {
  if (!cache || !cfg || !dev_mem) return KVQ_ERR_INVALID_ARG;
  Layout L;
  if (!compute_layout(*cfg, &L)) return KVQ_ERR_UNSUPPORTED;
  if (bytes < L.total) return KVQ_ERR_CAPACITY;
  if (!aligned16(dev_mem) || (block_table && !aligned16(block_table))) return KVQ_ERR_ALIGN;
  if (cfg->k_format == KVQ_TQ3_QJL && !qjl_proj_host) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;

  // header image on the host, copied in one piece
  const size_t hdr = L.off_ringk;
  std::vector<uint8_t> h(hdr, 0);
  rotation_signs(cfg->seed, reinterpret_cast<float*>(h.data() + L.off_signs));
  build_codebook(reinterpret_cast<CodebookDev*>(h.data() + L.off_cb));
  if (cfg->k_format == KVQ_TQ3_QJL) {
    float* t = reinterpret_cast<float*>(h.data() + L.off_qjl);
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) t[j * D + i] = qjl_proj_host[i * D + j];
  }
  const size_t nsig = (size_t)cfg->n_layers * cfg->n_kv_heads * D;
  uint16_t* sk = reinterpret_cast<uint16_t*>(h.data() + L.off_sigk);
  uint16_t* sv = reinterpret_cast<uint16_t*>(h.data() + L.off_sigv);
  for (size_t i = 0; i < nsig; ++i) sk[i] = sv[i] = 0x3C00;  // fp16 1.0
  int32_t* bt = reinterpret_cast<int32_t*>(h.data() + L.off_bt);
  for (long long i = 0; i < (long long)cfg->max_batch * L.max_pages_per_seq; ++i) bt[i] = (int32_t)i;
  cudaError_t e = cudaMemcpyAsync(dev_mem, h.data(), hdr, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;

  std::memset(cache, 0, sizeof(*cache));
  cache->cfg = *cfg;
  cache->dev = dev_mem;
  cache->bytes = bytes;
  cache->block_table = block_table ? block_table
                                   : reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(dev_mem) + L.off_bt);
  cache->max_pages_per_seq = L.max_pages_per_seq;
  cache->n_pages = L.n_pages;
  cache->device = dev;
  cache->magic = MAGIC;
  return KVQ_OK;
}

size_t kv_calibrate_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t n_tokens) {
  Layout L;
  if (check_cache(cache, &L) != KVQ_OK || n_tokens < 1 || n_tokens > 4096) return 0;
  int l0, nl;
  if (layers_of_call(cache, layer, &l0, &nl) != KVQ_OK) return 0;
  return (size_t)nl * cache->cfg.n_kv_heads * 2 * n_tokens * D * sizeof(float);
}

int kv_calibrate(kvq_cache* cache, int32_t layer, const void* k_calib, const void* v_calib,
                 int32_t n_tokens, void* scratch, size_t scratch_bytes, void* stream) {
  Layout L;
  int rc = check_cache(cache, &L);
  if (rc != KVQ_OK) return rc;
  if (!cache->cfg.sinkhorn) return KVQ_ERR_UNSUPPORTED;
  if (!k_calib || !v_calib || !scratch || n_tokens < 1 || n_tokens > 4096) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_calib) || !aligned16(v_calib) || !aligned16(scratch)) return KVQ_ERR_ALIGN;
  int l0, nl;
  if ((rc = layers_of_call(cache, layer, &l0, &nl)) != KVQ_OK) return rc;
  if (scratch_bytes < kv_calibrate_scratch_bytes(cache, layer, n_tokens)) return KVQ_ERR_CAPACITY;
  if ((rc = check_device(cache)) != KVQ_OK) return rc;
  CalibArgs a;
  a.p = dev_ptrs(*cache, L);
  a.kc = k_calib;
  a.vc = v_calib;
  a.work = static_cast<float*>(scratch);
  a.layer0 = l0;
  a.n_layers_call = nl;
  a.Hkv = cache->cfg.n_kv_heads;
  a.ntok = n_tokens;
  a.in_bf16 = cache->cfg.in_dtype == KVQ_IN_BF16;
  return cuda_err(launch_calibrate(a, static_cast<cudaStream_t>(stream)));
}

int kv_quant_append(kvq_cache* cache, int32_t layer, const void* k, const void* v,
                    const int32_t* pos, int32_t batch, int32_t n_tokens, void* stream) {
  Layout L;
  int rc = check_cache(cache, &L);
  if (rc != KVQ_OK) return rc;
  if (!k || !v || !pos) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > cache->cfg.max_batch || n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(pos)) return KVQ_ERR_ALIGN;
  int l0, nl;
  if ((rc = layers_of_call(cache, layer, &l0, &nl)) != KVQ_OK) return rc;
  if ((rc = check_device(cache)) != KVQ_OK) return rc;
  AppendArgs a;
  a.p = dev_ptrs(*cache, L);
  a.L = L;
  a.block_table = cache->block_table;
  a.k = k;
  a.v = v;
  a.pos = pos;
  a.layer0 = l0;
  a.n_layers_call = nl;
  a.batch = batch;
  a.T = n_tokens;
  a.Hkv = cache->cfg.n_kv_heads;
  a.W = cache->cfg.window;
  a.max_seq_len = cache->cfg.max_seq_len;
  a.k_format = cache->cfg.k_format;
  a.sinkhorn = cache->cfg.sinkhorn;
  a.in_bf16 = cache->cfg.in_dtype == KVQ_IN_BF16;
  a.max_batch = cache->cfg.max_batch;
  return cuda_err(launch_append(a, static_cast<cudaStream_t>(stream)));
}

size_t kv_decode_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t batch) {
  Layout L;
  if (check_cache(cache, &L) != KVQ_OK || batch < 1 || batch > cache->cfg.max_batch) return 0;
  int l0, nl;
  if (layers_of_call(cache, layer, &l0, &nl) != KVQ_OK) return 0;
  const int ctas = decode_ctas(cache->device);
  if (ctas <= 0) return 0;
  return decode_scratch_bytes(nl * batch * cache->cfg.n_kv_heads, ctas, cache->cfg.k_format);
}

int kv_decode_attention(kvq_cache* cache, int32_t layer, const void* q, float* out,
                        const int32_t* seq_lens, int32_t batch, void* scratch,
                        size_t scratch_bytes, void* stream) {
  Layout L;
  int rc = check_cache(cache, &L);
  if (rc != KVQ_OK) return rc;
  if (!q || !out || !seq_lens || !scratch) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > cache->cfg.max_batch) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(seq_lens) || !aligned16(scratch)) return KVQ_ERR_ALIGN;
  int l0, nl;
  if ((rc = layers_of_call(cache, layer, &l0, &nl)) != KVQ_OK) return rc;
  if ((rc = check_device(cache)) != KVQ_OK) return rc;
  const int ctas = decode_ctas(cache->device);
  if (ctas <= 0) return KVQ_ERR_CUDA;
  const int n_units = nl * batch * cache->cfg.n_kv_heads;
  if (scratch_bytes < decode_scratch_bytes(n_units, ctas, cache->cfg.k_format)) return KVQ_ERR_CAPACITY;
  DecodeArgs a;
  a.p = dev_ptrs(*cache, L);
  a.L = L;
  a.block_table = cache->block_table;
  a.q = q;
  a.out = out;
  a.seq_lens = seq_lens;
  // scratch: record ranges int2 [n_units], then the partial records
  a.unit_info = static_cast<int2*>(scratch);
  a.records = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + align256((size_t)n_units * sizeof(int2)));
  a.layer0 = l0;
  a.n_layers_call = nl;
  a.batch = batch;
  a.Hkv = cache->cfg.n_kv_heads;
  a.g = cache->cfg.n_q_heads / cache->cfg.n_kv_heads;
  a.W = cache->cfg.window;
  a.max_seq_len = cache->cfg.max_seq_len;
  a.k_format = cache->cfg.k_format;
  a.sinkhorn = cache->cfg.sinkhorn;
  a.in_bf16 = cache->cfg.in_dtype == KVQ_IN_BF16;
  a.max_batch = cache->cfg.max_batch;
  a.max_pages_per_seq = cache->max_pages_per_seq;
  a.identity_pages = cache->block_table == reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(cache->dev) + L.off_bt);
  a.n_units = n_units;
  a.n_ctas = ctas;
  a.wait_ns = decode_wait_ns();
  return cuda_err(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

size_t kv_prefill_scratch_bytes(const kvq_cache* cache, int32_t layer, int32_t batch) {
  Layout L;
  if (check_cache(cache, &L) != KVQ_OK || batch < 1 || batch > cache->cfg.max_batch) return 0;
  int l0, nl;
  if (layers_of_call(cache, layer, &l0, &nl) != KVQ_OK) return 0;
  return std::max<size_t>(256, prefill_scratch_bytes(nl, batch, cache->cfg.n_kv_heads, cache->cfg.window));
}

int kv_prefill_attention(kvq_cache* cache, int32_t layer, const void* k, const void* v, const void* q,
                         float* out, const int32_t* pos, int32_t batch, int32_t n_tokens, void* scratch,
                         size_t scratch_bytes, void* stream) {
  Layout L;
  int rc = check_cache(cache, &L);
  if (rc != KVQ_OK) return rc;
  if (!k || !v || !q || !out || !pos || !scratch) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > cache->cfg.max_batch || n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out) || !aligned16(pos) || !aligned16(scratch))
    return KVQ_ERR_ALIGN;
  int l0, nl;
  if ((rc = layers_of_call(cache, layer, &l0, &nl)) != KVQ_OK) return rc;
  if (scratch_bytes < kv_prefill_scratch_bytes(cache, layer, batch)) return KVQ_ERR_CAPACITY;
  if ((rc = check_device(cache)) != KVQ_OK) return rc;
  AppendArgs ap;
  ap.p = dev_ptrs(*cache, L);
  ap.L = L;
  ap.block_table = cache->block_table;
  ap.k = k;
  ap.v = v;
  ap.pos = pos;
  ap.layer0 = l0;
  ap.n_layers_call = nl;
  ap.batch = batch;
  ap.T = n_tokens;
  ap.Hkv = cache->cfg.n_kv_heads;
  ap.W = cache->cfg.window;
  ap.max_seq_len = cache->cfg.max_seq_len;
  ap.k_format = cache->cfg.k_format;
  ap.sinkhorn = cache->cfg.sinkhorn;
  ap.in_bf16 = cache->cfg.in_dtype == KVQ_IN_BF16;
  ap.max_batch = cache->cfg.max_batch;
  PrefillArgs a;
  a.p = ap.p;
  a.L = L;
  a.block_table = cache->block_table;
  a.k = k;
  a.v = v;
  a.q = q;
  a.out = out;
  a.pos = pos;
  const size_t snap = prefill_scratch_bytes(nl, batch, cache->cfg.n_kv_heads, cache->cfg.window) / 2;
  a.snap_k = static_cast<float*>(scratch);
  a.snap_v = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + snap);
  a.layer0 = l0;
  a.n_layers_call = nl;
  a.batch = batch;
  a.max_batch = cache->cfg.max_batch;
  a.Hkv = cache->cfg.n_kv_heads;
  a.g = cache->cfg.n_q_heads / cache->cfg.n_kv_heads;
  a.W = cache->cfg.window;
  a.T = n_tokens;
  a.k_format = cache->cfg.k_format;
  a.sinkhorn = cache->cfg.sinkhorn;
  a.in_bf16 = ap.in_bf16;
  a.max_pages_per_seq = cache->max_pages_per_seq;
  a.max_seq_len = cache->cfg.max_seq_len;
  return cuda_err(launch_prefill(a, ap, static_cast<cudaStream_t>(stream)));
}

int kv_status(kvq_cache* cache, uint32_t* flags, void* stream) {
  Layout L;
  int rc = check_cache(cache, &L);
  if (rc != KVQ_OK) return rc;
  if (!flags) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* st = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(cache->dev) + L.off_status);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, st, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st, 0, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  *flags = v;
  return KVQ_OK;
}

int kv_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1 || ns > 10000000000ull) return KVQ_ERR_INVALID_ARG;
  g_decode_wait_ns.store(ns);
  return KVQ_OK;
}

const char* kv_strerror(int code) {
  switch (code) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case KVQ_ERR_CAPACITY: return "buffer too small";
    case KVQ_ERR_CUDA: return "CUDA runtime error";
    case KVQ_ERR_NOT_INIT: return "cache not initialised";
    default: return "unknown status code";
  }
}

}  // extern "C"
