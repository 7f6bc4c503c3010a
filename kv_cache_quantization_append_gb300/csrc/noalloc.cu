// kv_decode_attention_noalloc: the decode entry point for callers that cannot allocate device
// memory.  Some hosts own every device allocation themselves (a serving engine that hands a
// plugin only pre-planned buffers, or a C ABI consumer with no allocator of its own) and cannot
// call cudaMalloc to provide the decode scratch buffer.  This variant takes its scratch from a
// fixed-size array in this library's device memory instead; everything else is the ordinary decode
// launch.
#include <mutex>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

// The scratch every call of this entry point shares (record ranges, then partial records).  It lives in
// the library's module on each device that uses it, until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)KVQ_NOALLOC_SCRATCH_MAX;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_addr[MAX_DEVICES] = {};

// Device address of the array for the current device: looked up once per device, with that device
// current (in host code the array's name is only a host-side stand-in, not a device address).
int scratch_address(int device, void** out) {
  if (device < 0 || device >= MAX_DEVICES) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return KVQ_OK;
}

}  // namespace

int decode_attention_noalloc(kvq_cache* cache, int32_t layer, const void* q, float* out,
                             const int32_t* seq_lens, int32_t batch, void* stream) {
  // argument errors first, so that a zero scratch size below can only mean a failed CUDA query
  if (layer < -1 || layer >= cache->cfg.n_layers) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > cache->cfg.max_batch) return KVQ_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev != cache->device) return KVQ_ERR_INVALID_ARG;
  const size_t need = kv_decode_scratch_bytes(cache, layer, batch);
  if (need == 0) return KVQ_ERR_CUDA;
  if (need > NOALLOC_SCRATCH_BYTES) return KVQ_ERR_CAPACITY;
  void* scratch = nullptr;
  const int rc = scratch_address(dev, &scratch);
  if (rc != KVQ_OK) return rc;
  // every decode call writes the parts of the scratch it reads, so it needs no clearing
  return kv_decode_attention(cache, layer, q, out, seq_lens, batch, scratch, NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace kvq

extern "C" int kv_decode_attention_noalloc(kvq_cache* cache, int32_t layer, const void* q, float* out,
                                           const int32_t* seq_lens, int32_t batch, void* stream) {
  if (!cache || cache->magic != kvq::MAGIC) return cache ? KVQ_ERR_NOT_INIT : KVQ_ERR_INVALID_ARG;
  return kvq::decode_attention_noalloc(cache, layer, q, out, seq_lens, batch, stream);
}
