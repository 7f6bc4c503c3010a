// Internal definitions shared by the translation units of libkvq: buffer layout, kernel
// parameter blocks, and small device helpers (warp Walsh-Hadamard butterfly, input loads).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int D = 128;           // head_dim
constexpr int PAGE = 64;         // tokens per page (block-table granularity)
constexpr int HALF = 32;         // tokens per half-page: one contiguous set of regions, one pipeline stage
constexpr int WCHUNK = 4;        // window slots per pipeline stage
constexpr int MAX_WINDOW = 1024;
constexpr int MAX_GQA = 4;
constexpr int MAX_BATCH = 1024;
constexpr uint32_t MAGIC = 0x4b565131u;  // "KVQ1"
constexpr unsigned FULL = 0xffffffffu;

// float32 round-to-nearest of 2^-3.5 = 1/sqrt(128)
constexpr float C_WHT = 0.0883883461356163f;
// log2(e) / sqrt(128): logits are kept in base-2 units so the softmax uses exp2
constexpr float LOGIT_SCALE = 0.127517431974411f;
// sqrt(pi / 2) / 128: QJL inner-product estimator constant for m = 128 projections
constexpr float QJL_CONST = 0.009791516698896885f;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t off_status, off_signs, off_cb, off_qjl, off_sigk, off_sigv, off_bt;
  size_t off_ringk, off_ringv, off_pages, total;
  int max_pages_per_seq, n_pages;
  // A 64-token page is two 32-token halves, each laid out as K main | V main | K meta | V meta.
  int page_bytes, half_bytes, off_vmain, off_kmeta, off_vmeta, kmeta_bytes;  // offsets within a half
};

// codebook block inside the header
struct CodebookDev {
  __half cent[8];        // TQ3 centroids (ascending)
  float bnd[8];          // 7 boundaries (midpoints), [7] unused
  // decode table of one TQ3 record byte v (two 3-bit codes in bits 0-5, two QJL sign bits in
  // bits 6-7): .x = half2 (cent[v & 7], cent[(v >> 3) & 7]), .y = half2 of the signs as +-1
  // (bit set = +1, the sign of a non-negative projection)
  uint2 lut8[256];
};

bool compute_layout(const kvq_config& c, Layout* L);

struct DevPtrs {
  unsigned* status;
  const float* signs;
  const CodebookDev* cb;
  const float* qjl_t;     // transposed projection: qjl_t[j][i] = S[i][j]
  __half* sigk;           // [L][H][128]
  __half* sigv;
  float* ringk;
  float* ringv;
  uint8_t* pages;
};

DevPtrs dev_ptrs(const kvq_cache& c, const Layout& L);

// ---------------------------------------------------------------- launchers
struct AppendArgs {
  DevPtrs p;
  Layout L;
  const int32_t* block_table;
  const void* k;
  const void* v;
  const int32_t* pos;
  int layer0, n_layers_call, batch, max_batch, T, Hkv, W, max_seq_len, k_format, sinkhorn, in_bf16;
  int kv_lo, kv_n;  // vectors handled by one launch: K (0) and/or V (1), kv_lo .. kv_lo + kv_n - 1
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
// after_keys: the values of a TurboQuant-key append, launched right after the keys kernel as its
// programmatic dependent (the two overlap; the values grid ends after the keys grid)
cudaError_t launch_append_bulk(const AppendArgs& a, cudaStream_t s, bool after_keys = false);

struct CalibArgs {
  DevPtrs p;
  const void* kc;
  const void* vc;
  float* work;            // [n_layers_call][Hkv][2][ntok][128]
  int layer0, n_layers_call, Hkv, ntok, in_bf16;
};
cudaError_t launch_calibrate(const CalibArgs& a, cudaStream_t s);

struct DecodeArgs {
  DevPtrs p;
  Layout L;
  const int32_t* block_table;
  const void* q;
  float* out;
  const int32_t* seq_lens;
  int2* unit_info;  // [n_units] first record index and record count of each unit
  float* records;   // partial records, index unit + global consumer warp
  int layer0, n_layers_call, batch, max_batch, Hkv, g, W, max_seq_len, k_format, sinkhorn, in_bf16;
  int max_pages_per_seq, n_units, n_ctas;
  int identity_pages;  // block_table is the cache's own identity table (page p of sequence b = b * max_pages_per_seq + p)
  unsigned long long wait_ns;  // give-up limit of the producer warps' wait for a released stage
};
int decode_ctas(int device);
unsigned long long decode_wait_ns();
size_t decode_scratch_bytes(int n_units, int n_ctas, int k_format);
size_t decode_record_slots(int n_units, int n_ctas, int k_format);
int decode_consumer_warps(int k_format);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

struct PrefillArgs {
  DevPtrs p;
  Layout L;
  const int32_t* block_table;
  const void* k;     // [L?][batch][Hkv][T][128] cfg.in_dtype: the chunk's raw keys
  const void* v;
  const void* q;     // [L?][batch][Hq][T][128] cfg.in_dtype
  float* out;        // [L?][batch][Hq][T][128]
  const int32_t* pos;
  float* snap_k;     // [n_layers_call][batch][Hkv][W][128]: the window ring before the chunk's append
  float* snap_v;
  int layer0, n_layers_call, batch, max_batch, Hkv, g, W, T, k_format, sinkhorn, in_bf16;
  int max_pages_per_seq, max_seq_len;
};
size_t prefill_scratch_bytes(int n_layers_call, int batch, int Hkv, int W);
cudaError_t launch_prefill(const PrefillArgs& a, const AppendArgs& app, cudaStream_t s);

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__
__device__ __forceinline__ float4 load4_in(const void* base, size_t elem_off, int bf16) {
  if (bf16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + elem_off);
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem_off);
}

// Packed pairs of IEEE fp32 operations (sm_100+ `add/sub/mul/fma.rn.f32x2`): each half is rounded
// exactly like the scalar __fadd_rn / __fsub_rn / __fmul_rn / __fmaf_rn, two values per instruction.
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void up2(unsigned long long r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)));
  up2(r, a0, a1);
}
__device__ __forceinline__ void sub2(float& a0, float& a1, float b0, float b1) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)));
  up2(r, a0, a1);
}
__device__ __forceinline__ void mul2(float& a0, float& a1, float b0, float b1) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)));
  up2(r, a0, a1);
}
// a = a * b + c, pairwise
__device__ __forceinline__ void fma2(float& a0, float& a1, float b0, float b1, float c0, float c1) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a0, a1)), "l"(pk2(b0, b1)), "l"(pk2(c0, c1)));
  up2(r, a0, a1);
}
// butterfly of two pairs: (a, b) -> (a + b, a - b), element by element
__device__ __forceinline__ void bfly2(float& a0, float& a1, float& b0, float& b1) {
  const float u0 = a0, u1 = a1;
  add2(a0, a1, b0, b1);
  float d0 = u0, d1 = u1;
  sub2(d0, d1, b0, b1);
  b0 = d0;
  b1 = d1;
}

// Unnormalised Hadamard butterfly over a warp: lane l holds elements 4l..4l+3.  Stages
// h = 1, 2 inside the lane, h = 4..64 across lanes (xor 1..16); every add/sub rounds once.
__device__ __forceinline__ void hadamard_warp(float& x0, float& x1, float& x2, float& x3, int lane) {
  float a0 = __fadd_rn(x0, x1), a1 = __fsub_rn(x0, x1);
  float a2 = __fadd_rn(x2, x3), a3 = __fsub_rn(x2, x3);
  x0 = __fadd_rn(a0, a2);
  x2 = __fsub_rn(a0, a2);
  x1 = __fadd_rn(a1, a3);
  x3 = __fsub_rn(a1, a3);
  // cross-lane stages: the lower lane of a pair gets a + b, the upper one a - b, both as one
  // fma(mine, +-1, partner): the product by +-1 is exact, so the single rounding equals that of the
  // plain add / subtract
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sg = (lane & m) ? -1.0f : 1.0f;
    const float y0 = __shfl_xor_sync(FULL, x0, m);
    const float y1 = __shfl_xor_sync(FULL, x1, m);
    const float y2 = __shfl_xor_sync(FULL, x2, m);
    const float y3 = __shfl_xor_sync(FULL, x3, m);
    x0 = __fmaf_rn(x0, sg, y0);
    x1 = __fmaf_rn(x1, sg, y1);
    x2 = __fmaf_rn(x2, sg, y2);
    x3 = __fmaf_rn(x3, sg, y3);
  }
}

// Fixed-order float32 sum of squares of a warp-held 128-vector: per lane
// ((x0^2 + x1^2) + (x2^2 + x3^2)), then halving over lanes (xor 16, 8, 4, 2, 1).  Every lane
// ends with the same value.
__device__ __forceinline__ float sumsq_warp(float x0, float x1, float x2, float x3) {
  float s = __fadd_rn(__fadd_rn(__fmul_rn(x0, x0), __fmul_rn(x1, x1)),
                      __fadd_rn(__fmul_rn(x2, x2), __fmul_rn(x3, x3)));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL, s, m));
  return s;
}
#endif

}  // namespace kvq
