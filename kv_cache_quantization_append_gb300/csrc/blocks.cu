// Block codecs next to the cache: the outlier-channel split behind TurboQuant's 2.5 / 3.5-bit
// results, and TBQ3_0 / TBQ4_0-style 256-value blocks.
//
// Both are the TurboQuant MSE quantiser of [TQ] "LLM memory saving: weights vs KV-cache
// quantization (2026)", "key idea" row -- a randomized Walsh-Hadamard rotation, the block's norm,
// and per-coordinate optimal (Lloyd-Max) codes of the unit vector -- on blocks other than one head
// vector:
//  * TBQ ("what the blogbot verified" list: the llama.cpp proposal adding TBQ3_0 / TBQ4_0; "limits
//    and counterpoints": about 3.0625 / 4.0625 bits): 256 consecutive values (two 128-value heads of
//    a token row), a 256-point rotation (c = 1/16), fp16 norm + 256 b-bit codes = 98 / 130 bytes.
//  * Outlier split ("method comparison" table: LongBench at 2.5 and 3.5 bits; non-integer widths
//    from splitting off outlier channels): the 64 channels with the largest mean square over a
//    calibration block at hi bits, the other 64 at hi - 1 bits, each set rotated by a 64-point
//    transform (c = 1/8) with signs 0..63 / 64..127: 44 / 60 bytes per 128-value vector.
// One warp per block (TBQ: 8 values a lane) or per vector (split: a half-warp per set, 4 values a
// lane); every floating-point step is one IEEE operation in the order of the definition, so the
// codes and the decoded values are reproducible bit for bit.
#include <cfloat>
#include <cmath>
#include <cstring>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int WARPS = 8;
constexpr int MAX_LEVELS = 16;

struct BlockArgs {
  uint32_t sign_bits[8];              // sign j of the SplitMix64 stream is -1 when bit j is set
  __half cent[2][MAX_LEVELS];         // [0] = the block's (TBQ) or the outlier set's codebook, [1] = the others'
  float bnd[2][MAX_LEVELS];
  int bits[2], levels[2];
  const void* x;                      // values (encode), in_dtype
  const uint8_t* rec_in;              // records (decode)
  uint8_t* rec;                       // records (encode)
  float* out;                         // values (decode)
  const int16_t* outliers;            // [n_sets][64] ascending (split)
  long long n_items, per_set;
  int in_bf16, rec_bytes;
};

__device__ __forceinline__ float sgn(const BlockArgs& a, int j) {
  return (a.sign_bits[j >> 5] >> (j & 31)) & 1u ? -1.0f : 1.0f;
}

// code = number of boundaries <= u (ties go up), by binary search over the levels - 1 ascending
// boundaries (a NaN compares false everywhere: code 0, as the plain count)
__device__ __forceinline__ int code_of(float u, const float* bnd, int levels) {
  int c = 0;
  for (int st = levels >> 1; st >= 1; st >>= 1)
    if (bnd[c + st - 1] <= u) c += st;
  return c;
}

// ------------------------------------------------------------------ TBQ: one warp per 256 values
// in-lane butterfly stages h = 1, 2, 4 of a lane's 8 consecutive values, then the cross-lane ones
// (h = 8 .. 128: partner lane ^ 1 .. 16, fma(mine, +-1, partner) rounds like the add / subtract).
// PACKED: stages h = 2, 4 and the cross-lane ones as packed f32x2 operations on the value pairs
// (2i, 2i+1), each half rounded like the scalar operation (the encoder, issue-bound: +12 %; the
// decoder, bound by HBM, measured 2 % slower with them and keeps the scalar form).
template <bool PACKED>
__device__ __forceinline__ void hadamard256(float (&v)[8], int lane) {
  if constexpr (PACKED) {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float p = v[j], q = v[j + 1];
      v[j] = __fadd_rn(p, q);
      v[j + 1] = __fsub_rn(p, q);
    }
    bfly2(v[0], v[1], v[2], v[3]);  // h = 2
    bfly2(v[4], v[5], v[6], v[7]);
    bfly2(v[0], v[1], v[4], v[5]);  // h = 4
    bfly2(v[2], v[3], v[6], v[7]);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
      for (int j = 0; j < 8; j += 2)
        fma2(v[j], v[j + 1], sg, sg, __shfl_xor_sync(FULL, v[j], m), __shfl_xor_sync(FULL, v[j + 1], m));
    }
  } else {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (!(j & h)) {
          const float p = v[j], q = v[j + h];
          v[j] = __fadd_rn(p, q);
          v[j + h] = __fsub_rn(p, q);
        }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __fmaf_rn(v[j], sg, __shfl_xor_sync(FULL, v[j], m));
    }
  }
}

// this lane's 8 rotation signs (values 8 lane .. 8 lane + 7) as bits
__device__ __forceinline__ uint32_t lane_signs8(const BlockArgs& a, int lane) {
  return (a.sign_bits[lane >> 2] >> (8 * (lane & 3))) & 0xffu;
}
// v * (+-1): the sign flip is exact, so it equals the multiply
__device__ __forceinline__ float flip(float v, uint32_t bits, int j) {
  return __uint_as_float(__float_as_uint(v) ^ (((bits >> j) & 1u) << 31));
}
__device__ __forceinline__ void load8(const BlockArgs& a, long long blk, int lane, float (&v)[8]) {
  const size_t e0 = (size_t)blk * 256 + 8 * lane;
  const float4 lo = load4_in(a.x, e0, a.in_bf16), hi = load4_in(a.x, e0 + 4, a.in_bf16);
  v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
  v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
}

// Each warp walks its blocks with the next block's values loaded before the current one is coded.
__global__ void __launch_bounds__(WARPS * 32) tbq_encode_kernel(const __grid_constant__ BlockArgs a) {
  __shared__ float sbnd[MAX_LEVELS];
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < MAX_LEVELS) sbnd[threadIdx.x] = a.bnd[0][threadIdx.x];
  __syncthreads();
  const int b = a.bits[0], L = a.levels[0];
  const float c = 0.0625f;  // 1/sqrt(256)
  const uint32_t sb = lane_signs8(a, lane);
  const long long stride = (long long)gridDim.x * WARPS;
  long long blk = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  float nxt[8];
  if (blk < a.n_items) load8(a, blk, lane, nxt);
  for (; blk < a.n_items; blk += stride) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = flip(nxt[j], sb, j);
    if (blk + stride < a.n_items) load8(a, blk + stride, lane, nxt);
    hadamard256<true>(v, lane);
#pragma unroll
    for (int j = 0; j < 8; j += 2) mul2(v[j], v[j + 1], c, c);
    // fixed-order sum of squares: blocks (8l .. 8l+3), (8l+4 .. 8l+7); block i meets i + 32, + 16,
    // ..., + 2 (lanes ^ 16 .. 1, even and odd blocks apart), then block 0 meets block 1
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      q[j] = v[j];
      q[j + 1] = v[j + 1];
      mul2(q[j], q[j + 1], v[j], v[j + 1]);
    }
    float se = __fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3]));
    float so = __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) add2(se, so, __shfl_xor_sync(FULL, se, m), __shfl_xor_sync(FULL, so, m));
    const float n = __fsqrt_rn(__fadd_rn(se, so));
    const float inv = __fdiv_rn(1.0f, fmaxf(n, FLT_MIN));
    uint32_t field = 0;  // this lane's 8 codes, b bits each, little endian
#pragma unroll
    for (int j = 0; j < 8; ++j) field |= (uint32_t)code_of(__fmul_rn(v[j], inv), sbnd, L) << (b * j);
    uint8_t* dst = a.rec + (size_t)blk * a.rec_bytes;
    for (int k = 0; k < b; ++k) dst[2 + b * lane + k] = (uint8_t)(field >> (8 * k));
    // the fp16 norm as one 16-bit store (records have even sizes, so it is aligned); written as two
    // byte stores it came out with a wrong low byte on the GPU
    if (lane == 0) *reinterpret_cast<uint16_t*>(dst) = __half_as_ushort(__float2half_rn(n));
  }
}

__global__ void __launch_bounds__(WARPS * 32) tbq_decode_kernel(const __grid_constant__ BlockArgs a) {
  __shared__ float scent[MAX_LEVELS];
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < MAX_LEVELS) scent[threadIdx.x] = __half2float(a.cent[0][threadIdx.x]);
  __syncthreads();
  const int b = a.bits[0];
  const uint32_t cmask = (1u << b) - 1u;
  const float c = 0.0625f;
  const uint32_t sb = lane_signs8(a, lane);
  const long long stride = (long long)gridDim.x * WARPS;
  long long blk = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  // the record's norm and this lane's code bytes, loaded one block ahead
  uint32_t field_n = 0, n_n = 0;
  auto fetch = [&](long long k) {
    const uint8_t* src = a.rec_in + (size_t)k * a.rec_bytes;
    uint32_t f = 0;
    for (int q = 0; q < b; ++q) f |= (uint32_t)__ldg(src + 2 + b * lane + q) << (8 * q);
    field_n = f;
    n_n = __ldg(reinterpret_cast<const uint16_t*>(src));
  };
  if (blk < a.n_items) fetch(blk);
  for (; blk < a.n_items; blk += stride) {
    const uint32_t field = field_n;
    const float n = __half2float(__ushort_as_half((unsigned short)n_n));
    if (blk + stride < a.n_items) fetch(blk + stride);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(n, scent[(field >> (b * j)) & cmask]);
    hadamard256<false>(v, lane);
    float* dst = a.out + (size_t)blk * 256 + 8 * lane;
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = flip(__fmul_rn(v[j], c), sb, j);
    reinterpret_cast<float4*>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
}

// ------------------------------------------------------------------ outlier split: one warp per vector
// half-warp s (0 = outlier set, 1 = the others), lane i of it holds positions 4i .. 4i+3 of its set.
// butterfly of 64 values: stages h = 1, 2 in the lane, h = 4 .. 32 across lanes ^ 1 .. 8
__device__ __forceinline__ void hadamard64(float (&v)[4], int lane) {
  float p0 = __fadd_rn(v[0], v[1]), p1 = __fsub_rn(v[0], v[1]);
  float p2 = __fadd_rn(v[2], v[3]), p3 = __fsub_rn(v[2], v[3]);
  v[0] = __fadd_rn(p0, p2);
  v[2] = __fsub_rn(p0, p2);
  v[1] = __fadd_rn(p1, p3);
  v[3] = __fsub_rn(p1, p3);
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __fmaf_rn(v[j], sg, __shfl_xor_sync(FULL, v[j], m));
  }
}

// perm[p] = channel of set position p (0..63 the outlier set, 64..127 the others, each ascending)
__device__ __forceinline__ void build_perm(const int16_t* outl, int16_t* perm, uint32_t* mask, int lane) {
  if (lane < 4) mask[lane] = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) perm[4 * lane + e] = (int16_t)(4 * lane + e);
  __syncwarp();
  for (int k = lane; k < 64; k += 32) {
    const int ch = outl[k] & 127;
    atomicOr(&mask[ch >> 5], 1u << (ch & 31));
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int ch = 4 * lane + e;
    int below = 0;  // outlier channels below ch
    for (int w = 0; w < (ch >> 5); ++w) below += __popc(mask[w]);
    below += __popc(mask[ch >> 5] & ((1u << (ch & 31)) - 1u));
    const bool isout = (mask[ch >> 5] >> (ch & 31)) & 1u;
    perm[isout ? below : 64 + (ch - below)] = (int16_t)ch;
  }
  __syncwarp();
}

// Each warp walks its vectors with the next vector's values gathered before the current one is coded
// (when it belongs to the same set; at a set boundary they are gathered after the new permutation).
__global__ void __launch_bounds__(WARPS * 32) split_encode_kernel(const __grid_constant__ BlockArgs a) {
  __shared__ int16_t sperm[WARPS][128];
  __shared__ uint32_t smask[WARPS][4];
  __shared__ uint32_t swords[WARPS][16];
  __shared__ float sbnd[2][MAX_LEVELS];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  if (threadIdx.x < 2 * MAX_LEVELS) sbnd[threadIdx.x / MAX_LEVELS][threadIdx.x % MAX_LEVELS] = a.bnd[threadIdx.x / MAX_LEVELS][threadIdx.x % MAX_LEVELS];
  __syncthreads();
  const int s = lane >> 4, i = lane & 15;
  const int b = a.bits[s], L = a.levels[s];
  const int bo = a.bits[0];
  float sg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sg[e] = sgn(a, 64 * s + 4 * i + e);
  const long long stride = (long long)gridDim.x * WARPS;
  long long vec = (long long)blockIdx.x * WARPS + wl;
  long long cur_set = -1;
  float nxt[4];
  auto gather = [&](long long k) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = 64 * s + 4 * i + e;
      const size_t idx = (size_t)k * D + (sperm[wl][p] & 127);  // in range even for a malformed list
      nxt[e] = a.in_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[idx])
                         : static_cast<const float*>(a.x)[idx];
    }
  };
  if (vec < a.n_items) {
    cur_set = vec / a.per_set;
    build_perm(a.outliers + cur_set * 64, sperm[wl], smask[wl], lane);
    gather(vec);
  }
  for (; vec < a.n_items; vec += stride) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(nxt[e], sg[e]);
    const long long next = vec + stride;
    const bool next_same = next < a.n_items && next / a.per_set == cur_set;
    if (next_same) gather(next);
    hadamard64(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __fmul_rn(v[e], 0.125f);
    float ss = __fadd_rn(__fadd_rn(__fmul_rn(v[0], v[0]), __fmul_rn(v[1], v[1])),
                         __fadd_rn(__fmul_rn(v[2], v[2]), __fmul_rn(v[3], v[3])));
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(FULL, ss, m));
    const float n = __fsqrt_rn(ss);
    const float inv = __fdiv_rn(1.0f, fmaxf(n, FLT_MIN));
    if (lane < 16) swords[wl][lane] = 0u;
    __syncwarp();
    // code stream of set s starts at bit 32 (after the two norms) + 64 * bits[0] for the others
    const int base = 32 + (s ? 64 * bo : 0) + b * 4 * i;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t code = (uint32_t)code_of(__fmul_rn(v[e], inv), sbnd[s], L);
      const int bit = base + b * e;
      atomicOr(&swords[wl][bit >> 5], code << (bit & 31));
      if ((bit & 31) + b > 32) atomicOr(&swords[wl][(bit >> 5) + 1], code >> (32 - (bit & 31)));
    }
    if (i == 0) {
      const uint32_t nh = __half_as_ushort(__float2half_rn(n));
      atomicOr(&swords[wl][0], nh << (16 * s));
    }
    __syncwarp();
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.rec + (size_t)vec * a.rec_bytes);
    if (lane < a.rec_bytes / 4) dst[lane] = swords[wl][lane];
    __syncwarp();
    if (next < a.n_items && !next_same) {
      cur_set = next / a.per_set;
      build_perm(a.outliers + cur_set * 64, sperm[wl], smask[wl], lane);
      gather(next);
    }
  }
}

__global__ void __launch_bounds__(WARPS * 32) split_decode_kernel(const __grid_constant__ BlockArgs a) {
  __shared__ int16_t sperm[WARPS][128];
  __shared__ uint32_t smask[WARPS][4];
  __shared__ uint32_t swords[WARPS][16];
  __shared__ float scent[2][MAX_LEVELS];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  if (threadIdx.x < 2 * MAX_LEVELS)
    scent[threadIdx.x / MAX_LEVELS][threadIdx.x % MAX_LEVELS] = __half2float(a.cent[threadIdx.x / MAX_LEVELS][threadIdx.x % MAX_LEVELS]);
  __syncthreads();
  const int s = lane >> 4, i = lane & 15;
  const int b = a.bits[s];
  const int bo = a.bits[0];
  const int nwords = a.rec_bytes / 4;
  float sg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sg[e] = sgn(a, 64 * s + 4 * i + e);
  const long long stride = (long long)gridDim.x * WARPS;
  long long vec = (long long)blockIdx.x * WARPS + wl;
  long long cur_set = -1;
  // this lane's word of the record (lanes < nwords), loaded one vector ahead
  uint32_t wnext = 0u;
  if (vec < a.n_items && lane < nwords) wnext = __ldg(reinterpret_cast<const uint32_t*>(a.rec_in + (size_t)vec * a.rec_bytes) + lane);
  for (; vec < a.n_items; vec += stride) {
    const long long set = vec / a.per_set;
    if (set != cur_set) {
      build_perm(a.outliers + set * 64, sperm[wl], smask[wl], lane);
      cur_set = set;
    }
    if (lane < 16) swords[wl][lane] = lane < nwords ? wnext : 0u;
    const long long next = vec + stride;
    if (next < a.n_items && lane < nwords)
      wnext = __ldg(reinterpret_cast<const uint32_t*>(a.rec_in + (size_t)next * a.rec_bytes) + lane);
    __syncwarp();
    const float n = __half2float(__ushort_as_half((uint16_t)(swords[wl][0] >> (16 * s))));
    const int base = 32 + (s ? 64 * bo : 0) + b * 4 * i;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int bit = base + b * e;
      uint32_t w = swords[wl][bit >> 5] >> (bit & 31);
      if ((bit & 31) + b > 32) w |= swords[wl][(bit >> 5) + 1] << (32 - (bit & 31));
      v[e] = __fmul_rn(n, scent[s][w & ((1u << b) - 1u)]);
    }
    __syncwarp();
    hadamard64(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = 64 * s + 4 * i + e;
      a.out[(size_t)vec * D + (sperm[wl][p] & 127)] = __fmul_rn(__fmul_rn(v[e], 0.125f), sg[e]);
    }
  }
}

// ------------------------------------------------------------------ outlier channels of a calibration block
// one block per set, one thread per channel: sum of squares in float64 over the tokens in order,
// then the 64 largest (ties to the lower channel), written ascending
__global__ void __launch_bounds__(D) split_outliers_kernel(const void* calib, int in_bf16, int n_tokens, int16_t* out) {
  __shared__ double ss[D];
  __shared__ int isout[D];
  const int ch = threadIdx.x;
  const size_t base = (size_t)blockIdx.x * n_tokens * D;
  double acc = 0.0;
  for (int t = 0; t < n_tokens; ++t) {
    const size_t idx = base + (size_t)t * D + ch;
    const double x = in_bf16 ? (double)__bfloat162float(static_cast<const __nv_bfloat16*>(calib)[idx])
                             : (double)static_cast<const float*>(calib)[idx];
    acc = __dadd_rn(acc, __dmul_rn(x, x));
  }
  ss[ch] = acc;
  __syncthreads();
  int rank = 0;
  for (int j = 0; j < D; ++j) rank += (ss[j] > acc || (ss[j] == acc && j < ch)) ? 1 : 0;
  isout[ch] = rank < 64 ? 1 : 0;
  __syncthreads();
  if (isout[ch]) {
    int pos = 0;
    for (int j = 0; j < ch; ++j) pos += isout[j];
    if (pos < 64) out[(size_t)blockIdx.x * 64 + pos] = (int16_t)ch;  // NaN sums could break the ranking
  }
}

// ------------------------------------------------------------------ host helpers
void lloyd_max(int levels, double* cent) {
  // Lloyd's iteration on the unit Gaussian in double: boundaries at midpoints, centroids at the
  // conditional means (phi(a) - phi(b)) / (Phi(b) - Phi(a)); start evenly spaced on [-2, 2]
  const double inv_sqrt2pi = 0.3989422804014327;
  for (int k = 0; k < levels; ++k) cent[k] = -2.0 + 4.0 * k / (levels - 1);
  for (int it = 0; it < 200000; ++it) {
    double edge[MAX_LEVELS + 1], next[MAX_LEVELS];
    edge[0] = -INFINITY;
    edge[levels] = INFINITY;
    for (int k = 1; k < levels; ++k) edge[k] = 0.5 * (cent[k - 1] + cent[k]);
    double change = 0.0;
    for (int k = 0; k < levels; ++k) {
      const double lo = edge[k], hi = edge[k + 1];
      const double pa = std::isinf(lo) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * lo * lo);
      const double pb = std::isinf(hi) ? 0.0 : inv_sqrt2pi * std::exp(-0.5 * hi * hi);
      const double Fa = 0.5 * std::erfc(-lo / std::sqrt(2.0));
      const double Fb = 0.5 * std::erfc(-hi / std::sqrt(2.0));
      next[k] = (pa - pb) / (Fb - Fa);
      change = std::fmax(change, std::fabs(next[k] - cent[k]));
    }
    for (int k = 0; k < levels; ++k) cent[k] = next[k];
    if (change < 1e-15) break;
  }
}

void codebook(int bits, int dim, __half* cent, float* bnd) {
  const int L = 1 << bits;
  double c[MAX_LEVELS];
  lloyd_max(L, c);
  float cf[MAX_LEVELS];
  for (int k = 0; k < L; ++k) {
    cent[k] = __double2half(c[k] / std::sqrt((double)dim));
    cf[k] = __half2float(cent[k]);
  }
  for (int k = 0; k + 1 < L; ++k) bnd[k] = (cf[k] + cf[k + 1]) / 2.0f;
  for (int k = L - 1; k < MAX_LEVELS; ++k) bnd[k] = INFINITY;
  for (int k = L; k < MAX_LEVELS; ++k) cent[k] = __float2half(0.f);
}

void sign_bits(uint64_t seed, uint32_t* bits) {
  uint64_t state = seed;
  for (int w = 0; w < 8; ++w) bits[w] = 0u;
  for (int j = 0; j < 256; ++j) {
    state += 0x9E3779B97F4A7C15ull;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    if (z & 1) bits[j >> 5] |= 1u << (j & 31);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int grid_for(long long items) {
  const long long blocks = (items + WARPS - 1) / WARPS;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  const long long cap = sms > 0 ? (long long)sms * 8 : 1024;  // resident blocks (8 warps of 64 registers or fewer)
  return (int)(blocks < cap ? blocks : cap);
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

}  // namespace

}  // namespace kvq

using namespace kvq;

extern "C" {

size_t kv_tbq_block_bytes(int32_t bits) { return (bits == 3 || bits == 4) ? 2 + 32 * (size_t)bits : 0; }

size_t kv_split_record_bytes(int32_t hi_bits) {
  return (hi_bits == 3 || hi_bits == 4) ? 4 + 8 * (size_t)hi_bits + 8 * (size_t)(hi_bits - 1) : 0;
}

int kv_tbq_encode(int32_t bits, uint64_t seed, const void* x, int32_t in_dtype, int64_t n_blocks, void* blocks,
                  void* stream) {
  if (kv_tbq_block_bytes(bits) == 0 || (in_dtype != KVQ_IN_F32 && in_dtype != KVQ_IN_BF16)) return KVQ_ERR_UNSUPPORTED;
  if (!x || !blocks || n_blocks < 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(x)) return KVQ_ERR_ALIGN;
  if (n_blocks == 0) return KVQ_OK;
  BlockArgs a;
  std::memset(&a, 0, sizeof(a));
  sign_bits(seed, a.sign_bits);
  codebook(bits, 256, a.cent[0], a.bnd[0]);
  a.bits[0] = bits;
  a.levels[0] = 1 << bits;
  a.x = x;
  a.rec = static_cast<uint8_t*>(blocks);
  a.n_items = n_blocks;
  a.in_bf16 = in_dtype == KVQ_IN_BF16;
  a.rec_bytes = (int)kv_tbq_block_bytes(bits);
  tbq_encode_kernel<<<grid_for(n_blocks), WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status(cudaGetLastError());
}

int kv_tbq_decode(int32_t bits, uint64_t seed, const void* blocks, int64_t n_blocks, float* x, void* stream) {
  if (kv_tbq_block_bytes(bits) == 0) return KVQ_ERR_UNSUPPORTED;
  if (!x || !blocks || n_blocks < 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(x)) return KVQ_ERR_ALIGN;
  if (n_blocks == 0) return KVQ_OK;
  BlockArgs a;
  std::memset(&a, 0, sizeof(a));
  sign_bits(seed, a.sign_bits);
  codebook(bits, 256, a.cent[0], a.bnd[0]);
  a.bits[0] = bits;
  a.levels[0] = 1 << bits;
  a.rec_in = static_cast<const uint8_t*>(blocks);
  a.out = x;
  a.n_items = n_blocks;
  a.rec_bytes = (int)kv_tbq_block_bytes(bits);
  tbq_decode_kernel<<<grid_for(n_blocks), WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status(cudaGetLastError());
}

int kv_split_outliers(const void* calib, int32_t in_dtype, int32_t n_sets, int32_t n_tokens, int16_t* outliers,
                      void* stream) {
  if (in_dtype != KVQ_IN_F32 && in_dtype != KVQ_IN_BF16) return KVQ_ERR_UNSUPPORTED;
  if (!calib || !outliers || n_sets < 1 || n_tokens < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(calib) || !aligned16(outliers)) return KVQ_ERR_ALIGN;
  split_outliers_kernel<<<n_sets, D, 0, static_cast<cudaStream_t>(stream)>>>(calib, in_dtype == KVQ_IN_BF16, n_tokens,
                                                                              outliers);
  return launch_status(cudaGetLastError());
}

static int split_args(int32_t hi_bits, uint64_t seed, const int16_t* outliers, int32_t n_sets, int64_t n_vectors,
                      BlockArgs* a) {
  if (kv_split_record_bytes(hi_bits) == 0) return KVQ_ERR_UNSUPPORTED;
  if (!outliers || n_sets < 1 || n_vectors < 0 || n_vectors % n_sets != 0) return KVQ_ERR_INVALID_ARG;
  std::memset(a, 0, sizeof(*a));
  sign_bits(seed, a->sign_bits);
  codebook(hi_bits, 64, a->cent[0], a->bnd[0]);
  codebook(hi_bits - 1, 64, a->cent[1], a->bnd[1]);
  a->bits[0] = hi_bits;
  a->bits[1] = hi_bits - 1;
  a->levels[0] = 1 << hi_bits;
  a->levels[1] = 1 << (hi_bits - 1);
  a->outliers = outliers;
  a->n_items = n_vectors;
  a->per_set = n_vectors / n_sets > 0 ? n_vectors / n_sets : 1;
  a->rec_bytes = (int)kv_split_record_bytes(hi_bits);
  return KVQ_OK;
}

int kv_split_encode(int32_t hi_bits, uint64_t seed, const int16_t* outliers, int32_t n_sets, const void* x,
                    int32_t in_dtype, int64_t n_vectors, void* records, void* stream) {
  if (in_dtype != KVQ_IN_F32 && in_dtype != KVQ_IN_BF16) return KVQ_ERR_UNSUPPORTED;
  if (!x || !records) return KVQ_ERR_INVALID_ARG;
  BlockArgs a;
  int rc = split_args(hi_bits, seed, outliers, n_sets, n_vectors, &a);
  if (rc != KVQ_OK) return rc;
  if (!aligned16(x) || !aligned16(records) || !aligned16(outliers)) return KVQ_ERR_ALIGN;
  if (n_vectors == 0) return KVQ_OK;
  a.x = x;
  a.rec = static_cast<uint8_t*>(records);
  a.in_bf16 = in_dtype == KVQ_IN_BF16;
  split_encode_kernel<<<grid_for(n_vectors), WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status(cudaGetLastError());
}

int kv_split_decode(int32_t hi_bits, uint64_t seed, const int16_t* outliers, int32_t n_sets, const void* records,
                    int64_t n_vectors, float* x, void* stream) {
  if (!x || !records) return KVQ_ERR_INVALID_ARG;
  BlockArgs a;
  int rc = split_args(hi_bits, seed, outliers, n_sets, n_vectors, &a);
  if (rc != KVQ_OK) return rc;
  if (!aligned16(x) || !aligned16(records) || !aligned16(outliers)) return KVQ_ERR_ALIGN;
  if (n_vectors == 0) return KVQ_OK;
  a.rec_in = static_cast<const uint8_t*>(records);
  a.out = x;
  split_decode_kernel<<<grid_for(n_vectors), WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status(cudaGetLastError());
}

}  // extern "C"
