// Append kernel: rotate, balance and quantise new K/V vectors into their pages, and keep the
// most recent ones raw in the window ring.
//
// [QC] "how it works": 4-bit everywhere except a 128-token FP32 window; v3.2 note: a batched
// write equals per-token writes bit for bit (here each token's record depends on that token only,
// and the ring is written only for the last `window` tokens of a call, so no two threads of one
// call write the same slot).
// [KV] TLDR: Walsh-Hadamard rotation, then Sinkhorn per-channel balancing, then 4-bit.
// [TQ] "key idea" row: random rotation, per-coordinate optimal scalar quantiser, 1-bit QJL
// sketch of the residual.
//
// One warp per (layer, sequence, kv-head, token, K|V) vector; lane l holds channels 4l..4l+3.
// Every floating-point step is one IEEE operation (explicit _rn intrinsics: no contraction), in
// the order the codec defines, so codes are reproducible bit for bit.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int WARPS = 8;

__device__ __forceinline__ uint32_t h16(__half h) { return (uint32_t)__half_as_ushort(h); }

// Q4G32: per group of 32 channels exact min/max, fp16 scale (max-min)/15 and zero min, codes
// clamp(rint((y - zero) / scale), 0, 15); 0 when the scale is 0.
__device__ __forceinline__ void q4_encode(const float (&y)[4], int lane, int kv, int tin, uint8_t* main,
                                          __half& s16, __half& z16) {
  float mn = fminf(fminf(y[0], y[1]), fminf(y[2], y[3]));
  float mx = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {  // lanes 8G .. 8G+7 hold group G
    mn = fminf(mn, __shfl_xor_sync(FULL, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, m));
  }
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
  z16 = __float2half_rn(mn);
  const float s = __half2float(s16), z = __half2float(z16);
  // code = clamp(rint(RN((y - z) / s)), 0, 15).  The quotient is first formed as (y - z) * RN(1/s),
  // within a few ulp of the IEEE quotient (|q| < 2^5, so well under 2^-17 away); its rounding to an
  // integer can differ from the IEEE quotient's only within that distance of a half-integer, and
  // there the IEEE division is done instead, so the code equals the exact definition.
  const float inv = __frcp_rn(s);
  uint32_t hw = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int c = 0;
    if (s > 0.0f) {
      const float num = __fsub_rn(y[e], z);
      float qt = __fmul_rn(num, inv);
      if (fabsf(qt - rintf(qt)) > 0.499f) qt = __fdiv_rn(num, s);
      c = min(max(__float2int_rn(qt), 0), 15);
    }
    hw |= (uint32_t)c << (4 * e);
  }
  // lane 8G + r holds channels 32G + 4r .. +3 as the halfword hw (byte 0: channels +0,+1; byte 1: +2,+3)
  if (kv == 0) {
    // K record (64 B per token at 64 * tin): 32-bit word (i, G) at byte 16i + 4G holds channels
    // 32G + 8i .. +7, i.e. the halfwords of lanes 8G + 2i (low) and 8G + 2i + 1 (high)
    const int j = lane & 15, i = j >> 2, G = j & 3;
    const uint32_t lo = __shfl_sync(FULL, hw, 8 * G + 2 * i);
    const uint32_t hi = __shfl_sync(FULL, hw, 8 * G + 2 * i + 1);
    if (lane < 16) reinterpret_cast<uint32_t*>(main + (size_t)tin * 64)[j] = lo | (hi << 16);
  } else {
    // V region: tokens 2p, 2p+1 share a 128-byte block; row r (= lane & 7) of group G sits at
    // 16 * ((r + 2 * (p & 3)) & 7) + 4G as bytes [t0 byte0, t1 byte0, t0 byte1, t1 byte1]
    const int r = lane & 7, G = lane >> 3, pp = tin >> 1, slot = tin & 1;
    uint8_t* dst = main + (size_t)pp * 128 + 16 * ((r + 2 * (pp & 3)) & 7) + 4 * G + slot;
    dst[0] = (uint8_t)(hw & 0xffu);
    dst[2] = (uint8_t)(hw >> 8);
  }
}

// Q8G32 key: per group of 32 channels (lanes 8G .. 8G+7) d = fp16(max |y| / 127) and codes
// clamp(rint(y / d), -127, 127) with round-half-even (IEEE division by the stored scale), 0 when
// d == 0; stored as u = c + 128.  Record of token t (128 B): chunk m = 2i + h at 16 (m ^ (t & 1)),
// word w of the chunk = channels k + 2i, k + 2i + 1, k + 2i + 8, k + 2i + 9 with k = 16 (4h + w).
__device__ __forceinline__ void q8_encode_key(const float (&y)[4], int lane, int tin, uint8_t* kmain,
                                              uint8_t* kmeta) {
  float amax = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, m));
  const __half d16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float d = __half2float(d16);
  uint8_t* rec = kmain + (size_t)tin * 128;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int c = 0;
    if (d > 0.0f) c = min(max(__float2int_rn(__fdiv_rn(y[e], d)), -127), 127);
    const int ch = 4 * lane + e, kk = ch >> 4, within = ch & 15;
    const int i = (within & 7) >> 1, byte = (within & 1) + ((within >> 3) << 1);
    const int m = 2 * i + (kk >> 2), w = kk & 3;
    rec[16 * (m ^ (tin & 1)) + 4 * w + byte] = (uint8_t)(c + 128);
  }
  if ((lane & 7) == 0) reinterpret_cast<__half*>(kmeta + (size_t)tin * 8)[lane >> 3] = d16;
}

constexpr int VPW = 4;  // vectors (consecutive tokens) per warp: their loads are issued together

// encode one vector (lane holds channels 4*lane..+3 of the raw input) into its page and ring slot
__device__ __forceinline__ void encode_vector(const AppendArgs& a, int lane, int kv, int layer, int b, int h,
                                              int t, int p, float4 xin) {
  const int H = a.Hkv;
  // raw copy into the window ring for the last `window` tokens of this call
  if (a.W > 0 && t >= a.T - a.W) {
    float* ring = kv ? a.p.ringv : a.p.ringk;
    const size_t slot = (size_t)(p % a.W);
    float* dst = ring + ((((size_t)layer * a.max_batch + b) * H + h) * a.W + slot) * D + 4 * lane;
    *reinterpret_cast<float4*>(dst) = xin;
  }

  const int lp = p / PAGE, tin = p % HALF;
  const int phys = a.block_table[(size_t)b * a.L.max_pages_per_seq + lp];
  if (phys < 0 || phys >= a.L.n_pages) {
    if (lane == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
    return;
  }
  // the half-page holding this token: K main | V main | K meta | V meta for 32 tokens
  uint8_t* pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
                (size_t)((p % PAGE) / HALF) * a.L.half_bytes;

  // rotation y = c * H (s . x): sign flip (exact), butterfly, one multiply by c
  const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
  float y0 = __fmul_rn(xin.x, sg.x), y1 = __fmul_rn(xin.y, sg.y);
  float y2 = __fmul_rn(xin.z, sg.z), y3 = __fmul_rn(xin.w, sg.w);
  hadamard_warp(y0, y1, y2, y3, lane);
  float y[4] = {__fmul_rn(y0, C_WHT), __fmul_rn(y1, C_WHT), __fmul_rn(y2, C_WHT), __fmul_rn(y3, C_WHT)};

  // ---- Q4G32 or Q8G32 (optionally Sinkhorn-balanced: y / sigma per channel)
  if (a.sinkhorn) {
    const __half* sig = (kv ? a.p.sigv : a.p.sigk) + ((size_t)layer * H + h) * D + 4 * lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = __fdiv_rn(y[e], __half2float(sig[e]));
  }
  if (kv == 0 && a.k_format == KVQ_Q8G32) {
    q8_encode_key(y, lane, tin, pg, pg + a.L.off_kmeta);
    return;
  }
  __half s16, z16;
  q4_encode(y, lane, kv, tin, pg + (kv ? a.L.off_vmain : 0), s16, z16);
  if (kv == 0) {
    // K meta: per token {scale[4], zero[4]} fp16
    const uint32_t sz = h16(s16) | (h16(z16) << 16);
    const uint32_t g0 = __shfl_sync(FULL, sz, 0), g1 = __shfl_sync(FULL, sz, 8);
    const uint32_t g2 = __shfl_sync(FULL, sz, 16), g3 = __shfl_sync(FULL, sz, 24);
    if (lane == 0)
      *reinterpret_cast<uint4*>(pg + a.L.off_kmeta + (size_t)tin * 16) =
          make_uint4((g0 & 0xffffu) | (g1 << 16), (g2 & 0xffffu) | (g3 << 16), (g0 >> 16) | (g1 & 0xffff0000u),
                     (g2 >> 16) | (g3 & 0xffff0000u));
  } else if ((lane & 7) == 0) {
    // V meta: group-major scale[4][32] then zero[4][32]
    __half* meta = reinterpret_cast<__half*>(pg + a.L.off_vmeta);
    const int G = lane >> 3;
    meta[G * HALF + tin] = s16;
    meta[4 * HALF + G * HALF + tin] = z16;
  }
}

__device__ __forceinline__ void append_warps_body(const AppendArgs& a) {
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  // a dependent decode launch may start its set-up now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  const int nq = (a.T + VPW - 1) / VPW;
  // 32-bit index arithmetic: the launcher keeps the warp count below 2^31
  const unsigned total = (unsigned)a.n_layers_call * a.batch * a.Hkv * nq * a.kv_n;
  const unsigned wid = blockIdx.x * WARPS + wl;
  if (wid >= total) return;
  const int kv = a.kv_lo + (int)(wid % a.kv_n);
  unsigned rest = wid / a.kv_n;
  const int tq = (int)(rest % nq);
  rest /= nq;
  const int h = (int)(rest % a.Hkv);
  rest /= a.Hkv;
  const int b = (int)(rest % a.batch);
  const int ll = (int)(rest / a.batch);
  const int layer = a.layer0 + ll;

  const int p0 = a.pos[b];
  if (p0 < 0) return;  // sequence not part of this append
  if ((long long)p0 + a.T > a.max_seq_len) {
    if (lane == 0 && tq == 0 && kv == 0 && h == 0) atomicOr(a.p.status, KVQ_DEV_POS_RANGE);
    return;
  }
  const int t0 = tq * VPW;
  const int nv = min(VPW, a.T - t0);
  const size_t vec0 = (((size_t)ll * a.batch + b) * a.Hkv + h) * a.T + t0;
  float4 x[VPW];
#pragma unroll
  for (int j = 0; j < VPW; ++j)
    if (j < nv) x[j] = load4_in(kv ? a.v : a.k, (vec0 + j) * D + 4 * lane, a.in_bf16);
#pragma unroll
  for (int j = 0; j < VPW; ++j)
    if (j < nv) encode_vector(a, lane, kv, layer, b, h, t0 + j, p0 + t0 + j, x[j]);
}

// As append_bulk_kernel: launched for the values of a TurboQuant-key append (AFTER_KEYS) as a
// programmatic dependent of the keys kernel, every thread waits for the keys grid before exiting.
template <bool AFTER_KEYS>
__global__ void __launch_bounds__(WARPS * 32) append_kernel(const AppendArgs a) {
  append_warps_body(a);
  if (AFTER_KEYS) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- TurboQuant keys
// [TQ] "key idea" row: unit vector, 3-bit Lloyd-Max codes, then the 1-bit QJL sketch of the
// residual: bit i = (t_i >= 0), t_i = sum over j = 0..127 in order of RN(S[i][j] * r_j).  The
// projection (128 x 128 separately rounded multiplies and adds per vector, in that order, so the
// signs are reproducible bit for bit) is the cost: the transposed projection is staged in shared
// memory once per CTA and every warp streams TQ_VPW vectors (one, for appends of fewer tokens per
// sequence) through it, the residuals read as
// broadcast shared-memory words, the products and sums as packed f32x2 operations (each half
// rounded like the scalar operation).
constexpr int TQ_WARPS = 8;
constexpr int TQ_VPW = 4;
constexpr size_t TQ_SMEM = (size_t)(D * D + TQ_WARPS * TQ_VPW * D) * sizeof(float);

struct TqKey {
  uint8_t* pg;     // the token's half-page (nullptr: no record written)
  int tin;         // token within the half-page
  uint32_t c12;    // this lane's four 3-bit codes
  float n, gamma;  // norm and residual norm
};

// Ring copy, page lookup, rotation, norm, codes and residual of one key vector; the residual
// (channels 4 lane .. +3) goes to rs[4 lane ..].
__device__ __forceinline__ TqKey tq_key_prepare(const AppendArgs& a, int lane, int layer, int b, int h, int t, int p,
                                                float4 xin, float* rs) {
  TqKey k{nullptr, p % HALF, 0u, 0.f, 0.f};
  const int H = a.Hkv;
  if (a.W > 0 && t >= a.T - a.W) {
    float* dst = a.p.ringk + ((((size_t)layer * a.max_batch + b) * H + h) * a.W + (size_t)(p % a.W)) * D + 4 * lane;
    *reinterpret_cast<float4*>(dst) = xin;
  }
  const int phys = a.block_table[(size_t)b * a.L.max_pages_per_seq + p / PAGE];
  if (phys < 0 || phys >= a.L.n_pages) {
    if (lane == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
  } else {
    k.pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
           (size_t)((p % PAGE) / HALF) * a.L.half_bytes;
  }
  // rotation y = c * H (s . x): sign flip (exact), butterfly, one multiply by c
  const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
  float y0 = __fmul_rn(xin.x, sg.x), y1 = __fmul_rn(xin.y, sg.y);
  float y2 = __fmul_rn(xin.z, sg.z), y3 = __fmul_rn(xin.w, sg.w);
  hadamard_warp(y0, y1, y2, y3, lane);
  const float y[4] = {__fmul_rn(y0, C_WHT), __fmul_rn(y1, C_WHT), __fmul_rn(y2, C_WHT), __fmul_rn(y3, C_WHT)};
  const CodebookDev* cb = a.p.cb;
  k.n = __fsqrt_rn(sumsq_warp(y[0], y[1], y[2], y[3]));
  const float inv = __fdiv_rn(1.0f, fmaxf(k.n, FLT_MIN));
  float r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float u = __fmul_rn(y[e], inv);
    int code = 0;
#pragma unroll
    for (int q = 0; q < 7; ++q) code += (cb->bnd[q] <= u) ? 1 : 0;
    r[e] = __fsub_rn(u, __half2float(cb->cent[code]));
    k.c12 |= (uint32_t)code << (3 * e);
  }
  k.gamma = __fsqrt_rn(sumsq_warp(r[0], r[1], r[2], r[3]));
  *reinterpret_cast<float4*>(rs + 4 * lane) = make_float4(r[0], r[1], r[2], r[3]);
  return k;
}

template <int VPW>
__global__ void __launch_bounds__(TQ_WARPS * 32) append_tq_keys_kernel(const AppendArgs a) {
  extern __shared__ __align__(16) float tq_smem[];
  const float* sT = tq_smem;  // [j][i] = S[i][j]
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  float* rs = tq_smem + D * D + wl * TQ_VPW * D;  // this warp's residuals [VPW][128]
  // a dependent decode launch may start its set-up now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  // the transposed projection, 64 KB: each thread's 16 rows of 16 bytes requested 8 at a time
  // before any is stored
  constexpr int STAGE_N = D * D / 4 / (TQ_WARPS * 32), STAGE_BATCH = 8;
  static_assert(STAGE_N % STAGE_BATCH == 0, "whole batches");
#pragma unroll 1
  for (int r0 = 0; r0 < STAGE_N; r0 += STAGE_BATCH) {
    float4 t[STAGE_BATCH];
#pragma unroll
    for (int r = 0; r < STAGE_BATCH; ++r)
      t[r] = reinterpret_cast<const float4*>(a.p.qjl_t)[threadIdx.x + (r0 + r) * TQ_WARPS * 32];
#pragma unroll
    for (int r = 0; r < STAGE_BATCH; ++r) reinterpret_cast<float4*>(tq_smem)[threadIdx.x + (r0 + r) * TQ_WARPS * 32] = t[r];
  }
  __syncthreads();
  const int nq = (a.T + VPW - 1) / VPW;
  const unsigned total = (unsigned)a.n_layers_call * a.batch * a.Hkv * nq;
  for (unsigned wid = blockIdx.x * TQ_WARPS + wl; wid < total; wid += gridDim.x * TQ_WARPS) {
    const int tq = (int)(wid % nq);
    unsigned rest = wid / nq;
    const int h = (int)(rest % a.Hkv);
    rest /= a.Hkv;
    const int b = (int)(rest % a.batch);
    const int ll = (int)(rest / a.batch);
    const int layer = a.layer0 + ll;
    const int p0 = a.pos[b];
    if (p0 < 0) continue;  // sequence not part of this append
    if ((long long)p0 + a.T > a.max_seq_len) {
      if (lane == 0 && tq == 0 && h == 0) atomicOr(a.p.status, KVQ_DEV_POS_RANGE);
      continue;
    }
    const int t0 = tq * VPW;
    const int nv = min(VPW, a.T - t0);
    const size_t vec0 = (((size_t)ll * a.batch + b) * a.Hkv + h) * a.T + t0;
    float4 x[VPW];
#pragma unroll
    for (int v = 0; v < VPW; ++v)
      if (v < nv) x[v] = load4_in(a.k, (vec0 + v) * D + 4 * lane, a.in_bf16);
    TqKey key[VPW];
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      if (v < nv) {
        key[v] = tq_key_prepare(a, lane, layer, b, h, t0 + v, p0 + t0 + v, x[v], rs + v * D);
      } else {
        key[v] = TqKey{nullptr, 0, 0u, 0.f, 0.f};
        *reinterpret_cast<float4*>(rs + v * D + 4 * lane) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncwarp();
    // t_i for i = 4 lane + e, e = 0..3, of each vector: pairs (0, 1) and (2, 3) packed
    float acc[VPW][4];
#pragma unroll
    for (int v = 0; v < VPW; ++v) acc[v][0] = acc[v][1] = acc[v][2] = acc[v][3] = 0.f;
    // the next quad's projection rows are read while the current quad's are used
    float4 s4n[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) s4n[e] = *reinterpret_cast<const float4*>(sT + e * D + 4 * lane);
#pragma unroll 2
    for (int jq = 0; jq < D / 4; ++jq) {
      float4 s4q[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) s4q[e] = s4n[e];
      if (jq + 1 < D / 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s4n[e] = *reinterpret_cast<const float4*>(sT + (4 * jq + 4 + e) * D + 4 * lane);
      }
      float4 r4[VPW];
#pragma unroll
      for (int v = 0; v < VPW; ++v) r4[v] = *reinterpret_cast<const float4*>(rs + v * D + 4 * jq);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 s4 = s4q[e];
#pragma unroll
        for (int v = 0; v < VPW; ++v) {
          const float rj = e == 0 ? r4[v].x : e == 1 ? r4[v].y : e == 2 ? r4[v].z : r4[v].w;
          float p0v = s4.x, p1v = s4.y, p2v = s4.z, p3v = s4.w;
          mul2(p0v, p1v, rj, rj);
          mul2(p2v, p3v, rj, rj);
          add2(acc[v][0], acc[v][1], p0v, p1v);
          add2(acc[v][2], acc[v][3], p2v, p3v);
        }
      }
    }
    // record byte 2 lane + e holds the codes of channels 4 lane + 2e, +1 (bits 0-2, 3-5) and the
    // sign bits of projections 4 lane + 2e, +1 (bits 6, 7): this lane's halfword
#pragma unroll
    for (int v = 0; v < VPW; ++v) {
      if (key[v].pg == nullptr) continue;
      uint32_t hw = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t code = (key[v].c12 >> (3 * e)) & 7u, bitv = acc[v][e] >= 0.0f ? 1u : 0u;
        hw |= (code << (8 * (e >> 1) + 3 * (e & 1))) | (bitv << (8 * (e >> 1) + 6 + (e & 1)));
      }
      reinterpret_cast<uint16_t*>(key[v].pg + (size_t)key[v].tin * 64)[lane] = (uint16_t)hw;
      if (lane == 0) {
        __half* meta = reinterpret_cast<__half*>(key[v].pg + a.L.off_kmeta);
        meta[key[v].tin] = __float2half_rn(key[v].n);
        meta[HALF + key[v].tin] = __float2half_rn(key[v].gamma);
      }
    }
    __syncwarp();  // the residual buffer is reused by the next group
  }
}

}  // namespace

cudaError_t launch_append_warps(const AppendArgs& a, cudaStream_t s, bool after_keys) {
  const long long warps = (long long)a.n_layers_call * a.batch * a.Hkv * ((a.T + VPW - 1) / VPW) * a.kv_n;
  const long long blocks = (warps + WARPS - 1) / WARPS;
  if (blocks <= 0) return cudaSuccess;
  if (warps > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(WARPS * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_keys ? 1 : 0;
  return after_keys ? cudaLaunchKernelEx(&cfg, append_kernel<true>, a) : cudaLaunchKernelEx(&cfg, append_kernel<false>, a);
}

cudaError_t launch_append_tq_keys(const AppendArgs& a, cudaStream_t s) {
  // a warp projects TQ_VPW vectors of a sequence at a time; appends of fewer tokens per sequence
  // (the decode step's one token) one vector per warp, so that no lane computes empty slots
  const int vpw = a.T >= TQ_VPW ? TQ_VPW : 1;
  const long long warps = (long long)a.n_layers_call * a.batch * a.Hkv * ((a.T + vpw - 1) / vpw);
  if (warps <= 0) return cudaSuccess;
  if (warps > 0x7fffffffLL) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(vpw == TQ_VPW ? (const void*)append_tq_keys_kernel<TQ_VPW> : (const void*)append_tq_keys_kernel<1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TQ_SMEM);
  if (e != cudaSuccess) return e;
  // the projection is loaded once per CTA: at most two CTAs per SM, each looping over warp groups
  const long long want = (warps + TQ_WARPS - 1) / TQ_WARPS;
  const long long cap = 2LL * (sms > 0 ? sms : 1);
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  if (vpw == TQ_VPW) append_tq_keys_kernel<TQ_VPW><<<grid, TQ_WARPS * 32, TQ_SMEM, s>>>(a);
  else append_tq_keys_kernel<1><<<grid, TQ_WARPS * 32, TQ_SMEM, s>>>(a);
  return cudaGetLastError();
}

// Appends of at least BULK_MIN_T tokens per sequence go to the four-lanes-per-token kernel
// (append_bulk.cu) for Q4G32 and Q8G32 vectors; shorter ones to the warp-per-vector kernel above;
// TurboQuant keys of any length to append_tq_keys_kernel.  All write identical bytes.
constexpr int BULK_MIN_T = 16;

cudaError_t launch_append(const AppendArgs& a0, cudaStream_t s) {
  AppendArgs a = a0;
  // the bulk kernel's grid has y = (layer, kv-head, K|V) and z = sequence (at most 65535 each)
  if (a.T < BULK_MIN_T || (long long)a.n_layers_call * a.Hkv * 2 > 65535 || a.batch > 65535) {
    if (a.k_format == KVQ_TQ3_QJL) {
      const cudaError_t e = launch_append_tq_keys(a, s);
      if (e != cudaSuccess) return e;
      a.kv_lo = 1;
      a.kv_n = 1;
      return launch_append_warps(a, s, true);
    }
    a.kv_lo = 0;
    a.kv_n = 2;
    return launch_append_warps(a, s, false);
  }
  if (a.k_format == KVQ_TQ3_QJL) {
    const cudaError_t e = launch_append_tq_keys(a, s);
    if (e != cudaSuccess) return e;
    a.kv_lo = 1;
    a.kv_n = 1;
    return launch_append_bulk(a, s, true);
  }
  a.kv_lo = 0;
  a.kv_n = 2;
  return launch_append_bulk(a, s, false);
}

}  // namespace kvq
