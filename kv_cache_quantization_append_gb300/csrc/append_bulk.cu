// Bulk append kernel for Q4G32 vectors: one thread per new token, one warp per 32-token half-page.
//
// Same codec as the per-vector append kernel ([QC] "how it works": 4-bit groups, FP32 window;
// [KV] TLDR: Walsh-Hadamard rotation, then Sinkhorn balancing, then 4-bit), same operations in
// the same order, so the stored bytes are identical; only the mapping onto the GPU differs.  For
// prefill-sized appends the per-vector kernel spends most of its issue slots on shuffles (the
// butterfly's cross-lane stages and the group reductions); here a thread holds its whole vector in
// registers, so the 7 butterfly stages, the group min/max and the codes are plain in-register
// arithmetic and a warp handles 32 vectors per instruction stream.
//
//  * A warp owns one (layer, sequence, kv-head, K|V, half-page) tile: the new tokens of the call
//    that fall into that half-page.  Their input rows are contiguous; the warp copies them into a
//    swizzled shared-memory tile (16-byte chunk c of row t at chunk c ^ (t & 7), so that each
//    thread reading its own row is conflict-free), converting bf16 to float on the way.
//  * Thread t takes the token at position 32 * half_page + t.  It writes the raw row into the
//    window ring when the token is among the call's last `window`, then sign-flips, rotates and
//    (with KVarN scales) balances it, and quantises each group of 32 channels.
//  * Code of y: the quotient (y - zero) / scale is formed as (y - zero) * RN(1/scale); where that
//    product lies within 10^-3 of a rounding boundary (or outside [0, 15]) the code is recomputed
//    from the IEEE division, so every code equals clamp(rint(RN((y - zero) / scale)), 0, 15).
//  * K records are 64 contiguous bytes per token (four 16-byte stores).  V codes of tokens 2p and
//    2p+1 share 16-byte rows; the two threads of a pair swap halves with one round of shuffles and
//    each stores four whole rows.  A token whose pair partner is not part of this call stores only
//    its own bytes.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int BW = 4;                       // warps per CTA
constexpr int ROW_BYTES = D * 4;            // one staged row of floats
constexpr int TILE_BYTES = HALF * ROW_BYTES;
constexpr int SMEM_BYTES = BW * TILE_BYTES + BW * D * 4 + D * 4;  // tiles, per-warp sigma, signs

__device__ __forceinline__ int chunk_off(int t, int c) { return t * ROW_BYTES + ((c ^ (t & 7)) << 4); }

__global__ void __launch_bounds__(BW * 32, 3) append_bulk_kernel(const __grid_constant__ AppendArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  uint8_t* tile = smem + wl * TILE_BYTES;
  float* sig = reinterpret_cast<float*>(smem + BW * TILE_BYTES) + wl * D;
  float* sgn = reinterpret_cast<float*>(smem + BW * TILE_BYTES + BW * D * 4);
  if (threadIdx.x < D) sgn[threadIdx.x] = a.p.signs[threadIdx.x];
  __syncthreads();

  const int H = a.Hkv, T = a.T;
  const int nhp = T / HALF + 2;  // half-pages one sequence's call can touch
  long long rest = (long long)blockIdx.x * BW + wl;
  const int hpi = (int)(rest % nhp);
  rest /= nhp;
  const int kv = a.kv_lo + (int)(rest % a.kv_n);
  rest /= a.kv_n;
  const int h = (int)(rest % H);
  rest /= H;
  const int b = (int)(rest % a.batch);
  const int ll = (int)(rest / a.batch);
  if (ll >= a.n_layers_call) return;
  const int layer = a.layer0 + ll;

  const int p0 = a.pos[b];
  if (p0 < 0) return;  // sequence not part of this append
  if ((long long)p0 + T > a.max_seq_len) {
    if (lane == 0 && hpi == 0 && kv == a.kv_lo && h == 0) atomicOr(a.p.status, KVQ_DEV_POS_RANGE);
    return;
  }
  const int hp = p0 / HALF + hpi;
  const int lo_pos = max(p0, hp * HALF), hi_pos = min(p0 + T, hp * HALF + HALF);
  if (lo_pos >= hi_pos) return;
  const int phys = a.block_table[(size_t)b * a.L.max_pages_per_seq + hp / 2];
  if (phys < 0 || phys >= a.L.n_pages) {
    if (lane == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
    return;
  }
  uint8_t* pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
                (size_t)(hp & 1) * a.L.half_bytes;

  // ---- stage rows [lo_pos, hi_pos) (input rows lo_pos - p0 ..) into the tile, as floats
  const int r0 = lo_pos - hp * HALF, nrows = hi_pos - lo_pos;
  const size_t row0 = (((size_t)ll * a.batch + b) * H + h) * T + (lo_pos - p0);
  const void* src = kv ? a.v : a.k;
  // all of a lane's loads are issued before the first shared-memory store, so the tile arrives in
  // about one memory latency
  if (a.in_bf16) {
    const uint4* g = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + row0 * D);
    const int nchunk = nrows * 16;  // 16-byte chunks of 8 bf16
    uint4 u[16];
#pragma unroll
    for (int it = 0; it < 16; ++it)
      if (lane + 32 * it < nchunk) u[it] = __ldcs(g + lane + 32 * it);
#pragma unroll
    for (int it = 0; it < 16; ++it) {
      const int idx = lane + 32 * it;
      if (idx < nchunk) {
        const int t = r0 + (idx >> 4), c8 = idx & 15;
        *reinterpret_cast<float4*>(tile + chunk_off(t, 2 * c8)) =
            make_float4(__uint_as_float(u[it].x << 16), __uint_as_float(u[it].x & 0xffff0000u),
                        __uint_as_float(u[it].y << 16), __uint_as_float(u[it].y & 0xffff0000u));
        *reinterpret_cast<float4*>(tile + chunk_off(t, 2 * c8 + 1)) =
            make_float4(__uint_as_float(u[it].z << 16), __uint_as_float(u[it].z & 0xffff0000u),
                        __uint_as_float(u[it].w << 16), __uint_as_float(u[it].w & 0xffff0000u));
      }
    }
  } else {
    const uint4* g = reinterpret_cast<const uint4*>(static_cast<const float*>(src) + row0 * D);
    const int nchunk = nrows * 32;  // 16-byte chunks of 4 floats
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint4 u[16];
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int idx = lane + 32 * (16 * half + it);
        if (idx < nchunk) u[it] = __ldcs(g + idx);
      }
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int idx = lane + 32 * (16 * half + it);
        if (idx < nchunk) *reinterpret_cast<uint4*>(tile + chunk_off(r0 + (idx >> 5), idx & 31)) = u[it];
      }
    }
  }
  if (a.sinkhorn) {
    const __half* sg = (kv ? a.p.sigv : a.p.sigk) + ((size_t)layer * H + h) * D;
    for (int j = lane; j < D; j += 32) sig[j] = __half2float(sg[j]);
  }
  __syncwarp();

  const int pos = hp * HALF + lane;
  const bool valid = pos >= lo_pos && pos < hi_pos;
  uint32_t W[16] = {};    // channel words: nibble m of W[n] = code of channel 8n + m
  uint32_t meta[4] = {};  // fp16 {scale, zero} of group G packed as scale | zero << 16
  if (valid) {
    float x[D];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float4 v = *reinterpret_cast<const float4*>(tile + chunk_off(lane, c));
      x[4 * c] = v.x;
      x[4 * c + 1] = v.y;
      x[4 * c + 2] = v.z;
      x[4 * c + 3] = v.w;
    }
    // raw copy into the window ring for the last `window` tokens of this call
    if (a.W > 0 && pos - p0 >= T - a.W) {
      float* ring = kv ? a.p.ringv : a.p.ringk;
      float4* dst = reinterpret_cast<float4*>(
          ring + ((((size_t)layer * a.max_batch + b) * H + h) * a.W + (size_t)(pos % a.W)) * D);
#pragma unroll
      for (int c = 0; c < 32; ++c) dst[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
    }
    // rotation y = c * H (s . x): sign flip (exact), butterfly stages h = 1 .. 64, one multiply by c
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float4 s = *reinterpret_cast<const float4*>(sgn + 4 * c);
      x[4 * c] = __fmul_rn(x[4 * c], s.x);
      x[4 * c + 1] = __fmul_rn(x[4 * c + 1], s.y);
      x[4 * c + 2] = __fmul_rn(x[4 * c + 2], s.z);
      x[4 * c + 3] = __fmul_rn(x[4 * c + 3], s.w);
    }
#pragma unroll
    for (int hs = 1; hs < D; hs <<= 1) {
#pragma unroll
      for (int j = 0; j < D; ++j) {
        if (j & hs) continue;
        const float u = x[j], v = x[j + hs];
        x[j] = __fadd_rn(u, v);
        x[j + hs] = __fsub_rn(u, v);
      }
    }
#pragma unroll
    for (int j = 0; j < D; ++j) x[j] = __fmul_rn(x[j], C_WHT);
    if (a.sinkhorn) {
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float4 s = *reinterpret_cast<const float4*>(sig + 4 * c);
        x[4 * c] = __fdiv_rn(x[4 * c], s.x);
        x[4 * c + 1] = __fdiv_rn(x[4 * c + 1], s.y);
        x[4 * c + 2] = __fdiv_rn(x[4 * c + 2], s.z);
        x[4 * c + 3] = __fdiv_rn(x[4 * c + 3], s.w);
      }
    }
    // ---- Q4G32 per group: exact min/max, fp16 scale (max-min)/15 and zero min, codes
    uint32_t fix[4];
    float sc[4], zr[4];
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      float mn = x[32 * G], mx = x[32 * G];
#pragma unroll
      for (int e = 1; e < 32; ++e) {
        mn = fminf(mn, x[32 * G + e]);
        mx = fmaxf(mx, x[32 * G + e]);
      }
      const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.0f));
      const __half z16 = __float2half_rn(mn);
      meta[G] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
      const float s = __half2float(s16), z = __half2float(z16);
      sc[G] = s;
      zr[G] = z;
      const float inv = __frcp_rn(s);
      uint32_t f = 0;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        uint32_t w = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int e = 8 * n + m;
          const float qt = __fmul_rn(__fsub_rn(x[32 * G + e], z), inv);
          const float r = rintf(qt);
          const bool bad = fabsf(__fsub_rn(qt, r)) > 0.499f || !(r >= 0.0f && r <= 15.0f);
          f |= (bad ? 1u : 0u) << e;
          w |= ((uint32_t)__float2int_rz(bad ? 0.0f : r)) << (4 * m);
        }
        W[4 * G + n] = s > 0.0f ? w : 0u;
      }
      fix[G] = s > 0.0f ? f : 0u;
    }
    if (fix[0] | fix[1] | fix[2] | fix[3]) {
      // rare: redo the flagged codes from the IEEE quotient; the rotated row goes to this thread's
      // own tile row so that a flagged channel can be read by index
      float* row = reinterpret_cast<float*>(tile + lane * ROW_BYTES);
#pragma unroll
      for (int j = 0; j < D; ++j) row[j] = x[j];
#pragma unroll
      for (int G = 0; G < 4; ++G) {
        uint32_t f = fix[G];
        while (f) {
          const int e = __ffs(f) - 1;
          f &= f - 1;
          const float qt = __fdiv_rn(__fsub_rn(row[32 * G + e], zr[G]), sc[G]);
          const uint32_t c = (uint32_t)min(max(__float2int_rn(qt), 0), 15);
          const int n = e >> 3, sh = 4 * (e & 7);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (k == n) W[4 * G + k] = (W[4 * G + k] & ~(15u << sh)) | (c << sh);
        }
      }
    }
  }
  const int tin = lane;  // token index within the half-page
  if (kv == 0) {
    if (valid) {
      // K record: 32-bit word (i, G) at byte 16i + 4G holds channels 32G + 8i .. +7 = W[4G + i]
      uint4* rec = reinterpret_cast<uint4*>(pg + (size_t)tin * 64);
#pragma unroll
      for (int i = 0; i < 4; ++i) rec[i] = make_uint4(W[i], W[4 + i], W[8 + i], W[12 + i]);
      *reinterpret_cast<uint4*>(pg + a.L.off_kmeta + (size_t)tin * 16) =
          make_uint4((meta[0] & 0xffffu) | (meta[1] << 16), (meta[2] & 0xffffu) | (meta[3] << 16),
                     (meta[0] >> 16) | (meta[1] & 0xffff0000u), (meta[2] >> 16) | (meta[3] & 0xffff0000u));
    }
    return;
  }
  // ---- V: tokens 2p, 2p+1 share 128 bytes; row R of group G sits at 16 * ((R + 2 * (p & 3)) & 7) + 4G
  // as bytes [t0 byte0, t1 byte0, t0 byte1, t1 byte1] of the halfword hw(R, G) = channels
  // 32G + 4R .. +3 = half (R & 1) of W[4G + R / 2].  The even token stores rows 0-3, the odd one
  // rows 4-7, each with its partner's halfwords for those rows.
  const bool odd = lane & 1;
  const bool paired = valid && (__shfl_xor_sync(FULL, valid ? 1 : 0, 1) != 0);
  uint32_t M[4][2], P[4][2];
#pragma unroll
  for (int G = 0; G < 4; ++G)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      M[G][q] = odd ? W[4 * G + 2 + q] : W[4 * G + q];
      P[G][q] = __shfl_xor_sync(FULL, odd ? W[4 * G + q] : W[4 * G + 2 + q], 1);
    }
  uint8_t* vmain = pg + a.L.off_vmain;
  const int pp = tin >> 1;
  if (paired) {
    const uint32_t sel0 = odd ? 0x1504u : 0x5140u, sel1 = odd ? 0x3726u : 0x7362u;
    const int R0 = odd ? 4 : 0;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int R = R0 + rr, q = rr >> 1;
      const uint32_t sel = (rr & 1) ? sel1 : sel0;
      const uint4 row = make_uint4(__byte_perm(M[0][q], P[0][q], sel), __byte_perm(M[1][q], P[1][q], sel),
                                   __byte_perm(M[2][q], P[2][q], sel), __byte_perm(M[3][q], P[3][q], sel));
      *reinterpret_cast<uint4*>(vmain + (size_t)pp * 128 + 16 * ((R + 2 * (pp & 3)) & 7)) = row;
    }
  } else if (valid) {
#pragma unroll
    for (int R = 0; R < 8; ++R)
#pragma unroll
      for (int G = 0; G < 4; ++G) {
        const uint32_t hw = (W[4 * G + (R >> 1)] >> (16 * (R & 1))) & 0xffffu;
        uint8_t* dst = vmain + (size_t)pp * 128 + 16 * ((R + 2 * (pp & 3)) & 7) + 4 * G + (tin & 1);
        dst[0] = (uint8_t)(hw & 0xffu);
        dst[2] = (uint8_t)(hw >> 8);
      }
  }
  if (valid) {
    // V meta: group-major scale[4][32] then zero[4][32]
    uint16_t* vm = reinterpret_cast<uint16_t*>(pg + a.L.off_vmeta);
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      vm[G * HALF + tin] = (uint16_t)(meta[G] & 0xffffu);
      vm[4 * HALF + G * HALF + tin] = (uint16_t)(meta[G] >> 16);
    }
  }
}

}  // namespace

cudaError_t launch_append_bulk(const AppendArgs& a, cudaStream_t s) {
  const long long warps = (long long)a.n_layers_call * a.batch * a.Hkv * a.kv_n * (a.T / HALF + 2);
  const long long blocks = (warps + BW - 1) / BW;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  static bool attr_set = false;  // per process; the attribute is a property of the kernel
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(append_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  append_bulk_kernel<<<(unsigned)blocks, BW * 32, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
