// Bulk append kernel for Q4G32 vectors and Q8G32 keys: four lanes per new token, eight tokens per
// warp.
//
// Same codec as the per-vector append kernel ([QC] "how it works": 4-bit groups, FP32 window;
// [KV] TLDR: Walsh-Hadamard rotation, then Sinkhorn balancing, then 4-bit), same operations in
// the same order, so the stored bytes are identical; only the mapping onto the GPU differs.  For
// prefill-sized appends the per-vector kernel spends most of its issue slots on shuffles (five of
// the seven butterfly stages and the group reductions cross lanes).  Here lane 4v + G of a warp
// holds channels 32G .. 32G+31 of the warp's token v, which is exactly one quantisation group:
//  * butterfly stages h = 1 .. 16 stay inside the lane; h = 32 and 64 pair lane G with G ^ 1 and
//    G ^ 2 (one shuffle per value, combined as fma(mine, +-1, partner), whose single rounding is
//    that of the plain add or subtract since the product by +-1 is exact);
//  * the group min/max, scale, zero and codes need no other lane;
//  * a lane holds 32 values (64 registers: 32 warps per SM), and the code is small.
//
// Work unit: 8 consecutive positions (aligned to 8, so that a V token pair 2p, 2p+1 is always in
// one warp) of one (layer, sequence, kv-head, K|V).  fp32 inputs: one unit per warp, inputs read
// straight from global memory.  bf16 inputs: a pipelined form in which each warp codes 16
// consecutive units and copies the next unit's inputs into shared memory (cp.async, one 512-byte
// run of the unit per instruction) while it codes the current one, so the DRAM latency is paid
// once per 16 units instead of once per unit.
//
// Code of y: the quotient (y - zero) / scale is formed as (y - zero) * rcp(scale), with rcp the
// hardware reciprocal (within 1 ulp, relative 2^-23), which for |q| <= 16 is within 3.9e-6 of the
// IEEE quotient RN((y - zero) / scale) (the product's and the quotient's roundings of relative
// 2^-24 and the reciprocal's 2^-23); rint is taken on the FMA pipe as (q + 1.5 * 2^23) - 1.5 * 2^23.
// Where q lies within 2^-17 of a half-integer, or the code falls outside [0, 15], the lane
// recomputes its group from the IEEE division, so every code equals
// clamp(rint(RN((y - zero) / scale)), 0, 15).  The fast quotient is monotone in y (a subtraction
// and a product by a positive constant, each rounded), so all of a group's codes lie in [0, 15]
// when those of its minimum and maximum do; the codes are then the low nibbles of the rint sums,
// gathered a byte at a time.  The scale itself, RN((max - min) / 15), is exact: Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990) of the product by RN(1/15) with the exact fma residual.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int BW = 8;     // warps per CTA
constexpr int TPW = 8;    // tokens per warp
constexpr float RINT_MAGIC = 12582912.0f;                 // 1.5 * 2^23
constexpr float FAST_Q_LIMIT = 0.5f - 7.62939453125e-6f;  // 0.5 - 2^-17
constexpr float FAST_Q8_LIMIT = 0.5f - 6.103515625e-5f;   // 0.5 - 2^-14
constexpr int NB = 16;                  // 8-position blocks per warp in the pipelined (bf16) kernel
constexpr int SLOT = 80;                // shared bytes per lane and stage: 64 B of inputs + 16 B of padding
constexpr int STAGE_BYTES = 32 * SLOT;  // one stage of one warp

// RN(a / D) for the odd constants D = 15 and 127: q0 = RN(a * c) with c = RN(1/D) is within an ulp
// of a / D, r = a - D * q0 is exact (one fma), and RN(q0 + r * c) is the correctly rounded quotient
// (Markstein's correction; checked for every fp32 mantissa, the result being scale-free in the
// normal range, by an exact integer model in the tests).  Below 2^-21 the quotient's fp16 image is
// 0 whichever way it rounds.  Infinity and NaN pass through as the IEEE division gives them.
template <int DIV>
__device__ __forceinline__ float div_const_rn(float a) {
  static_assert(DIV == 15 || DIV == 127, "only the two group divisors");
  const float c = DIV == 15 ? 0.0666666701436043f : 0.007874015718698502f;  // RN(1/15), RN(1/127)
  const float q0 = __fmul_rn(a, c);
  const float r = __fmaf_rn(-(float)DIV, q0, a);
  const float q = __fmaf_rn(r, c, q0);
  return fabsf(a) < INFINITY ? q : a;
}

// hardware reciprocal, within 1 ulp (the fast quotients' error bounds allow for it)
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// three-input IEEE min / max (sm_100+); like the two-input forms they are exact and ignore a NaN
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// three-input max that returns NaN when an input is NaN
__device__ __forceinline__ float max3nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bytes 0 of four words, in order
__device__ __forceinline__ uint32_t gather_low_bytes(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x4000u), 0x7610u);
}

// Everything after the loads for one lane: the window copy of the raw inputs, the rotation, the
// codes of the lane's group (channels 32G .. 32G + 31 of token `pos`) and their stores into the
// half-page `pg` at token index `tin`.  Warp-collective (V token pairs exchange halfwords); a lane
// without a token (`valid` false) works on zeros and stores nothing.
__device__ __forceinline__ void code_and_store(float (&x)[32], const AppendArgs& a, int G, int kv, int layer,
                                               int h, int b, uint8_t* pg, int tin, int pos, int p0, bool valid) {
  const int H = a.Hkv, T = a.T;
  // raw copy into the window ring for the last `window` tokens of this call
  if (valid && a.W > 0 && pos - p0 >= T - a.W) {
    float* ring = kv ? a.p.ringv : a.p.ringk;
    float4* dst = reinterpret_cast<float4*>(
        ring + ((((size_t)layer * a.max_batch + b) * H + h) * a.W + (size_t)(pos % a.W)) * D + 32 * G);
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
  }

  // ---- rotation y = c * H (s . x): sign flip (exact), butterfly stages h = 1 .. 64, multiply by c
  {
    const float4* sg = reinterpret_cast<const float4*>(a.p.signs + 32 * G);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 s = sg[c];
      mul2(x[4 * c], x[4 * c + 1], s.x, s.y);
      mul2(x[4 * c + 2], x[4 * c + 3], s.z, s.w);
    }
  }
  // stage h = 1 pairs neighbours (scalar); stages h = 2 .. 16 pair (j, j+1) with (j+h, j+h+1)
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float u = x[j], v = x[j + 1];
    x[j] = __fadd_rn(u, v);
    x[j + 1] = __fsub_rn(u, v);
  }
#pragma unroll
  for (int hs = 2; hs < 32; hs <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      if (j & hs) continue;
      bfly2(x[j], x[j + 1], x[j + hs], x[j + hs + 1]);
    }
  }
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {  // h = 32 m: partner lane G ^ m holds the other channel
    const float sg = (G & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      fma2(x[j], x[j + 1], sg, sg, __shfl_xor_sync(FULL, x[j], m), __shfl_xor_sync(FULL, x[j + 1], m));
  }
#pragma unroll
  for (int j = 0; j < 32; j += 2) mul2(x[j], x[j + 1], C_WHT, C_WHT);
  if (a.sinkhorn) {
    const __half2* sg = reinterpret_cast<const __half2*>((kv ? a.p.sigv : a.p.sigk) + ((size_t)layer * H + h) * D + 32 * G);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float2 s = __half22float2(sg[j]);
      x[2 * j] = __fdiv_rn(x[2 * j], s.x);
      x[2 * j + 1] = __fdiv_rn(x[2 * j + 1], s.y);
    }
  }

  if (kv == 0 && a.k_format == KVQ_Q8G32) {
    // ---- Q8G32 key for the lane's group: d = fp16(max |y| / 127), codes clamp(rint(y / d), -127,
    // 127) against the stored d (0 when d == 0), stored as u = c + 128.  The quotient is formed as
    // y * rcp(d), within 3.1e-5 of the IEEE quotient for |y / d| <= 127.5; where it lies within
    // 2^-14 of a half-integer, or the quotient of max |y| (the largest in magnitude) reaches 127.5,
    // the lane redoes its group with the IEEE division.
    float am4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float* v = x + 8 * k;
      am4[k] = fmaxf(max3f(max3f(max3f(fabsf(v[0]), fabsf(v[1]), fabsf(v[2])), fabsf(v[3]), fabsf(v[4])),
                           fabsf(v[5]), fabsf(v[6])), fabsf(v[7]));
    }
    const float amax = fmaxf(max3f(am4[0], am4[1], am4[2]), am4[3]);
    const __half d16 = __float2half_rn(div_const_rn<127>(amax));
    const float d = __half2float(d16);
    uint32_t u8[8];  // byte-packed codes: u8[j] holds local channels 4j .. 4j+3
    if (d > 0.0f) {
      const float inv = rcp_approx(d);
      float dmax8 = 0.f;  // NaN if a quotient is
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t tb[4];
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          float q0 = x[4 * j + e], q1 = x[4 * j + e + 1];
          mul2(q0, q1, inv, inv);
          float t0 = q0, t1 = q1;
          add2(t0, t1, RINT_MAGIC, RINT_MAGIC);
          float n0 = RINT_MAGIC, n1 = RINT_MAGIC;
          sub2(n0, n1, t0, t1);
          add2(q0, q1, n0, n1);
          dmax8 = max3nan(dmax8, fabsf(q0), fabsf(q1));
          tb[e] = __float_as_uint(t0);
          tb[e + 1] = __float_as_uint(t1);
        }
        // the low byte of t's bits is its code c in two's complement; bit 7 flipped gives c + 128
        u8[j] = gather_low_bytes(tb[0], tb[1], tb[2], tb[3]) ^ 0x80808080u;
      }
      // |quotient| <= that of max |y|; codes in -127 .. 127 need it below 127.5
      const float qmax = __fmul_rn(amax, inv);
      if ((!(dmax8 <= FAST_Q8_LIMIT) || !(qmax < 127.5f)) && valid) {
        // rare: the group's codes from the IEEE quotient
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t word = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = min(max(__float2int_rn(__fdiv_rn(x[4 * j + e], d)), -127), 127);
            word |= (uint32_t)(c + 128) << (8 * e);
          }
          u8[j] = word;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) u8[j] = 0x80808080u;
    }
    if (valid) {
      // k-step kk = 2G + s (s = 0, 1) covers local channels 16 s .. 16 s + 15; word (i, kk) = local
      // channels 16 s + 2i, +1, +8, +9: bytes of u8[4 s + (i >> 1)] and u8[4 s + 2 + (i >> 1)]
      uint8_t* rec = pg + (size_t)tin * 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t wd[2];
#pragma unroll
        for (int sdx = 0; sdx < 2; ++sdx) {
          const uint32_t lo = u8[4 * sdx + (i >> 1)], hi = u8[4 * sdx + 2 + (i >> 1)];
          wd[sdx] = __byte_perm(lo, hi, (i & 1) ? 0x7632u : 0x5410u);
        }
        const int m = 2 * i + (G >> 1);
        *reinterpret_cast<uint2*>(rec + 16 * (m ^ (tin & 1)) + 8 * (G & 1)) = make_uint2(wd[0], wd[1]);
      }
      reinterpret_cast<__half*>(pg + a.L.off_kmeta + (size_t)tin * 8)[G] = d16;
    }
    return;
  }

  // ---- Q4G32 for the lane's group: exact min/max, fp16 scale (max-min)/15 and zero min, codes
  float mn4[4], mx4[4];  // min and max are exact: any order gives the same result
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float* v = x + 8 * k;
    mn4[k] = fminf(min3f(min3f(min3f(v[0], v[1], v[2]), v[3], v[4]), v[5], v[6]), v[7]);
    mx4[k] = fmaxf(max3f(max3f(max3f(v[0], v[1], v[2]), v[3], v[4]), v[5], v[6]), v[7]);
  }
  const float mn = fminf(min3f(mn4[0], mn4[1], mn4[2]), mn4[3]);
  const float mx = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]);
  const __half s16 = __float2half_rn(div_const_rn<15>(__fsub_rn(mx, mn)));
  const __half z16 = __float2half_rn(mn);
  const uint32_t meta = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
  const float s = __half2float(s16), z = __half2float(z16);
  const float inv = rcp_approx(s);
  uint32_t w[4];      // nibble m of w[i] = code of channel 32G + 8i + m
  float dmax = 0.f;   // largest distance of a quotient from its rounded integer (NaN if a quotient is)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t pb[4];   // byte 0 of pb[j] = codes of channels 8i + 2j (low nibble) and 8i + 2j + 1
#pragma unroll
    for (int m = 0; m < 8; m += 2) {
      // qt = (y - z) * inv, t = qt + 1.5 * 2^23, -r = 1.5 * 2^23 - t, d = qt - r: pairwise, all but
      // the first two exact
      float q0 = x[8 * i + m], q1 = x[8 * i + m + 1];
      sub2(q0, q1, z, z);
      mul2(q0, q1, inv, inv);
      float t0 = q0, t1 = q1;
      add2(t0, t1, RINT_MAGIC, RINT_MAGIC);
      float n0 = RINT_MAGIC, n1 = RINT_MAGIC;
      sub2(n0, n1, t0, t1);
      add2(q0, q1, n0, n1);
      dmax = max3nan(dmax, fabsf(q0), fabsf(q1));
      // the low byte of t's bits is its code while the code is in 0 .. 15
      pb[m >> 1] = __float_as_uint(t0) + (__float_as_uint(t1) << 4);
    }
    w[i] = gather_low_bytes(pb[0], pb[1], pb[2], pb[3]);
  }
  // every quotient lies between those of mn and mx; codes in 0 .. 15 need them in [-0.5, 15.5)
  const float qlo = __fmul_rn(__fsub_rn(mn, z), inv), qhi = __fmul_rn(__fsub_rn(mx, z), inv);
  const bool redo = !(dmax <= FAST_Q_LIMIT) || !(qlo >= -0.5f) || !(qhi < 15.5f);
  if (!(s > 0.0f)) {
    w[0] = w[1] = w[2] = w[3] = 0u;
  } else if (redo && valid) {
    // rare: the group's codes from the IEEE quotient
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int c = min(max(__float2int_rn(__fdiv_rn(__fsub_rn(x[8 * i + m], z), s)), 0), 15);
        word |= (uint32_t)c << (4 * m);
      }
      w[i] = word;
    }
  }

  if (kv == 0) {
    if (valid) {
      // K record: 32-bit word (i, G) at byte 16i + 4G holds channels 32G + 8i .. +7 = w[i];
      // K meta: fp16 scale[G] at 2G, zero[G] at 8 + 2G
      uint32_t* rec = reinterpret_cast<uint32_t*>(pg + (size_t)tin * 64);
#pragma unroll
      for (int i = 0; i < 4; ++i) rec[4 * i + G] = w[i];
      uint16_t* km = reinterpret_cast<uint16_t*>(pg + a.L.off_kmeta + (size_t)tin * 16);
      km[G] = (uint16_t)(meta & 0xffffu);
      km[4 + G] = (uint16_t)(meta >> 16);
    }
    return;
  }
  // ---- V: tokens 2p, 2p+1 share 128 bytes; row R of group G sits at 16 * ((R + 2 * (p & 3)) & 7) + 4G
  // as bytes [t0 byte0, t1 byte0, t0 byte1, t1 byte1] of the halfword hw(R) = channels 32G + 4R .. +3
  // = half (R & 1) of w[R / 2].  The even token stores rows 0-3, the odd one rows 4-7, each with
  // its partner's halfwords (lane ^ 4) for those rows.
  const bool odd = tin & 1;
  // every lane takes part in the shuffle (a short-circuited one would leave lanes of the mask out)
  const int partner_valid = __shfl_xor_sync(FULL, valid ? 1 : 0, 4);
  const bool paired = valid && partner_valid != 0;
  const uint32_t pa = __shfl_xor_sync(FULL, odd ? w[0] : w[2], 4);
  const uint32_t pb = __shfl_xor_sync(FULL, odd ? w[1] : w[3], 4);
  uint8_t* vmain = pg + a.L.off_vmain;
  const int pp = tin >> 1;
  if (paired) {
    const uint32_t sel0 = odd ? 0x1504u : 0x5140u, sel1 = odd ? 0x3726u : 0x7362u;
    const uint32_t m0 = odd ? w[2] : w[0], m1 = odd ? w[3] : w[1];
    const int R0 = odd ? 4 : 0;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const uint32_t mine = (rr >> 1) ? m1 : m0, part = (rr >> 1) ? pb : pa;
      *reinterpret_cast<uint32_t*>(vmain + (size_t)pp * 128 + 16 * ((R0 + rr + 2 * (pp & 3)) & 7) + 4 * G) =
          __byte_perm(mine, part, (rr & 1) ? sel1 : sel0);
    }
  } else if (valid) {
#pragma unroll
    for (int R = 0; R < 8; ++R) {
      const uint32_t hw = (w[R >> 1] >> (16 * (R & 1))) & 0xffffu;
      uint8_t* dst = vmain + (size_t)pp * 128 + 16 * ((R + 2 * (pp & 3)) & 7) + 4 * G + (tin & 1);
      dst[0] = (uint8_t)(hw & 0xffu);
      dst[2] = (uint8_t)(hw >> 8);
    }
  }
  if (valid) {
    // V meta: group-major scale[4][32] then zero[4][32]
    uint16_t* vm = reinterpret_cast<uint16_t*>(pg + a.L.off_vmeta);
    vm[G * HALF + tin] = (uint16_t)(meta & 0xffffu);
    vm[4 * HALF + G * HALF + tin] = (uint16_t)(meta >> 16);
  }
}

// One 8-position block per warp, inputs loaded straight from global memory (fp32 inputs).
__device__ __forceinline__ void append_bulk_body(const AppendArgs& a) {
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int G = lane & 3, tv = lane >> 2;  // group (channels 32G ..) and token of this lane
  // a dependent decode launch may start its set-up now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  const int H = a.Hkv, T = a.T;
  // grid: x = 8-position blocks of a sequence's call (8 per CTA), y = (layer, kv-head, K|V), z = sequence
  const int bi = blockIdx.x * BW + wl;
  if (bi >= T / TPW + 2) return;  // 8-position blocks one sequence's call can touch
  const int kv = a.kv_lo + (a.kv_n == 2 ? (int)(blockIdx.y & 1) : 0);
  const int hl = a.kv_n == 2 ? (int)(blockIdx.y >> 1) : (int)blockIdx.y;
  const int h = hl % H, ll = hl / H;
  const int b = blockIdx.z;
  const int layer = a.layer0 + ll;

  const int p0 = a.pos[b];
  if (p0 < 0) return;  // sequence not part of this append
  if ((long long)p0 + T > a.max_seq_len) {
    if (lane == 0 && bi == 0 && kv == a.kv_lo && h == 0) atomicOr(a.p.status, KVQ_DEV_POS_RANGE);
    return;
  }
  const int blk0 = p0 / TPW + bi;
  const int lo_pos = max(p0, blk0 * TPW), hi_pos = min(p0 + T, blk0 * TPW + TPW);
  if (lo_pos >= hi_pos) return;
  const int hp = blk0 * TPW / HALF;  // half-page (all 8 positions share it)
  const int phys = a.block_table[(size_t)b * a.L.max_pages_per_seq + hp / 2];
  if (phys < 0 || phys >= a.L.n_pages) {
    if (lane == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
    return;
  }
  uint8_t* pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
                (size_t)(hp & 1) * a.L.half_bytes;

  const int pos = blk0 * TPW + tv;
  const bool valid = pos >= lo_pos && pos < hi_pos;
  const int tin = pos % HALF;  // token index within the half-page

  // ---- the lane's 32 input values (channels 32G ..); a lane without a token works on zeros
  float x[32];
  {
    const size_t row = ((((size_t)ll * a.batch + b) * H + h) * T + (size_t)(valid ? pos - p0 : 0)) * D + 32 * G;
    const void* src = kv ? a.v : a.k;
    if (a.in_bf16) {
      const uint4* g = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + row);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 u = valid ? __ldcs(g + c) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[8 * c + 2 * e] = __uint_as_float(uu[e] << 16);
          x[8 * c + 2 * e + 1] = __uint_as_float(uu[e] & 0xffff0000u);
        }
      }
    } else {
      const float4* g = reinterpret_cast<const float4*>(static_cast<const float*>(src) + row);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float4 f = valid ? __ldcs(g + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[4 * c] = f.x;
        x[4 * c + 1] = f.y;
        x[4 * c + 2] = f.z;
        x[4 * c + 3] = f.w;
      }
    }
  }
  code_and_store(x, a, G, kv, layer, h, b, pg, tin, pos, p0, valid);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// bf16 inputs: NB consecutive 8-position blocks per warp, two shared-memory stages per warp.  The
// block's 2 KB of inputs (8 rows of 256 B) are copied as four 512-byte runs, lane l taking bytes
// 16l .. 16l + 15 of each: run c holds tokens 2c + (l >> 4), group (l >> 2) & 3, 16-byte chunk l & 3,
// which lands in the slot of the lane that codes it (lane 4 * token + group, 80 bytes apart so that
// the 16-byte reads of eight neighbouring lanes hit distinct banks).  Rows of positions outside the
// call are zero-filled, not read.  Waits are the copy unit's own (cp.async.wait_group, then a warp
// barrier, since a lane reads what other lanes copied), no spin.
__device__ __forceinline__ void append_bulk_bf16_body(const AppendArgs& a, uint8_t (*stage)[2][STAGE_BYTES]) {
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int G = lane & 3, tv = lane >> 2;  // group (channels 32G ..) and token of this lane
  // a dependent decode launch may start its set-up now; it waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;");
  const int H = a.Hkv, T = a.T;
  // grid: x = runs of NB 8-position blocks (BW runs per CTA), y = (layer, kv-head, K|V), z = sequence
  const int kv = a.kv_lo + (a.kv_n == 2 ? (int)(blockIdx.y & 1) : 0);
  const int hl = a.kv_n == 2 ? (int)(blockIdx.y >> 1) : (int)blockIdx.y;
  const int h = hl % H, ll = hl / H;
  const int b = blockIdx.z;
  const int layer = a.layer0 + ll;

  const int p0 = a.pos[b];
  if (p0 < 0) return;  // sequence not part of this append
  if ((long long)p0 + T > a.max_seq_len) {
    if (lane == 0 && blockIdx.x == 0 && wl == 0 && kv == a.kv_lo && h == 0) atomicOr(a.p.status, KVQ_DEV_POS_RANGE);
    return;
  }
  const int blk_first = p0 / TPW;                                  // first 8-position block of the call
  const int n_blk = (p0 + T + TPW - 1) / TPW - blk_first;          // blocks the call touches
  const int bi0 = (blockIdx.x * BW + wl) * NB;
  const int nb = min(NB, n_blk - bi0);
  if (nb <= 0) return;

  const char* src = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(kv ? a.v : a.k) +
                                                  (((size_t)ll * a.batch + b) * H + h) * (size_t)T * D);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(&stage[wl][0][0]);
  // copier side of lane l for run c: token 2c + (l >> 4), destination slot of its coder
  const int cp_tok = lane >> 4;
  const uint32_t cp_dst = sbase + (uint32_t)((4 * cp_tok + ((lane >> 2) & 3)) * SLOT + 16 * (lane & 3));
  auto issue = [&](int k) {  // copies of block bi0 + k into stage k & 1
    const int base_pos = (blk_first + bi0 + k) * TPW;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int pos = base_pos + 2 * c + cp_tok;
      const bool in = pos >= p0 && pos < p0 + T;
      const char* g = src + (size_t)(in ? pos - p0 : 0) * (D * 2) + 16 * (lane & 15);
      cp_async16(cp_dst + (uint32_t)((k & 1) * STAGE_BYTES + c * 8 * SLOT), g, in ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  issue(0);
  for (int k = 0; k < nb; ++k) {
    __syncwarp();  // every lane is done reading the stage that block k + 1 overwrites
    if (k + 1 < nb) issue(k + 1);
    else asm volatile("cp.async.commit_group;" ::: "memory");  // an empty group keeps the count
    asm volatile("cp.async.wait_group 1;" ::: "memory");       // this lane's copies of block k have landed
    __syncwarp();  // and so have the other lanes' (each lane reads rows that other lanes copied)

    const int blk0 = blk_first + bi0 + k;
    const int hp = blk0 * TPW / HALF;  // half-page (all 8 positions share it)
    const int phys = a.block_table[(size_t)b * a.L.max_pages_per_seq + hp / 2];
    if (phys < 0 || phys >= a.L.n_pages) {
      if (lane == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
      continue;
    }
    uint8_t* pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
                  (size_t)(hp & 1) * a.L.half_bytes;
    const int pos = blk0 * TPW + tv;
    const bool valid = pos >= p0 && pos < p0 + T;
    const int tin = pos % HALF;  // token index within the half-page

    float x[32];
    const uint4* sp = reinterpret_cast<const uint4*>(&stage[wl][k & 1][lane * SLOT]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 u = sp[c];
      const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[8 * c + 2 * e] = __uint_as_float(uu[e] << 16);
        x[8 * c + 2 * e + 1] = __uint_as_float(uu[e] & 0xffff0000u);
      }
    }
    code_and_store(x, a, G, kv, layer, h, b, pg, tin, pos, p0, valid);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// A TurboQuant-key append launches this kernel for the values (AFTER_KEYS) as a programmatic
// dependent of the keys kernel (the two write disjoint bytes, so they may overlap); every thread then
// waits for the keys grid before exiting, so that whatever waits for this grid (the decode) also
// waits for the keys.
template <bool AFTER_KEYS>
__global__ void __launch_bounds__(BW * 32, 4) append_bulk_kernel(const __grid_constant__ AppendArgs a) {
  append_bulk_body(a);
  if (AFTER_KEYS) asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <bool AFTER_KEYS>
__global__ void __launch_bounds__(BW * 32, 4) append_bulk_bf16_kernel(const __grid_constant__ AppendArgs a) {
  __shared__ __align__(16) uint8_t stage[BW][2][STAGE_BYTES];
  append_bulk_bf16_body(a, stage);
  if (AFTER_KEYS) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_append_bulk(const AppendArgs& a, cudaStream_t s, bool after_keys) {
  const long long per_cta = a.in_bf16 ? (long long)BW * NB : BW;  // 8-position blocks per CTA
  const long long gx = ((long long)a.T / TPW + 2 + per_cta - 1) / per_cta;
  const long long gy = (long long)a.n_layers_call * a.Hkv * a.kv_n;
  if (gx <= 0 || gy <= 0 || a.batch <= 0) return cudaSuccess;
  if (gx > 0x7fffffffLL || gy > 65535 || a.batch > 65535) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)gx, (unsigned)gy, (unsigned)a.batch);
  cfg.blockDim = dim3(BW * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_keys ? 1 : 0;
  if (a.in_bf16) {
    return after_keys ? cudaLaunchKernelEx(&cfg, append_bulk_bf16_kernel<true>, a)
                      : cudaLaunchKernelEx(&cfg, append_bulk_bf16_kernel<false>, a);
  }
  return after_keys ? cudaLaunchKernelEx(&cfg, append_bulk_kernel<true>, a)
                    : cudaLaunchKernelEx(&cfg, append_bulk_kernel<false>, a);
}

}  // namespace kvq
