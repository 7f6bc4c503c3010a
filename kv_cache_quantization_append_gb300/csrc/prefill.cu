// Chunked prefill: append a chunk of new tokens and compute the attention of their queries over the
// compressed cache.
//
// What it computes ([QC] "Beyond RAG: load the whole document on your laptop", v3.2 batched-prefill
// note: a batched prefill writes exactly what per-token steps write; read the same way for its
// attention): query t of sequence b attends to positions [0, pos[b] + t] exactly as its own
// single-token decode step would -- the newest `window` of those positions through their raw
// values, the rest through their quantised records ([QC] "how it works"; [KV] TLDR; [TQ] "key
// idea" row for TQ3 keys), one softmax with scale 1/sqrt(128).
//
// One call: (1) copy the window ring of the call's units to scratch -- the chunk's append
// overwrites ring slots whose old positions early queries of the chunk still read raw; (2) the
// append kernels write the chunk (pages and ring); (3) the attention kernel below.
//
// Attention kernel (one CTA = 64 (query, head) rows of one (layer, sequence, kv-head) unit, four
// warps of 16 rows):
//  * Every key tile -- 32 positions, either one quantised half-page or 32 raw window positions --
//    is written to shared memory as fp16 hi/lo pairs of its value in the quantised keys' space:
//    the rotated, balanced vector for Q4G32 / Q8G32 keys (raw keys and values are rotated and
//    divided by sigma on the fly), and for TQ3 keys the 256-wide vector
//    [n c^, n sqrt(pi/2)/128 gamma (2b - 1)] that dots with [q~, S q~] to the QJL estimate (raw keys
//    padded with zeros).  So one rotated query tile and one output accumulator serve both parts.
//  * Logits and P.V are mma.sync products of the hi/lo pairs (hi*hi + hi*lo + lo*hi, about 22
//    significant bits: attention outputs are small against the values they average, so fp16 alone
//    would not meet the 2e-3 bar), with an online softmax in base 2 in registers; the weights go
//    from the logit accumulators straight into the P.V operand registers.
//  * Quantised and raw tiles cover disjoint (row, position) pairs through their masks: position j
//    is quantised for query P when j <= P - window, raw when P - window < j <= P.
//  * The output row is unfolded (sigma_v) and unrotated at the end.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int ROWS = 64;     // (query, head) rows per CTA
constexpr int NT = 32;       // key positions per tile
constexpr int NWARP = 4;
constexpr int THREADS = NWARP * 32;
constexpr int VS = NT + 8;   // row stride (halves) of the transposed value tile: conflict-free ldmatrix

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp16 hi/lo split of v: hi = fp16(v), lo = fp16(v - hi)
__device__ __forceinline__ void split(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}
__device__ __forceinline__ uint32_t pack2(__half a, __half b) {
  return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

template <int KF>
struct Tile {
  static constexpr bool TQ = KF == KVQ_TQ3_QJL;
  static constexpr int KD = TQ ? 256 : 128;  // width of the key space the logits are taken in
  static constexpr int QS = KD + 8;          // row stride (halves) of the query and key tiles
  static constexpr size_t Q_HALVES = (size_t)2 * ROWS * QS;
  static constexpr size_t K_HALVES = (size_t)2 * NT * QS;
  static constexpr size_t V_HALVES = (size_t)2 * D * VS;
  static constexpr size_t BYTES = (Q_HALVES + K_HALVES + V_HALVES) * 2;
  static_assert((K_HALVES + V_HALVES) * 2 >= (size_t)ROWS * D * 4, "output staging must fit");
};

// Copy the window ring of every (layer, sequence < batch, kv-head) of the call to scratch.
__global__ void snapshot_kernel(const __grid_constant__ PrefillArgs a) {
  const size_t per_layer = (size_t)a.batch * a.Hkv * a.W * D / 4;  // float4s of one layer's sequences
  const size_t n = per_layer * a.n_layers_call;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t ll = i / per_layer, r = i - ll * per_layer;
    const size_t src = ((size_t)(a.layer0 + ll) * a.max_batch * a.Hkv * a.W * D) / 4 + r;
    reinterpret_cast<float4*>(a.snap_k)[i] = reinterpret_cast<const float4*>(a.p.ringk)[src];
    reinterpret_cast<float4*>(a.snap_v)[i] = reinterpret_cast<const float4*>(a.p.ringv)[src];
  }
}

template <int KF>
__global__ void __launch_bounds__(THREADS) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  using TL = Tile<KF>;
  constexpr int KD = TL::KD, QS = TL::QS;
  extern __shared__ __align__(16) uint8_t smem[];
  __half* sQ = reinterpret_cast<__half*>(smem);  // [hi, lo][ROWS][QS]
  __half* sK = sQ + TL::Q_HALVES;                // [hi, lo][NT][QS]
  __half* sV = sK + TL::K_HALVES;                // [hi, lo][D][VS]: values transposed (channel, position)
  float* sO = reinterpret_cast<float*>(sK);      // [ROWS][D]: output staging at the end

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.Hkv, g = a.g, B = a.batch, T = a.T, W = a.W, Hq = a.Hkv * a.g;
  const int h = blockIdx.y, b = (int)(blockIdx.z % B), ll = (int)(blockIdx.z / B);
  const int layer = a.layer0 + ll;
  const int qpt = ROWS / g;  // queries per CTA
  const int t0 = blockIdx.x * qpt;
  if (t0 >= T) return;
  const int nq = min(qpt, T - t0);
  const int nrows = nq * g;
  const int p0 = a.pos[b];
  const bool in_range = p0 >= 0 && (long long)p0 + T <= (long long)a.max_seq_len;
  auto out_row = [&](int row) -> float* {
    const int tl = row / g, hh = row % g;
    return a.out + ((((size_t)ll * B + b) * Hq + (size_t)h * g + hh) * T + t0 + tl) * D;
  };
  if (!in_range) {
    // sequence not part of this call (pos < 0), or flagged by the append (past capacity): zeros
    for (int idx = tid; idx < nrows * (D / 4); idx += THREADS)
      reinterpret_cast<float4*>(out_row(idx / (D / 4)))[idx % (D / 4)] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }

  // ---- query tile: q~ = c H (s . q) [. sigma_k] in base-2 logit units, as fp16 hi/lo (TQ3: also S q~)
  {
    const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
    float4 sk = make_float4(1.f, 1.f, 1.f, 1.f);
    if (a.sinkhorn) {
      const __half* sig = a.p.sigk + ((size_t)layer * H + h) * D + 4 * lane;
      sk = make_float4(__half2float(sig[0]), __half2float(sig[1]), __half2float(sig[2]), __half2float(sig[3]));
    }
    float* qtmp = reinterpret_cast<float*>(sK) + warp * D;  // this warp's rotated query (TQ3 projection)
    for (int rr = 0; rr < 16; ++rr) {
      const int row = 16 * warp + rr;
      const int tl = row / g, hh = row % g;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < nrows)
        x = load4_in(a.q, ((((size_t)ll * B + b) * Hq + (size_t)h * g + hh) * T + t0 + tl) * D + 4 * lane, a.in_bf16);
      float y0 = x.x * sg.x, y1 = x.y * sg.y, y2 = x.z * sg.z, y3 = x.w * sg.w;
      hadamard_warp(y0, y1, y2, y3, lane);
      const float sc = C_WHT * LOGIT_SCALE;
      const float yv[4] = {y0 * sc * sk.x, y1 * sc * sk.y, y2 * sc * sk.z, y3 * sc * sk.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __half hi, lo;
        split(yv[e], hi, lo);
        sQ[(size_t)row * QS + 4 * lane + e] = hi;
        sQ[TL::Q_HALVES / 2 + (size_t)row * QS + 4 * lane + e] = lo;
      }
      if (TL::TQ) {
        *reinterpret_cast<float4*>(qtmp + 4 * lane) = make_float4(yv[0], yv[1], yv[2], yv[3]);
        __syncwarp();
        // projections 4 lane .. +3 of S q~ (the transposed projection is stored row j = column j of S)
        const float4* stp = reinterpret_cast<const float4*>(a.p.qjl_t) + lane;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int j = 0; j < D; ++j) {
          const float qj = qtmp[j];
          const float4 s4 = stp[j * (D / 4)];
          acc.x += s4.x * qj;
          acc.y += s4.y * qj;
          acc.z += s4.z * qj;
          acc.w += s4.w * qj;
        }
        const float av[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half hi, lo;
          split(av[e], hi, lo);
          sQ[(size_t)row * QS + D + 4 * lane + e] = hi;
          sQ[TL::Q_HALVES / 2 + (size_t)row * QS + D + 4 * lane + e] = lo;
        }
        __syncwarp();
      }
    }
  }

  // positions of this CTA's queries: P = p0 + t0 + tl; the quantised positions any of them reads are
  // [0, qend), the raw ones [rlo, Pmax]
  const int Pmin = p0 + t0, Pmax = p0 + t0 + nq - 1;
  const int qend = W > 0 ? max(0, Pmax - W + 1) : Pmax + 1;
  const int rlo = W > 0 ? max(0, Pmin - W + 1) : 0;
  const int nqt = (qend + NT - 1) / NT;
  const int rbeg = rlo & ~(NT - 1);
  const int nrt = W > 0 ? (Pmax - rbeg) / NT + 1 : 0;

  // this lane's two rows (r, r + 8 of the warp's 16) and their query positions (-1: no query)
  const int r = lane >> 2, i4 = lane & 3;
  int Prow[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int row = 16 * warp + r + 8 * k;
    Prow[k] = row < nrows ? p0 + t0 + row / g : -1;
  }
  float O[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const __half* sig_v = a.p.sigv + ((size_t)layer * H + h) * D;
  const __half* sig_k = a.p.sigk + ((size_t)layer * H + h) * D;

  for (int it = 0; it < nqt + nrt; ++it) {
    const bool raw = it >= nqt;
    const int j0 = raw ? rbeg + (it - nqt) * NT : it * NT;
    __syncthreads();  // the previous tile's shared reads are done (and the query tile is written)
    bool bad = false;
    if (!raw) {
      // ---- quantised half-page: positions j0 .. j0 + 31 (those at or past qend are zeroed)
      const int hp = j0 / HALF;
      const int page = b * a.max_pages_per_seq + (hp >> 1);
      const int phys = a.block_table[page];
      bad = phys < 0 || phys >= a.L.n_pages;
      const uint8_t* pg = bad ? nullptr
                              : a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes +
                                    (size_t)(hp & 1) * a.L.half_bytes;
      if (bad && tid == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
      // keys: one (position, part) task per thread
      {
        const int t = tid >> 2, part = tid & 3;
        const bool ok = !bad && j0 + t < qend;
        __half* dh = sK + (size_t)t * QS;
        __half* dl = sK + TL::K_HALVES / 2 + (size_t)t * QS;
        if (KF == KVQ_Q4G32) {
          // group G = part: word (i, G) at 16i + 4G holds channels 32G + 8i .. +7 (nibble pairs)
          const int G = part;
          float s = 0.f, z = 0.f;
          uint32_t wd[4] = {0u, 0u, 0u, 0u};
          if (ok) {
            const __half* km = reinterpret_cast<const __half*>(pg + a.L.off_kmeta + (size_t)t * 16);
            s = __half2float(km[G]);
            z = __half2float(km[4 + G]);
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) wd[ii] = *reinterpret_cast<const uint32_t*>(pg + (size_t)t * 64 + 16 * ii + 4 * G);
          }
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int ch = 32 * G + 8 * ii + m;
              const float v = ok ? z + s * (float)((wd[ii] >> (4 * m)) & 15u) : 0.f;
              __half hi, lo;
              split(v, hi, lo);
              dh[ch] = hi;
              dl[ch] = lo;
            }
        } else if (KF == KVQ_Q8G32) {
          // chunks m = 2 part + hh (hh = 0, 1) of the token: 16 stored bytes u = c + 128 each
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int m = 2 * part + hh, i = m >> 1, h2 = m & 1;
            uint4 c4 = make_uint4(0u, 0u, 0u, 0u);
            float dsc[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
              c4 = *reinterpret_cast<const uint4*>(pg + (size_t)t * 128 + 16 * (m ^ (t & 1)));
              const __half* km = reinterpret_cast<const __half*>(pg + a.L.off_kmeta + (size_t)t * 8);
#pragma unroll
              for (int G = 0; G < 4; ++G) dsc[G] = __half2float(km[G]);
            }
            const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
            for (int w = 0; w < 4; ++w)
#pragma unroll
              for (int bb = 0; bb < 4; ++bb) {
                const int ch = 16 * (4 * h2 + w) + 2 * i + (bb & 1) + 8 * (bb >> 1);
                const float v = ok ? dsc[ch >> 5] * (float)((int)((cw[w] >> (8 * bb)) & 0xffu) - 128) : 0.f;
                __half hi, lo;
                split(v, hi, lo);
                dh[ch] = hi;
                dl[ch] = lo;
              }
          }
        } else {
          // TQ3: bytes 16 part .. +15: codes of channels 2j, 2j+1 and signs of projections 2j, 2j+1
          uint4 c4 = make_uint4(0u, 0u, 0u, 0u);
          float nn = 0.f, wq = 0.f;
          if (ok) {
            c4 = *reinterpret_cast<const uint4*>(pg + (size_t)t * 64 + 16 * part);
            const __half* km = reinterpret_cast<const __half*>(pg + a.L.off_kmeta);
            nn = __half2float(km[t]);
            wq = nn * QJL_CONST * __half2float(km[HALF + t]);
          }
          const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
          for (int jb = 0; jb < 16; ++jb) {
            const uint32_t byte = (cw[jb >> 2] >> (8 * (jb & 3))) & 0xffu;
            const int j = 16 * part + jb;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float cv = __half2float(a.p.cb->cent[(byte >> (3 * e)) & 7u]);
              const float kv = ok ? nn * cv : 0.f;
              const float sv = ok ? (((byte >> (6 + e)) & 1u) ? wq : -wq) : 0.f;
              __half hi, lo;
              split(kv, hi, lo);
              dh[2 * j + e] = hi;
              dl[2 * j + e] = lo;
              split(sv, hi, lo);
              dh[D + 2 * j + e] = hi;
              dl[D + 2 * j + e] = lo;
            }
          }
        }
      }
      // values (Q4G32): tasks (token pair p, row rr, group G); bytes [t0 b0, t1 b0, t0 b1, t1 b1]
      for (int task = tid; task < 16 * 8 * 4; task += THREADS) {
        const int p = task >> 5, rr = (task >> 2) & 7, G = task & 3;
        uint32_t w4 = 0u;
        float sc[2] = {0.f, 0.f}, zr[2] = {0.f, 0.f};
        bool okt[2];
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) okt[s2] = !bad && j0 + 2 * p + s2 < qend;
        if (okt[0] || okt[1]) {
          w4 = *reinterpret_cast<const uint32_t*>(pg + a.L.off_vmain + (size_t)p * 128 + 16 * ((rr + 2 * (p & 3)) & 7) +
                                                  4 * G);
          const __half* vm = reinterpret_cast<const __half*>(pg + a.L.off_vmeta);
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            sc[s2] = __half2float(vm[G * HALF + 2 * p + s2]);
            zr[s2] = __half2float(vm[4 * HALF + G * HALF + 2 * p + s2]);
          }
        }
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // channel 32G + 4rr + e: byte (e >> 1) of token s2 = byte index 2 (e >> 1) + s2, nibble e & 1
            const uint32_t byte = (w4 >> (8 * (2 * (e >> 1) + s2))) & 0xffu;
            const uint32_t c = (e & 1) ? (byte >> 4) : (byte & 15u);
            const float v = okt[s2] ? zr[s2] + sc[s2] * (float)c : 0.f;
            __half hi, lo;
            split(v, hi, lo);
            const int ch = 32 * G + 4 * rr + e, t = 2 * p + s2;
            sV[(size_t)ch * VS + t] = hi;
            sV[TL::V_HALVES / 2 + (size_t)ch * VS + t] = lo;
          }
      }
    } else {
      // ---- raw window positions j0 .. j0 + 31 in the quantised space: rotated, divided by sigma
      // (positions before the chunk from the ring copy, the chunk's own from its inputs); positions
      // no query of this CTA reads raw are zeroed
      const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
      for (int vec = warp; vec < 2 * NT; vec += NWARP) {
        const int kv = vec / NT, t = vec % NT, j = j0 + t;
        const bool ok = j >= rlo && j <= Pmax;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok) {
          if (j < p0) {
            const float* snap = kv ? a.snap_v : a.snap_k;
            x = *reinterpret_cast<const float4*>(snap + ((((size_t)ll * B + b) * H + h) * W + (j % W)) * D + 4 * lane);
          } else {
            x = load4_in(kv ? a.v : a.k, ((((size_t)ll * B + b) * H + h) * T + (j - p0)) * D + 4 * lane, a.in_bf16);
          }
        }
        float y0 = x.x * sg.x, y1 = x.y * sg.y, y2 = x.z * sg.z, y3 = x.w * sg.w;
        hadamard_warp(y0, y1, y2, y3, lane);
        float yv[4] = {y0 * C_WHT, y1 * C_WHT, y2 * C_WHT, y3 * C_WHT};
        if (a.sinkhorn) {
          const __half* sig = (kv ? sig_v : sig_k) + 4 * lane;
#pragma unroll
          for (int e = 0; e < 4; ++e) yv[e] = yv[e] / __half2float(sig[e]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half hi, lo;
          split(ok ? yv[e] : 0.f, hi, lo);
          const int ch = 4 * lane + e;
          if (kv == 0) {
            sK[(size_t)t * QS + ch] = hi;
            sK[TL::K_HALVES / 2 + (size_t)t * QS + ch] = lo;
            if (TL::TQ) {
              sK[(size_t)t * QS + D + ch] = __float2half_rn(0.f);
              sK[TL::K_HALVES / 2 + (size_t)t * QS + D + ch] = __float2half_rn(0.f);
            }
          } else {
            sV[(size_t)ch * VS + t] = hi;
            sV[TL::V_HALVES / 2 + (size_t)ch * VS + t] = lo;
          }
        }
      }
    }
    __syncthreads();

    // ---- logits of this warp's 16 rows against the tile's 32 positions (4 n-tiles of 8)
    float S[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
    {
      const uint32_t qa_hi = smem_u32(sQ + (size_t)(16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1)) * QS + 8 * (lane >> 4));
      const uint32_t qa_lo = qa_hi + (uint32_t)(TL::Q_HALVES / 2) * 2u;
      const uint32_t kb_hi = smem_u32(sK + (size_t)((lane & 7) + 8 * (lane >> 4)) * QS + 8 * ((lane >> 3) & 1));
      const uint32_t kb_lo = kb_hi + (uint32_t)(TL::K_HALVES / 2) * 2u;
#pragma unroll 4
      for (int ks = 0; ks < KD / 16; ++ks) {
        uint32_t ah[4], al[4];
        ldsm_x4(qa_hi + 32u * ks, ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(qa_lo + 32u * ks, al[0], al[1], al[2], al[3]);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t bh[4], bl[4];
          const uint32_t off = 32u * ks + (uint32_t)(16 * np * QS) * 2u;
          ldsm_x4(kb_hi + off, bh[0], bh[1], bh[2], bh[3]);
          ldsm_x4(kb_lo + off, bl[0], bl[1], bl[2], bl[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float(&acc)[4] = S[2 * np + e];
            mma16816(acc, ah[0], ah[1], ah[2], ah[3], bh[2 * e], bh[2 * e + 1]);
            mma16816(acc, ah[0], ah[1], ah[2], ah[3], bl[2 * e], bl[2 * e + 1]);
            mma16816(acc, al[0], al[1], al[2], al[3], bh[2 * e], bh[2 * e + 1]);
          }
        }
      }
    }

    // ---- masks: quantised j <= P - window (window 0: j <= P); raw P - window < j <= P
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int P = Prow[e >> 1];
        const int j = j0 + 8 * n + 2 * i4 + (e & 1);
        const bool valid = P >= 0 && !bad && (raw ? (j > P - W && j <= P) : (j <= (W > 0 ? P - W : P)));
        if (!valid) S[n][e] = -INFINITY;
      }

    // ---- online softmax (rows r and r + 8), base 2
    float alpha[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float mx = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n) mx = fmaxf(mx, fmaxf(S[n][2 * k], S[n][2 * k + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
      const float mnew = fmaxf(mrow[k], mx);
      alpha[k] = (mnew == -INFINITY) ? 1.f : ex2(mrow[k] - mnew);
      mrow[k] = mnew;
      lrow[k] *= alpha[k];
      const float mref = (mnew == -INFINITY) ? 0.f : mnew;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        S[n][2 * k] = ex2(S[n][2 * k] - mref);
        S[n][2 * k + 1] = ex2(S[n][2 * k + 1] - mref);
        lrow[k] += S[n][2 * k] + S[n][2 * k + 1];
      }
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      O[n][0] *= alpha[0];
      O[n][1] *= alpha[0];
      O[n][2] *= alpha[1];
      O[n][3] *= alpha[1];
    }

    // ---- P.V: the weights (fp16 hi/lo) straight from the logit accumulators into A operands
    {
      const uint32_t vb_hi = smem_u32(sV + (size_t)((lane & 7) + 8 * (lane >> 4)) * VS + 8 * ((lane >> 3) & 1));
      const uint32_t vb_lo = vb_hi + (uint32_t)(TL::V_HALVES / 2) * 2u;
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        uint32_t ph[4], pl[4];
        const float* s0 = S[2 * kt];
        const float* s1 = S[2 * kt + 1];
        const float pv[8] = {s0[0], s0[1], s0[2], s0[3], s1[0], s1[1], s1[2], s1[3]};
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          __half h0, l0, h1, l1;
          split(pv[2 * q2], h0, l0);
          split(pv[2 * q2 + 1], h1, l1);
          ph[q2] = pack2(h0, h1);
          pl[q2] = pack2(l0, l1);
        }
        // A: a0 = (row r, k 2i..) = n-tile 2kt rows r; a1 = rows r + 8; a2 = n-tile 2kt + 1 rows r; a3
        const uint32_t a0h = ph[0], a1h = ph[1], a2h = ph[2], a3h = ph[3];
        const uint32_t a0l = pl[0], a1l = pl[1], a2l = pl[2], a3l = pl[3];
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t bh[4], bl[4];
          const uint32_t off = (uint32_t)(16 * kt) * 2u + (uint32_t)(16 * np * VS) * 2u;
          ldsm_x4(vb_hi + off, bh[0], bh[1], bh[2], bh[3]);
          ldsm_x4(vb_lo + off, bl[0], bl[1], bl[2], bl[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float(&acc)[4] = O[2 * np + e];
            mma16816(acc, a0h, a1h, a2h, a3h, bh[2 * e], bh[2 * e + 1]);
            mma16816(acc, a0h, a1h, a2h, a3h, bl[2 * e], bl[2 * e + 1]);
            mma16816(acc, a0l, a1l, a2l, a3l, bh[2 * e], bh[2 * e + 1]);
          }
        }
      }
    }
  }

  // ---- normalise, unfold sigma_v, undo the rotation, write the rows
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    lrow[k] += __shfl_xor_sync(FULL, lrow[k], 1);
    lrow[k] += __shfl_xor_sync(FULL, lrow[k], 2);
  }
  const float inv0 = lrow[0] > 0.f ? 1.f / lrow[0] : 0.f, inv1 = lrow[1] > 0.f ? 1.f / lrow[1] : 0.f;
  __syncthreads();  // every warp is done with the last tile before its space is reused
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int ch = 8 * n + 2 * i4;
    float* o0 = sO + (size_t)(16 * warp + r) * D + ch;
    float* o1 = sO + (size_t)(16 * warp + r + 8) * D + ch;
    o0[0] = O[n][0] * inv0;
    o0[1] = O[n][1] * inv0;
    o1[0] = O[n][2] * inv1;
    o1[1] = O[n][3] * inv1;
  }
  __syncwarp();
  const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
  float4 sv = make_float4(1.f, 1.f, 1.f, 1.f);
  if (a.sinkhorn)
    sv = make_float4(__half2float(sig_v[4 * lane]), __half2float(sig_v[4 * lane + 1]), __half2float(sig_v[4 * lane + 2]),
                     __half2float(sig_v[4 * lane + 3]));
  for (int rr = 0; rr < 16; ++rr) {
    const int row = 16 * warp + rr;
    if (row >= nrows) break;
    const float4 o = *reinterpret_cast<const float4*>(sO + (size_t)row * D + 4 * lane);
    float y0 = o.x * sv.x, y1 = o.y * sv.y, y2 = o.z * sv.z, y3 = o.w * sv.w;
    hadamard_warp(y0, y1, y2, y3, lane);
    *reinterpret_cast<float4*>(out_row(row) + 4 * lane) =
        make_float4(y0 * C_WHT * sg.x, y1 * C_WHT * sg.y, y2 * C_WHT * sg.z, y3 * C_WHT * sg.w);
  }
}

template <int KF>
cudaError_t launch_kf(const PrefillArgs& a, cudaStream_t s) {
  const size_t smem = Tile<KF>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int qpt = ROWS / a.g;
  const long long gx = (a.T + qpt - 1) / qpt;
  const long long gz = (long long)a.batch * a.n_layers_call;
  if (gx > 0x7fffffffLL || a.Hkv > 65535 || gz > 65535) return cudaErrorInvalidValue;
  prefill_kernel<KF><<<dim3((unsigned)gx, (unsigned)a.Hkv, (unsigned)gz), THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_scratch_bytes(int n_layers_call, int batch, int Hkv, int W) {
  // the window ring of the call's units, K and V
  return 2 * align256((size_t)n_layers_call * batch * Hkv * W * D * sizeof(float));
}

cudaError_t launch_prefill(const PrefillArgs& a, const AppendArgs& app, cudaStream_t s) {
  if (a.W > 0) {
    const size_t n4 = (size_t)a.n_layers_call * a.batch * a.Hkv * a.W * D / 4;
    const size_t want = (n4 + 255) / 256;
    const unsigned blocks = (unsigned)(want < 4096 ? want : 4096);
    snapshot_kernel<<<blocks, 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_append(app, s);
  if (e != cudaSuccess) return e;
  return a.k_format == KVQ_TQ3_QJL ? launch_kf<KVQ_TQ3_QJL>(a, s)
         : a.k_format == KVQ_Q8G32 ? launch_kf<KVQ_Q8G32>(a, s)
                                   : launch_kf<KVQ_Q4G32>(a, s);
}

}  // namespace kvq
