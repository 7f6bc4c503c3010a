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
// Attention kernel: one CTA = 128 (query, head) rows of one (layer, sequence, kv-head) unit, one
// row per TMEM lane; the products run on the 5th-generation tensor cores (tcgen05.mma, kind::f16,
// fp32 accumulators in tensor memory):
//  * Every key tile -- 64 positions: one quantised page, or 64 raw window positions -- is written
//    to shared memory as fp16 hi/lo planes of its value in the quantised keys' space: the rotated,
//    balanced vector for Q4G32 / Q8G32 keys (raw keys and values rotated and divided by sigma on
//    the fly), and for TQ3 keys the 256-wide vector [n c^, n sqrt(pi/2)/128 gamma (2b - 1)] that
//    dots with [q~, S q~] to the QJL estimate (raw keys padded with zeros).  Values go in
//    transposed (channel-major) planes.  Both use the canonical K-major, no-swizzle core-matrix
//    layout (8 rows x 16 bytes per core matrix).
//  * The query tile (hi/lo) sits in tensor memory for the whole CTA and is the A operand of the
//    logits S = Qhi Khi + Qhi Klo + Qlo Khi (about 22 significant bits: attention outputs are small
//    against the values they average, so fp16 alone would not meet the 2e-3 bar).
//  * Softmax warps read S from tensor memory (one row per thread), mask, take the online softmax in
//    base 2 against a lazily raised reference (raised only when a row's maximum passes it by 8, so
//    weights stay below 2^8 and the output rows are rescaled rarely), and write the weights back in
//    place as fp16 hi/lo: the A operand of O += Phi Vhi + Phi Vlo + Plo Vhi.
//  * Warp roles: 4 softmax warps (TMEM lane quarters), 2 MMA-issuing warps (the logits, and P.V;
//    the first owns the TMEM allocation), 8 dequantising warps filling an NS-stage shared-memory
//    ring; every hand-off is an mbarrier (tcgen05.commit for the tensor-core side), every wait
//    bounded.
//  * Quantised and raw tiles cover disjoint (row, position) pairs through their masks: position j
//    is quantised for query P when j <= P - window, raw when P - window < j <= P.
//  * The output row is normalised, unfolded (sigma_v) and unrotated at the end.
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int ROWS = 128;    // (query, head) rows per CTA = MMA M = TMEM lanes
constexpr int NT = 64;       // key positions per tile (one page) = logits N
constexpr int N_SOFT = 4;    // softmax warps
constexpr int MMA_WARP = 4;  // issues the logits products; the warp owns the TMEM allocation
constexpr int PV_WARP = 5;   // issues the P.V products
constexpr int DQ_WARP0 = 6;  // first dequantising warp
constexpr int N_DQ = 8;
constexpr int THREADS = (DQ_WARP0 + N_DQ) * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_AT = 8.f;  // raise a row's softmax reference when its maximum passes it by this
constexpr unsigned long long WAIT_NS = 1000000000ull;  // give up a wait after ~1 s

// instruction descriptors (kind::f16): fp32 accumulator, fp16 A and B, both K-major, dense
constexpr uint32_t idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t IDESC_S = idesc(ROWS, NT);  // logits: 128 x 64
constexpr uint32_t IDESC_O = idesc(ROWS, D);   // P.V: 128 x 128

template <int KF>
struct Cfg {
  static constexpr bool TQ = KF == KVQ_TQ3_QJL;
  static constexpr int KD = TQ ? 256 : 128;          // width of the query: [q~] or [q~, S q~]
  static constexpr int NS = TQ ? 2 : 3;              // pipeline stages
  static constexpr uint32_t K_PLANE = NT * D * 2;    // one fp16 plane of a key tile: 64 positions x 128
  // key planes: hi, lo (Q4G32 / Q8G32 keys and every raw tile); TQ3 quantised tiles: exact
  // centroids, then the QJL part's hi and lo
  static constexpr int K_PLANES = TQ ? 3 : 2;
  static constexpr uint32_t V_PLANE = D * NT * 2;    // one fp16 plane of a transposed value tile
  static constexpr uint32_t V_OFF = K_PLANES * K_PLANE;
  static constexpr uint32_t STAGE = V_OFF + 2 * V_PLANE;
  static constexpr uint32_t SMEM = NS * STAGE;
  static constexpr uint32_t Q_STRIDE = 2 * KD * 2 + 16;  // query staging row: hi halves, lo halves, pad
  // tensor-memory columns: Q hi | Q lo | O | S/P buffer 0 | S/P buffer 1
  static constexpr uint32_t C_QHI = 0, C_QLO = KD / 2, C_O = KD, C_S = KD + D;
  static_assert(C_S + 2 * NT <= TMEM_COLS, "tensor memory");
  static_assert((uint32_t)ROWS * Q_STRIDE + (uint32_t)(THREADS / 32) * D * 4 <= SMEM,
                "query staging and the projection rows fit the ring");
  static_assert((uint32_t)ROWS * (D + 4) * 4 <= SMEM, "output staging fits the ring");
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on a phase.  false: this CTA gave up (another role gave up first, or ~1 s passed:
// the status word gets KVQ_DEV_TIMEOUT and the CTA's abort flag is raised).
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* status) {
  if (bar_try(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (true) {
    for (int i = 0; i < 16; ++i)
      if (bar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (gtimer() - t0 > WAIT_NS) {
      atomicOr(status, KVQ_DEV_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
// make this thread's generic shared-memory writes visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: K-major, no swizzle; lbo = byte stride between core matrices
// along K, sbo = byte stride between 8-row groups
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// D[tmem] (+)= A[tmem] * B[smem]^T, issued by the warp's elected lane (lane 0 of a converged warp);
// every lane of the warp executes the call
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p, e;\nelect.sync _|e, 0xffffffff;\nsetp.ne.b32 p, %4, 0;\n"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}
// arrive on bar once every tcgen05 operation the elected lane issued so far has completed (the
// same lane that issued the products: elect.sync picks the lowest lane of a converged warp)
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(smem_u32(bar))
      : "memory");
}

#define KVQ_R8(o, i) o(r[i + 0]), o(r[i + 1]), o(r[i + 2]), o(r[i + 3]), o(r[i + 4]), o(r[i + 5]), o(r[i + 6]), o(r[i + 7])
#define KVQ_OUT(x) "=r"(x)
#define KVQ_IN(x) "r"(x)

// this warp's 32 lanes x 32 consecutive 32-bit columns
__device__ __forceinline__ void tm_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : KVQ_R8(KVQ_OUT, 0), KVQ_R8(KVQ_OUT, 8), KVQ_R8(KVQ_OUT, 16), KVQ_R8(KVQ_OUT, 24)
      : "r"(taddr));
}
__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      KVQ_R8(KVQ_IN, 0), KVQ_R8(KVQ_IN, 8), KVQ_R8(KVQ_IN, 16), KVQ_R8(KVQ_IN, 24)
      : "memory");
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      KVQ_R8(KVQ_IN, 0), KVQ_R8(KVQ_IN, 8)
      : "memory");
}
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
// fp16 hi/lo split of a pair: hi = fp16(v), lo = fp16(v - hi); element a in the low half
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2u(h);
  lo = h2u(__floats2half2_rn(a - hf.x, b - hf.y));
}
// 8 consecutive K-elements of one row as hi and lo 16-byte chunks
__device__ __forceinline__ void store8(uint8_t* hi_plane, uint8_t* lo_plane, uint32_t off, const float (&v)[8]) {
  uint4 h, l;
  split2(v[0], v[1], h.x, l.x);
  split2(v[2], v[3], h.y, l.y);
  split2(v[4], v[5], h.z, l.z);
  split2(v[6], v[7], h.w, l.w);
  *reinterpret_cast<uint4*>(hi_plane + off) = h;
  *reinterpret_cast<uint4*>(lo_plane + off) = l;
}
// byte offset of element (row, k) of a K-major no-swizzle operand with R rows, core matrices
// ordered K-group-major: (k / 8) (R / 8) 128 + (row / 8) 128 + (row % 8) 16 + (k % 8) 2
__device__ __forceinline__ uint32_t cm_off(int row, int k, int R) {
  return (uint32_t)((k >> 3) * (R >> 3) * 128 + (row >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

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
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  using C = Cfg<KF>;
  constexpr int KD = C::KD, NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t kfull[NS], kempty[NS], vfull[NS], vempty[NS];
  __shared__ __align__(8) uint64_t sfull[2], pfull[2], pvdone[2], ofull, sdone;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t cent2_sh[64];
  __shared__ uint4 nbuf[N_SOFT][8];  // TQ3: the current tile's 64 position norms (fp16), per softmax warp  // TQ3: half2 (cent[v & 7], cent[v >> 3]) of a record byte's codes v
  __shared__ int abort_sh;

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

  // positions of this CTA's queries: P = p0 + t0 + tl; the quantised positions any of them reads are
  // [0, qend), the raw ones [rlo, Pmax]; tiles: quantised pages 0 .. nqt-1, then raw tiles from rbeg
  const int Pmin = p0 + t0, Pmax = p0 + t0 + nq - 1;
  const int qend = W > 0 ? max(0, Pmax - W + 1) : Pmax + 1;
  const int rlo = W > 0 ? max(0, Pmin - W + 1) : 0;
  const int nqt = (qend + NT - 1) / NT;
  const int rbeg = rlo & ~(NT - 1);
  const int ntiles = nqt + (W > 0 ? (Pmax - rbeg) / NT + 1 : 0);
  const int* bt_seq = a.block_table + (size_t)b * a.max_pages_per_seq;

  // ---- set-up: barriers, tensor memory, codebook
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      bar_init(&kfull[s], N_DQ);
      bar_init(&kempty[s], 1);
      bar_init(&vfull[s], N_DQ);
      bar_init(&vempty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&sfull[i], 1);
      bar_init(&pfull[i], N_SOFT);
      bar_init(&pvdone[i], 1);
    }
    bar_init(&ofull, 1);
    bar_init(&sdone, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (C::TQ && tid < 64)
    cent2_sh[tid] = (uint32_t)__half_as_ushort(a.p.cb->cent[tid & 7]) |
                    ((uint32_t)__half_as_ushort(a.p.cb->cent[tid >> 3]) << 16);
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_sh)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }

  // ---- query tile: q~ = c H (s . q) [. sigma_k] in base-2 logit units (TQ3: also S q~), staged as
  // fp16 hi/lo rows in shared memory, then copied to tensor memory by the lane's own softmax thread
  {
    const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
    float4 sk = make_float4(1.f, 1.f, 1.f, 1.f);
    if (a.sinkhorn) {
      const __half* sig = a.p.sigk + ((size_t)layer * H + h) * D + 4 * lane;
      sk = make_float4(__half2float(sig[0]), __half2float(sig[1]), __half2float(sig[2]), __half2float(sig[3]));
    }
    // TQ3 projection scratch: one 128-float row per warp, after the staging rows
    float* qtmp = reinterpret_cast<float*>(smem + (size_t)ROWS * C::Q_STRIDE) + warp * D;
    for (int row = warp; row < ROWS; row += THREADS / 32) {
      const int tl = row / g, hh = row % g;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < nrows)
        x = load4_in(a.q, ((((size_t)ll * B + b) * Hq + (size_t)h * g + hh) * T + t0 + tl) * D + 4 * lane, a.in_bf16);
      float y0 = x.x * sg.x, y1 = x.y * sg.y, y2 = x.z * sg.z, y3 = x.w * sg.w;
      hadamard_warp(y0, y1, y2, y3, lane);
      const float sc = C_WHT * LOGIT_SCALE;
      const float yv[4] = {y0 * sc * sk.x, y1 * sc * sk.y, y2 * sc * sk.z, y3 * sc * sk.w};
      uint8_t* st = smem + (size_t)row * C::Q_STRIDE;
      uint2 hv, lv;
      split2(yv[0], yv[1], hv.x, lv.x);
      split2(yv[2], yv[3], hv.y, lv.y);
      *reinterpret_cast<uint2*>(st + 8 * lane) = hv;
      *reinterpret_cast<uint2*>(st + 2 * KD + 8 * lane) = lv;
      if (C::TQ) {
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
        split2(acc.x, acc.y, hv.x, lv.x);
        split2(acc.z, acc.w, hv.y, lv.y);
        *reinterpret_cast<uint2*>(st + 2 * D + 8 * lane) = hv;
        *reinterpret_cast<uint2*>(st + 2 * KD + 2 * D + 8 * lane) = lv;
        __syncwarp();
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (warp < N_SOFT) {
    // row = TMEM lane 32 warp + lane: column c of a plane holds K-elements 2c (low half), 2c + 1
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const uint8_t* st = smem + (size_t)tid * C::Q_STRIDE;
#pragma unroll 1
    for (int part = 0; part < 2; ++part)
#pragma unroll 1
      for (int c0 = 0; c0 < KD / 2; c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 u = *reinterpret_cast<const uint4*>(st + part * 2 * KD + 4 * c0 + 16 * i);
          r[4 * i] = u.x;
          r[4 * i + 1] = u.y;
          r[4 * i + 2] = u.z;
          r[4 * i + 3] = u.w;
        }
        tm_st32(lane_addr + (part ? C::C_QLO : C::C_QHI) + c0, r);
      }
    tm_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  auto tile_j0 = [&](int it) { return it < nqt ? it * NT : rbeg + (it - nqt) * NT; };

  if (warp == MMA_WARP || warp == PV_WARP) {
    // ================================================================ MMA issue
    // Two issuing warps on different schedulers: MMA_WARP issues every logits product, PV_WARP
    // every P.V product.  Each whole warp runs its loop (so descriptors and addresses stay
    // warp-uniform) and one elected lane issues each tcgen05.mma / commit: issued from a divergent
    // single-lane branch, every product cost ~1.7x more issue time.  The k-step loops stay rolled
    // (descriptors advanced by constants in their 14-bit start-address field): four roles share
    // each scheduler's instruction cache.
    const uint32_t sbase = smem_u32(smem);
    bool ok = true;
    if (warp == MMA_WARP) {
      for (int it = 0; it < ntiles; ++it) {
        // logits of tile it into S buffer it & 1 (free once P.V of tile it - 2 has read its weights)
        const int s = it % NS, bb = it & 1;
        ok = __all_sync(FULL, bar_wait(&kfull[s], (it / NS) & 1, &abort_sh, a.p.status) &&
                                  (it < 2 || bar_wait(&pvdone[bb], ((it - 2) >> 1) & 1, &abort_sh, a.p.status)));
        if (!ok) break;
        tc_fence_after();
        uint64_t kh = sdesc(sbase + s * C::STAGE, 1024, 128);
        uint32_t qa = tmem + C::C_QHI;
        const uint32_t dS = tmem + C::C_S + NT * bb;
        if (C::TQ && it < nqt) {
          // TQ3 quantised tile: S' = Q~ . C (exact centroids: hi and lo of the query) + (S q~) . W
          // (hi/lo of the QJL part); the softmax multiplies column j by the position's norm
#pragma unroll 1
          for (int ks = 0; ks < D / 16; ++ks, kh += 128, qa += 8) {
            mma_ts(dS, qa, kh, IDESC_S, ks > 0);
            mma_ts(dS, qa + (C::C_QLO - C::C_QHI), kh, IDESC_S, 1);
          }
          kh += (C::K_PLANE >> 4) - 128 * (D / 16);  // the QJL planes; qa now at the S q~ columns
#pragma unroll 1
          for (int ks = 0; ks < D / 16; ++ks, kh += 128, qa += 8) {
            mma_ts(dS, qa, kh, IDESC_S, 1);
            mma_ts(dS, qa, kh + (C::K_PLANE >> 4), IDESC_S, 1);
            mma_ts(dS, qa + (C::C_QLO - C::C_QHI), kh, IDESC_S, 1);
          }
        } else {
          // hi/lo key planes against the first 128 query columns
#pragma unroll 1
          for (int ks = 0; ks < D / 16; ++ks, kh += 128, qa += 8) {
            mma_ts(dS, qa, kh, IDESC_S, ks > 0);
            mma_ts(dS, qa, kh + (C::K_PLANE >> 4), IDESC_S, 1);
            mma_ts(dS, qa + (C::C_QLO - C::C_QHI), kh, IDESC_S, 1);
          }
        }
        mma_commit(&sfull[bb]);
        mma_commit(&kempty[s]);
      }
    } else {
      for (int it = 0; it < ntiles; ++it) {
        // P.V of tile it: weights from S buffer it & 1 (k-step ks: hi pairs in columns 16 ks .. +7,
        // lo pairs in 16 ks + 8 .. +15), values from its stage
        const int s = it % NS, bb = it & 1;
        ok = __all_sync(FULL, bar_wait(&pfull[bb], (it >> 1) & 1, &abort_sh, a.p.status) &&
                                  bar_wait(&vfull[s], (it / NS) & 1, &abort_sh, a.p.status));
        if (!ok) break;
        tc_fence_after();
        uint64_t vh = sdesc(sbase + s * C::STAGE + C::V_OFF, 2048, 128);
        uint32_t pa = tmem + C::C_S + NT * bb;
#pragma unroll 1
        for (int ks = 0; ks < NT / 16; ++ks, vh += 256, pa += 16) {
          mma_ts(tmem + C::C_O, pa, vh, IDESC_O, (it > 0 || ks > 0));
          mma_ts(tmem + C::C_O, pa, vh + (C::V_PLANE >> 4), IDESC_O, 1);
          mma_ts(tmem + C::C_O, pa + 8, vh, IDESC_O, 1);
        }
        mma_commit(&vempty[s]);
        mma_commit(&pvdone[bb]);
      }
    }
    // every product this warp issued lands before the output is read or the columns are freed
    // (the wait is bounded; a CTA that gave up still waits here for what it issued)
    uint64_t* done = warp == PV_WARP ? &ofull : &sdone;
    mma_commit(done);
    const unsigned long long t0w = gtimer();
    while (!bar_try(done, 0) && gtimer() - t0w < WAIT_NS) {
    }
    __syncwarp();
  } else if (warp >= DQ_WARP0) {
    // ================================================================ dequantising warps
    // Key task (position t = dq & 63, part = dq >> 6): 8 consecutive lanes write 8 consecutive
    // positions of one K-group, conflict-free.  Value task (octet pq, channel row rr, group G) with
    // the lane bits ordered (rr0, pq0, pq1, rr1, rr2, pq2, G0, G1) and the channel order within the
    // task rotated by pq: the 8 lanes of a store phase write 8 distinct channel rows of one core
    // matrix, conflict-free.  The next page's words are loaded into registers before the current
    // page is coded, so their latency hides behind the current tile's work.
    const int dq = tid - DQ_WARP0 * 32, dw = dq >> 5;
    const int kt = dq & 63, kpart = dq >> 6, ktt = kt & 31;
    const int vrr = (dq & 1) | (((dq >> 3) & 3) << 1), vpq = ((dq >> 1) & 3) | (((dq >> 5) & 1) << 2), vG = dq >> 6;
    const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
    const __half* sig_k = a.p.sigk + ((size_t)layer * H + h) * D;
    const __half* sig_v = a.p.sigv + ((size_t)layer * H + h) * D;
    struct Words {
      uint4 k0, k1;    // key words: Q4 (codes, scales|zeros), Q8 (chunks 0-1, 2-3), TQ3 (codes|signs, -)
      uint32_t kx;     // Q8: the group's scale; TQ3: (norm, residual norm) as half2
      uint32_t v[4];   // value words of the task's four position pairs
      uint4 vs, vz;    // value scales and zeros of the octet
      bool bad;
    };
    // block-table entries are read two tiles ahead (bt1: tile it + 1, bt2: tile it + 2), so the page
    // addresses of a prefetch never wait on a table load
    auto bt_at = [&](int it) { return it < nqt ? __ldg(bt_seq + it) : 0; };
    auto load_words = [&](int it, int phys, Words& w) {
      const int j0 = it * NT;  // quantised tiles only (one page each)
      w.bad = phys < 0 || phys >= a.L.n_pages;
      w.k0 = w.k1 = w.vs = w.vz = make_uint4(0u, 0u, 0u, 0u);
      w.kx = 0u;
      w.v[0] = w.v[1] = w.v[2] = w.v[3] = 0u;
      if (w.bad) return;
      const uint8_t* pg = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes;
      if (j0 + kt < qend) {
        const uint8_t* hb = pg + (size_t)(kt >> 5) * a.L.half_bytes;
        if (KF == KVQ_Q4G32) {
          w.k0 = __ldg(reinterpret_cast<const uint4*>(hb + ktt * 64 + 16 * kpart));
          w.k1 = __ldg(reinterpret_cast<const uint4*>(hb + a.L.off_kmeta + ktt * 16));
        } else if (KF == KVQ_Q8G32) {
          const int hq = kpart >> 1, wh = kpart & 1;
          uint2 c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            c[i] = __ldg(reinterpret_cast<const uint2*>(hb + ktt * 128 + 16 * ((2 * i + hq) ^ (ktt & 1)) + 8 * wh));
          w.k0 = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
          w.k1 = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
          w.kx = __ldg(reinterpret_cast<const unsigned short*>(hb + a.L.off_kmeta + ktt * 8) + 2 * hq + wh);
        } else {
          w.k0 = __ldg(reinterpret_cast<const uint4*>(hb + ktt * 64 + 16 * kpart));
          const unsigned short* km = reinterpret_cast<const unsigned short*>(hb + a.L.off_kmeta);
          w.kx = (uint32_t)__ldg(km + ktt) | ((uint32_t)__ldg(km + HALF + ktt) << 16);
        }
      }
      if (j0 + 8 * vpq < qend) {
        const uint8_t* hb = pg + (size_t)(vpq >> 2) * a.L.half_bytes;
        const int tq = 8 * (vpq & 3);  // first position of the octet within its half
#pragma unroll
        for (int x = 0; x < 4; ++x)
          w.v[x] = __ldg(reinterpret_cast<const uint32_t*>(hb + a.L.off_vmain + ((tq >> 1) + x) * 128 +
                                                           16 * ((vrr + 2 * x) & 7) + 4 * vG));
        w.vs = __ldg(reinterpret_cast<const uint4*>(hb + a.L.off_vmeta + 2 * (vG * HALF + tq)));
        w.vz = __ldg(reinterpret_cast<const uint4*>(hb + a.L.off_vmeta + 2 * (4 * HALF + vG * HALF + tq)));
      }
    };
    Words cur, nxt;
    if (nqt > 0) load_words(0, bt_at(0), cur);
    int bt1 = bt_at(1), bt2 = bt_at(2);
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % NS;
      const uint32_t ph = (uint32_t)((it / NS) & 1) ^ 1u;  // phase of the stage's previous use
      const bool raw = it >= nqt;
      const int j0 = tile_j0(it);
      if (it + 1 < nqt) load_words(it + 1, bt1, nxt);
      bt1 = bt2;
      bt2 = bt_at(it + 3);
      uint8_t* khi = smem + s * C::STAGE;
      uint8_t* klo = khi + C::K_PLANE;
      uint8_t* vhi = khi + C::V_OFF;
      uint8_t* vlo = vhi + C::V_PLANE;
      if (!raw && cur.bad && dq == 0) atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
      // ---------------- keys
      // every wait is decided warp-wide, so the warp leaves its loop as one
      if (it >= NS && !__all_sync(FULL, bar_wait(&kempty[s], ph, &abort_sh, a.p.status))) break;
      if (!raw) {
        if (KF == KVQ_Q4G32) {
          // words (part, G) hold channels 32 G + 8 part .. +7 = K-group 4 G + part; meta: 4 scales, 4 zeros
          const uint32_t wd[4] = {cur.k0.x, cur.k0.y, cur.k0.z, cur.k0.w};
          const __half* mh = reinterpret_cast<const __half*>(&cur.k1);
#pragma unroll
          for (int G = 0; G < 4; ++G) {
            const float sc = __half2float(mh[G]), zr = __half2float(mh[4 + G]);
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = zr + sc * (float)((wd[G] >> (4 * e)) & 15u);
            store8(khi, klo, cm_off(kt, 8 * (4 * G + kpart), NT), v);
          }
        } else if (KF == KVQ_Q8G32) {
          // part = (h, wh): chunks m = 2 i + h, words w = 2 wh + wi; word w byte bb is channel
          // 16 (4 h + w) + 2 i + (bb & 1) + 8 (bb >> 1), stored u = c + 128
          const int hq = kpart >> 1, wh = kpart & 1;
          const float d = __half2float(__ushort_as_half((unsigned short)cur.kx));
          const uint32_t cw[4][2] = {{cur.k0.x, cur.k0.y}, {cur.k0.z, cur.k0.w}, {cur.k1.x, cur.k1.y}, {cur.k1.z, cur.k1.w}};
#pragma unroll
          for (int wi = 0; wi < 2; ++wi)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              float v[8];
#pragma unroll
              for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  v[2 * i + e] = d * (float)((int)((cw[i][wi] >> (8 * (2 * hf + e))) & 0xffu) - 128);
              store8(khi, klo, cm_off(kt, 8 * (2 * (4 * hq + 2 * wh + wi) + hf), NT), v);
            }
        } else {
          // TQ3: bytes 16 part .. +15 = codes of channels 32 part .. +31 and signs of projections
          // 32 part .. +31 (byte j: channels 2j, 2j+1).  The norm n is left out (the softmax applies
          // it per position): plane 0 gets the exact fp16 centroids, planes 1 and 2 the hi and lo of
          // w = sqrt(pi/2)/128 gamma with the sign of each projection (sign flips are exact)
          const bool okk = !cur.bad && j0 + kt < qend;
          const float w = QJL_CONST * __half2float(__ushort_as_half((unsigned short)(cur.kx >> 16)));
          const __half whi = __float2half_rn(okk ? w : 0.f);
          const __half wlo = __float2half_rn(okk ? w - __half2float(whi) : 0.f);
          const uint32_t whi2 = (uint32_t)__half_as_ushort(whi) * 0x10001u;
          const uint32_t wlo2 = (uint32_t)__half_as_ushort(wlo) * 0x10001u;
          uint8_t* kw2 = khi + 2 * C::K_PLANE;
          uint4 cw = cur.k0;  // word x of the 16 bytes is consumed at step x (the loop stays rolled)
#pragma unroll 1
          for (int x = 0; x < 4; ++x) {
            uint32_t cc[4], sh[4], sl[4];
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const uint32_t byte = (cw.x >> (8 * y)) & 0xffu, nb = ~byte;
              const uint32_t m = ((nb & 0x40u) << 9) | ((nb & 0x80u) << 24);  // clear bit: -w
              cc[y] = okk ? cent2_sh[byte & 63u] : 0u;
              sh[y] = whi2 ^ m;
              sl[y] = wlo2 ^ m;
            }
            const uint32_t off = cm_off(kt, 8 * (4 * kpart + x), NT);
            *reinterpret_cast<uint4*>(khi + off) = make_uint4(cc[0], cc[1], cc[2], cc[3]);
            *reinterpret_cast<uint4*>(klo + off) = make_uint4(sh[0], sh[1], sh[2], sh[3]);
            *reinterpret_cast<uint4*>(kw2 + off) = make_uint4(sl[0], sl[1], sl[2], sl[3]);
            cw = make_uint4(cw.y, cw.z, cw.w, 0u);
          }
        }
      } else {
        // raw keys j0 .. j0 + 63 in the quantised space (rotated, divided by sigma_k), one warp per
        // position; positions no query of this CTA reads raw are zeroed
        for (int t = dw; t < NT; t += N_DQ) {
          const int j = j0 + t;
          const bool ok = j >= rlo && j <= Pmax;
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ok)
            x = j < p0 ? *reinterpret_cast<const float4*>(a.snap_k + ((((size_t)ll * B + b) * H + h) * W + (j % W)) * D + 4 * lane)
                       : load4_in(a.k, ((((size_t)ll * B + b) * H + h) * T + (j - p0)) * D + 4 * lane, a.in_bf16);
          float y0 = x.x * sg.x, y1 = x.y * sg.y, y2 = x.z * sg.z, y3 = x.w * sg.w;
          hadamard_warp(y0, y1, y2, y3, lane);
          float yv[4] = {y0 * C_WHT, y1 * C_WHT, y2 * C_WHT, y3 * C_WHT};
          if (a.sinkhorn) {
#pragma unroll
            for (int e = 0; e < 4; ++e) yv[e] = yv[e] / __half2float(sig_k[4 * lane + e]);
          }
          uint2 hv, lv;
          split2(ok ? yv[0] : 0.f, ok ? yv[1] : 0.f, hv.x, lv.x);
          split2(ok ? yv[2] : 0.f, ok ? yv[3] : 0.f, hv.y, lv.y);
          const uint32_t off = cm_off(t, 4 * lane, NT);
          *reinterpret_cast<uint2*>(khi + off) = hv;
          *reinterpret_cast<uint2*>(klo + off) = lv;
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) bar_arrive(&kfull[s]);

      // ---------------- values (transposed: row = channel, K = position)
      if (it >= NS && !__all_sync(FULL, bar_wait(&vempty[s], ph, &abort_sh, a.p.status))) break;
      if (!raw) {
        // words of pairs p = 4 (pq & 3) .. +3 at 16 ((rr + 2 (p & 3)) & 7) + 4 G hold channels
        // 32 G + 4 rr .. +3 of both positions of the pair as bytes [t0 b0, t1 b0, t0 b1, t1 b1]
        // (channel 4 rr + e: byte e >> 1, nibble e & 1)
        const __half* scs = reinterpret_cast<const __half*>(&cur.vs);
        const __half* zrs = reinterpret_cast<const __half*>(&cur.vz);
        float sc[8], zr[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const bool okt = !cur.bad && j0 + 8 * vpq + k < qend;
          sc[k] = okt ? __half2float(scs[k]) : 0.f;
          zr[k] = okt ? __half2float(zrs[k]) : 0.f;
        }
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int e = (k + vpq) & 3;
          const int sh = 16 * (e >> 1) + 4 * (e & 1);
          float v[8];
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2)
              v[2 * x + s2] = zr[2 * x + s2] + sc[2 * x + s2] * (float)((cur.v[x] >> (sh + 8 * s2)) & 15u);
          store8(vhi, vlo, cm_off(32 * vG + 4 * vrr + e, 8 * vpq, D), v);
        }
      } else {
        for (int t = dw; t < NT; t += N_DQ) {
          const int j = j0 + t;
          const bool ok = j >= rlo && j <= Pmax;
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (ok)
            x = j < p0 ? *reinterpret_cast<const float4*>(a.snap_v + ((((size_t)ll * B + b) * H + h) * W + (j % W)) * D + 4 * lane)
                       : load4_in(a.v, ((((size_t)ll * B + b) * H + h) * T + (j - p0)) * D + 4 * lane, a.in_bf16);
          float y0 = x.x * sg.x, y1 = x.y * sg.y, y2 = x.z * sg.z, y3 = x.w * sg.w;
          hadamard_warp(y0, y1, y2, y3, lane);
          float yv[4] = {y0 * C_WHT, y1 * C_WHT, y2 * C_WHT, y3 * C_WHT};
          if (a.sinkhorn) {
#pragma unroll
            for (int e = 0; e < 4; ++e) yv[e] = yv[e] / __half2float(sig_v[4 * lane + e]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float val = ok ? yv[e] : 0.f;
            const __half hi = __float2half_rn(val);
            const __half lo = __float2half_rn(val - __half2float(hi));
            const uint32_t off = cm_off(4 * lane + e, t, D);
            *reinterpret_cast<__half*>(vhi + off) = hi;
            *reinterpret_cast<__half*>(vlo + off) = lo;
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) bar_arrive(&vfull[s]);
      cur = nxt;
    }
  } else {
    // ================================================================ softmax (thread = row)
    const int row = tid;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const int P = row < nrows ? p0 + t0 + row / g : -1;
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    // block-table entries of tiles it and it + 1, read ahead
    int bt0 = nqt > 0 ? __ldg(bt_seq) : 0, bt1 = nqt > 1 ? __ldg(bt_seq + 1) : 0;
    for (int it = 0; it < ntiles && ok; ++it) {
      const int bb = it & 1;
      const bool raw = it >= nqt;
      const int j0 = tile_j0(it);
      const int phys = bt0;
      bt0 = bt1;
      bt1 = it + 2 < nqt ? __ldg(bt_seq + it + 2) : 0;
      const bool bad = !raw && (phys < 0 || phys >= a.L.n_pages);
      // valid positions of this row in the tile: [lo, hi]
      int lo = 1, hi = 0;
      if (P >= 0 && !bad) {
        if (!raw) {
          lo = 0;
          hi = W > 0 ? P - W : P;
        } else {
          lo = P - W + 1;
          hi = P;
        }
      }
      // TQ3 quantised tile: the positions' norms n (fp16, the page's key metadata), requested before
      // the wait; column j of the tile's logits is n_j S'_j
      if (C::TQ && !raw && !bad) {
        __syncwarp();  // the previous tile's reads of the warp's buffer are done
        if (lane < 8) {
          const uint8_t* pgp = a.p.pages + (((size_t)layer * a.L.n_pages + phys) * H + h) * (size_t)a.L.page_bytes;
          nbuf[warp][lane] =
              __ldg(reinterpret_cast<const uint4*>(pgp + (size_t)(lane >> 2) * a.L.half_bytes + a.L.off_kmeta) + (lane & 3));
        }
        __syncwarp();
      }
      // waits are decided warp-wide: the tensor-memory loads and stores below are warp-collective
      if (!__all_sync(FULL, bar_wait(&sfull[bb], (it >> 1) & 1, &abort_sh, a.p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[2][32];
      tm_ld32(lane_addr + C::C_S + NT * bb, sr[0]);
      tm_ld32(lane_addr + C::C_S + NT * bb + 32, sr[1]);
      tm_wait_ld();
      const bool all_valid = j0 >= lo && j0 + NT - 1 <= hi;
      float x[NT];
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const bool scale_n = C::TQ && !raw && !bad;
#pragma unroll
      for (int c = 0; c < NT; ++c) {
        float sv = __uint_as_float(sr[c >> 5][c & 31]);
        if (C::TQ && scale_n) sv *= __half2float(reinterpret_cast<const __half*>(nbuf[warp])[c]);
        x[c] = (all_valid || (j0 + c >= lo && j0 + c <= hi)) ? sv : -INFINITY;
        m4[c & 3] = fmaxf(m4[c & 3], x[c]);
      }
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      // raise the reference when the row's maximum passes it by RESCALE_AT (the first finite
      // maximum included); the output row accumulated so far is rescaled in tensor memory once the
      // previous tile's P.V has landed
      const bool raise = mx > mref + RESCALE_AT;
      float alpha = 1.f;
      if (raise) {
        alpha = mref == -INFINITY ? 1.f : ex2(mref - mx);
        lsum *= alpha;
        mref = mx;
      }
      if (__any_sync(FULL, raise && alpha != 1.f) && it >= 1) {
        if (!__all_sync(FULL, bar_wait(&pvdone[(it - 1) & 1], ((it - 1) >> 1) & 1, &abort_sh, a.p.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tm_ld32(lane_addr + C::C_O + c0, o);
          tm_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tm_st32(lane_addr + C::C_O + c0, o);
        }
      }
      // weights p = 2^(s - m0) as fp16 hi/lo pairs, written in place: the 16 positions of chunk k
      // become hi pairs in columns 16 k .. +7 and lo pairs in 16 k + 8 .. +15 (the A operand of
      // P.V k-step k)
      const float m0 = mref == -INFINITY ? 0.f : mref;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int k = 0; k < NT / 16; ++k) {
        uint32_t pw[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float pa = ex2(x[16 * k + 2 * i] - m0), pb = ex2(x[16 * k + 2 * i + 1] - m0);
          if (i & 1)
            ls1 += pa + pb;
          else
            ls0 += pa + pb;
          split2(pa, pb, pw[i], pw[8 + i]);
        }
        tm_st16(lane_addr + C::C_S + NT * bb + 16 * k, pw);
      }
      lsum += ls0 + ls1;
      tm_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&pfull[bb]);
    }
    // ---- epilogue: O / l, unfold sigma_v, undo the rotation
    if (ok && __all_sync(FULL, bar_wait(&ofull, 0, &abort_sh, a.p.status))) {
      tc_fence_after();
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      float* sO = reinterpret_cast<float*>(smem);  // [ROWS][D + 4]: the ring is idle once every product landed
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tm_ld32(lane_addr + C::C_O + c0, o);
        tm_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(sO + (size_t)row * (D + 4) + c0 + i) =
              make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv, __uint_as_float(o[i + 2]) * inv,
                          __uint_as_float(o[i + 3]) * inv);
      }
      __syncwarp();
      const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
      float4 sv = make_float4(1.f, 1.f, 1.f, 1.f);
      if (a.sinkhorn) {
        const __half* sig_v = a.p.sigv + ((size_t)layer * H + h) * D;
        sv = make_float4(__half2float(sig_v[4 * lane]), __half2float(sig_v[4 * lane + 1]),
                         __half2float(sig_v[4 * lane + 2]), __half2float(sig_v[4 * lane + 3]));
      }
      for (int rr = 0; rr < 32; ++rr) {
        const int orow = 32 * warp + rr;
        if (orow >= nrows) break;
        const float4 o = *reinterpret_cast<const float4*>(sO + (size_t)orow * (D + 4) + 4 * lane);
        float y0 = o.x * sv.x, y1 = o.y * sv.y, y2 = o.z * sv.z, y3 = o.w * sv.w;
        hadamard_warp(y0, y1, y2, y3, lane);
        *reinterpret_cast<float4*>(out_row(orow) + 4 * lane) =
            make_float4(y0 * C_WHT * sg.x, y1 * C_WHT * sg.y, y2 * C_WHT * sg.z, y3 * C_WHT * sg.w);
      }
    }
  }

  // ---- tear-down: every tensor-memory access of the CTA is done before the columns are freed
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

template <int KF>
cudaError_t launch_kf(const PrefillArgs& a, cudaStream_t s) {
  const size_t smem = Cfg<KF>::SMEM;
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
