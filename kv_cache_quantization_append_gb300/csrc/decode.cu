// Decode attention over the quantised KV cache (one launch per call).
//
// What it computes ([QC] "how it works" + PPL table; [KV] TLDR; [TQ] "key idea" and "inference
// cost" rows): for every (layer, sequence b, kv-head h) and each of its g query heads,
//   softmax over t < L of  q.k_t / sqrt(128)  applied to v_t,
// where tokens t < L - window are read from the packed pages and scored in rotated space
// (q~ = c H (s . q) [. sigma_k]), and the last `window` tokens come raw from the FP32 ring.
//
// Design for GB300 (one CTA per SM: 15 consumer warps for Q4G32 keys, 11 for TQ3 keys, + 1
// producer warp):
//  * The work of a call is a list of "steps" -- one 32-token half-page or one 4-slot window chunk
//    of one (layer, sequence, kv-head) unit, window chunks first.
//  * The list is cut into contiguous ranges of equal cost, one per consumer warp of every CTA
//    (stream-K at warp granularity), so every warp streams about the same bytes whatever the
//    sequence lengths and touches only one to a few units.  Consumer warp w owns NSLOT
//    shared-memory stages (slots w + NCW k); lane w of the producer warp streams exactly that
//    warp's range with cp.async.bulk (the 1D TMA path) completing on mbarriers.  Every wait gives
//    up after ~1 s and sets a status bit.
//  * Consumer warps turn nibbles into exact fp16 values in registers (a nibble read as an FP8 E4M3
//    bit pattern is c * 2^-9; the 2^9 is folded into q) and run the logits and P.V as tensor-core
//    mma.sync m16n8k16 (fp32 accumulate): GQA query heads are the N axis (hi and lo halves of q
//    in adjacent columns), per-group scales and zero points are folded out of the products.
//  * Each warp keeps an online-softmax state per unit and, when it leaves the unit, writes a
//    partial record (max, sum, accumulator) to scratch.  A second, small kernel, launched as a
//    programmatic dependent of the first (it starts as the streaming grid completes), merges each
//    query head's records in a fixed order (deterministic), undoes the rotation of the quantised
//    part and combines it with the window part.  No inter-CTA flags, fences or atomics inside the
//    streaming kernel.
#include <atomic>
#include <cfloat>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int REC_FLOATS = 16 + 2 * MAX_GQA * D;
constexpr int KIND_WINDOW = 0, KIND_QUANT = 1;
constexpr unsigned long long WAIT_NS = 1000000000ull;  // give up a pipeline wait after ~1 s
constexpr float LAZY_RAISE = 4.0f;  // log2 headroom of the softmax reference (weights up to 16)
constexpr int MERGE_WARPS = 8;  // warps per CTA of the merge kernels
constexpr long long WIDE_MERGE_RECORDS = 48;  // above this many records per unit, merge with a CTA per head
constexpr int WIDE_MERGE_WARPS = 16;          // warps per CTA of merge_wide_kernel (15 on slices of the records, 1 on the window parts)

// Per-format CTA geometry and shared-memory carve-up (bytes): consumer warps + 1 producer warp.
// Q4G32 keys: 15 consumer warps with 2 stages each at 128 registers (more warps to hide the math's
// latency; measured faster than 11 warps with 3 stages at 168 registers); TQ3 and Q8 keys, whose
// fragments need more registers: 11 consumer warps (12 warps in all: three per SM sub-partition, so
// 168 registers a thread; 13-16 warps leave 128 and spill, measured slower for both).  Build flags
// KVQ_Q4_CONSUMER_WARPS, KVQ_Q4_SLOTS, KVQ_TQ_CONSUMER_WARPS and KVQ_Q8_CONSUMER_WARPS override the
// counts.
template <int KF>
struct Geo {
  static constexpr bool TQ = KF == KVQ_TQ3_QJL;
  static constexpr bool Q8 = KF == KVQ_Q8G32;
#ifndef KVQ_TQ_CONSUMER_WARPS
#define KVQ_TQ_CONSUMER_WARPS 11
#endif
#ifndef KVQ_Q4_CONSUMER_WARPS
#define KVQ_Q4_CONSUMER_WARPS 15
#endif
#ifndef KVQ_Q8_CONSUMER_WARPS
#define KVQ_Q8_CONSUMER_WARPS 11
#endif
  static constexpr int NCW = TQ ? KVQ_TQ_CONSUMER_WARPS : Q8 ? KVQ_Q8_CONSUMER_WARPS : KVQ_Q4_CONSUMER_WARPS;
  static constexpr int NTHREADS = (NCW + 1) * 32;      // + 1 producer warp
#ifndef KVQ_Q4_SLOTS
#define KVQ_Q4_SLOTS 2
#endif
  static constexpr int NSLOT = (TQ || Q8) ? 2 : KVQ_Q4_SLOTS;   // stages owned by each consumer warp
  static constexpr int NSTAGE = NSLOT * NCW;
  // a stage holds one half-page (Q4/Q4 5120 B, TQ3/Q4 4736 B, Q8/Q4 6912 B) or one window chunk
  // (4096 B)
  static constexpr int STAGE = TQ ? 4736 : Q8 ? 6912 : 5120;
  // TQ3 record-byte table: entry v (256 of them) at 256 v: lane j's copy of the centroid pair at
  // +4 j, of the sign pair at +128 + 4 j
  static constexpr int LUT_BYTES = TQ ? 256 * 256 : 0;
  static constexpr int SM_LUT = 0;
  static constexpr int SM_STAGES = SM_LUT + LUT_BYTES;
  static constexpr int SM_BARS = SM_STAGES + NSTAGE * STAGE;
  static constexpr int SM_DESC = SM_BARS + 2 * NSTAGE * 8;
  static constexpr int SM_Q = SM_DESC + NSTAGE * 16;                         // [NCW][4][128] float
  static constexpr int SM_QSUM = SM_Q + NCW * MAX_GQA * D * 4;               // [NCW][4][4] float
  static constexpr int SM_P = SM_QSUM + NCW * 16 * 4;                        // [NCW][2][4][32] fp16
  static constexpr int SM_WML = SM_P + NCW * 2 * MAX_GQA * HALF * 2;         // [NCW][8] float
  static constexpr int SM_WPOS = SM_WML + NCW * 8 * 4;                       // [NCW+1] int4, i64
  static constexpr int SM_SEQ = SM_WPOS + (NCW + 1) * 24;                     // 6 int[batch+1]
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false (and the status bit set) if the phase did not complete within ~1 s.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* status) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try(bar, parity)) return true;
    if (globaltimer() - t0 > WAIT_NS) {
      atomicOr(status, KVQ_DEV_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 2^x in one MUFU op (max relative error 2^-22); 2^-inf = +0
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 32-bit shared-memory load at a shared-window address, for tables written before the loop that
// reads them (behind a barrier).  Not volatile and without a memory clobber, so the compiler may
// schedule it freely; the addresses used depend on record bytes read from a stage after its
// barrier wait, which keeps each load after that wait.
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// The same at a shared-window address given as a register plus a constant offset (the offset
// goes into the load's immediate field: no add instruction).
template <int OFF>
__device__ __forceinline__ uint32_t lds_u32_at(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}
// Shared-window address at which this kernel's dynamic shared memory starts when the kernel has no
// static shared memory: the block's first 1 KB is reserved by the system on this architecture.
// Checked at run time (a kernel that finds another base takes the path with explicit adds).
constexpr uint32_t DYN_SMEM_WINDOW_BASE = 0x400;
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Eight nibbles of w -> four exact fp16 pairs scaled by 2^-9: each nibble is moved into its own
// byte and converted as an FP8 E4M3 value, which for bit patterns 0..15 (exponent field 0 or 1)
// is exactly c * 2^-9.  lo0 = (n0, n2), lo1 = (n4, n6), hi0 = (n1, n3), hi1 = (n5, n7) where n_m is
// the m-th nibble (low nibble of byte k is n_2k).
__device__ __forceinline__ void cvt8(uint32_t w, uint32_t& lo0, uint32_t& lo1, uint32_t& hi0, uint32_t& hi1) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  // a plain shift: the multiply-high form of w >> 4 (integer pipe) measured 4-5 % slower here
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;
  asm("{\n .reg .b16 a, b, c, d;\n mov.b32 {a, b}, %4;\n mov.b32 {c, d}, %5;\n"
      " cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n"
      " cvt.rn.f16x2.e4m3x2 %2, c;\n cvt.rn.f16x2.e4m3x2 %3, d;\n}"
      : "=r"(lo0), "=r"(lo1), "=r"(hi0), "=r"(hi1)
      : "r"(lo), "r"(hi));
}
constexpr float CODE_UNSCALE = 512.0f;  // undoes the 2^-9 of cvt8

__device__ __forceinline__ uint32_t split_pick(float v, bool lo) {
  const __half hi = __float2half_rn(v);
  return lo ? (uint32_t)__half_as_ushort(__float2half_rn(v - __half2float(hi))) : (uint32_t)__half_as_ushort(hi);
}

// floor(n / d) for n >= 0, d > 0: a 32-bit division when both fit (the usual case), else 64-bit
__device__ __forceinline__ long long div_nn(long long n, long long d) {
  if (((unsigned long long)n | (unsigned long long)d) < 0x80000000ull) return (long long)((unsigned)n / (unsigned)d);
  return n / d;
}

struct Seq {
  const int* S;     // steps per sequence
  const int* pre;   // exclusive prefix of S, [batch + 1]
  const int* L;     // validated lengths
  const int* NW;    // window steps per sequence
  const int* C;     // cost of one unit of the sequence (0 when it has no steps)
  const int* cpre;  // exclusive prefix of C, [batch + 1]
};

// Relative costs used to split a call's steps over the warps, in sixteenths of a quantised
// half-page step (measured with per-warp timestamps): a window chunk costs about as much as a
// half-page, and the set-up of a unit (query rotation, its record) about two, charged to the
// unit's first step; with TQ3 keys the set-up also projects each query head through the 128 x 128
// QJL matrix, and a charge of eight half-pages measured best (cost 128: the all-layer call 2,250 →
// 2,236 us; 64, 96, 160-256 no better).  Relative speeds of the consumer warps: the three (two) that
// share an SM sub-partition with the producer warp get about 10 % more issue slots than the others
// and finish their ranges that much earlier, so they get proportionally longer ranges.
constexpr int COST_Q = 16, COST_WIN = 16;
template <int KF>
constexpr int cost_unit() { return KF == KVQ_TQ3_QJL ? 128 : 32; }
template <int KF>
constexpr int cost_max_step() { return cost_unit<KF>() + COST_Q; }
constexpr int SPEED_NORMAL = 10, SPEED_FAST = 11;

// ---- the shared-memory arrays behind Seq, filled by the decode kernel's set-up
// sequence b of (validated) length L: its steps (window chunks first, then quantised half-pages)
template <int KF>
__device__ __forceinline__ void seq_steps(int b, int L, int W, int* sL, int* sNW, int* sS, int* sC) {
  const int Lq = W > 0 ? max(0, L - W) : L;
  const int nw = W > 0 ? (min(L, W) + WCHUNK - 1) / WCHUNK : 0;
  const int nq = (Lq + HALF - 1) / HALF;
  sL[b] = L;
  sNW[b] = nw;
  sS[b] = nw + nq;
  sC[b] = (nw + nq) > 0 ? cost_unit<KF>() + nw * COST_WIN + nq * COST_Q : 0;
}
// warp 0: exclusive prefix sums of the steps and costs of the B sequences, totals at index B
__device__ __forceinline__ void seq_prefix(int lane, int B, const int* sS, const int* sC, int* sPre, int* sCpre) {
  const int per = (B + 31) / 32, b0 = lane * per, b1 = min(B, b0 + per);
  int s = 0, c = 0;
  for (int b = b0; b < b1; ++b) {
    s += sS[b];
    c += sC[b];
  }
  int incl = s, cincl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    const int z = __shfl_up_sync(FULL, cincl, o);
    if (lane >= o) {
      incl += y;
      cincl += z;
    }
  }
  int run = incl - s, crun = cincl - c;
  for (int b = b0; b < b1; ++b) {
    sPre[b] = run;
    run += sS[b];
    sCpre[b] = crun;
    crun += sC[b];
  }
  if (lane == 31) {
    sPre[B] = incl;
    sCpre[B] = cincl;
  }
}

struct Pos {
  int ll, b, h, local;
};

// move a position forward by `by` steps (only called while the target step exists)
__device__ __forceinline__ void advance(Pos& p, int by, int B, int H, const Seq& sq) {
  p.local += by;
  while (p.local >= sq.S[p.b]) {
    p.local -= sq.S[p.b];
    if (++p.h == H) {
      p.h = 0;
      do {
        if (++p.b == B) {
          p.b = 0;
          p.ll++;
        }
      } while (sq.S[p.b] == 0);
    }
  }
}

// ------------------------------------------------------------------ per-warp state
struct QuantState {
  uint32_t qb[8][2];   // B fragments of q~ (K logits), hi/lo interleaved columns
  uint32_t sb[8][2];   // B fragments of S q~ (TQ sign dot)
  uint32_t zb;         // B fragment of the per-group sums of q~ (Q4 zero-point term), hi/lo columns
  float acc[8][4];     // P.V accumulators, m-tile j (16 channels), C fragment
  float zacc[4];       // sum_t p_t z_{t,G}: rows = groups, cols = heads
  float m, l;          // running max / partial sum for head (lane & 3)
};

// Window-part state of a warp: q [4][128] in its shared-memory q slice (reused by the quantised
// part only after the window steps of the unit), m and l in a small shared slice; the accumulator
// [4][128] (16 values per lane) borrows the first four rows of the quantised part's accumulator
// registers, which the unit's quantised steps only start using after its window steps.
struct WinState {
  float* q;
  float* ml;
};

// Partial record of (unit u, global consumer warp gw): [header 16][quantised acc MAX_GQA][128]
// [window acc MAX_GQA][128] floats.  The index u + gw is unique because both the units and the
// warps' step ranges are ordered along the step list.
__device__ __forceinline__ float* record_at(const DecodeArgs& a, int u, int gw) {
  return a.records + (size_t)(u + gw) * REC_FLOATS;
}

template <int KF>
struct Kernel {
  using GE = Geo<KF>;
  static constexpr int NCW = GE::NCW;
  static constexpr int SM_Q = GE::SM_Q, SM_QSUM = GE::SM_QSUM, SM_LUT = GE::SM_LUT;
  static constexpr int SM_P = GE::SM_P;
  const DecodeArgs& a;
  uint8_t* smem;
  int lane, warp;
  bool lut_base_known;  // dynamic shared memory starts at DYN_SMEM_WINDOW_BASE (TQ3 table addressing)
  int B, H, W, g, Hq;
  long long S_layer, S;  // steps per layer, steps of the call
  long long C_layer, C;  // costs per layer, cost of the call
  long long nw;     // warps that own steps; every warp's cost range holds at least one step start
  long long SPtot;  // summed speeds of the nw warps
  Seq sq;

  __device__ Kernel(const DecodeArgs& args, uint8_t* s) : a(args), smem(s) {}

  __device__ __forceinline__ long long steps_before(int ll, int b, int h) const {
    return (long long)ll * S_layer + (long long)H * sq.pre[b] + (long long)h * sq.S[b];
  }
  // Work split: the steps are laid on a cost line in order (step `local` of unit (ll, b, h)
  // starts at cost_at(...)), the line is cut into nw ranges in proportion to the warps' speeds,
  // and warp gw (= CTA * NCW + warp) owns the steps that start in [lb(gw), lb(gw + 1)) with
  // lb(g) = floor(C * SP(g) / SPtot), SP(g) = the summed speeds of warps 0 .. g-1.
  // summed speeds of consumer warps 0 .. w-1 of a CTA
  __device__ __forceinline__ long long speed_prefix(int w) const {
    const int f = NCW & 3;  // sub-partition of the producer warp (warp NCW)
    const int nf = w > f ? (w - f - 1) / 4 + 1 : 0;
    return (long long)SPEED_NORMAL * w + (long long)(SPEED_FAST - SPEED_NORMAL) * nf;
  }
  __device__ __forceinline__ long long speed_before(long long g) const {
    return (g / NCW) * speed_prefix(NCW) + speed_prefix((int)(g % NCW));
  }
  __device__ __forceinline__ long long lb(long long g) const { return div_nn(C * speed_before(g), SPtot); }
  __device__ __forceinline__ long long cost_at(int ll, int b, int h, int local) const {
    long long c = (long long)ll * C_layer + (long long)H * sq.cpre[b] + (long long)h * sq.C[b];
    if (local > 0) {
      const int nwin = sq.NW[b];
      c += cost_unit<KF>() + (long long)min(local, nwin) * COST_WIN + (long long)max(0, local - nwin) * COST_Q;
    }
    return c;
  }
  // warp whose cost range holds cost position c: the last g with speed_before(g) <= T, where
  // lb(g) <= c  <=>  speed_before(g) <= T = floor(((c + 1) SPtot - 1) / C)
  __device__ __forceinline__ int owner(long long c) const {
    const long long T = div_nn((c + 1) * SPtot - 1, C);
    const long long scta = speed_prefix(NCW);
    const long long cta = T / scta, rem = T - cta * scta;
    int w = NCW - 1;
    while (speed_prefix(w) > rem) --w;
    return (int)(cta * NCW + w);
  }
  // global step index of a position
  __device__ __forceinline__ long long step_index(const Pos& p) const {
    return steps_before(p.ll, p.b, p.h) + p.local;
  }
  // first step of warp gw (gw < nw): the first step starting at or after lb(gw)
  __device__ Pos first_step(long long gw) const {
    const long long y = lb(gw);
    Pos p;
    p.ll = (int)div_nn(y, C_layer);
    const long long r = y - (long long)p.ll * C_layer;
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)H * sq.cpre[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    p.b = lo;
    const long long r2 = r - (long long)H * sq.cpre[lo];
    p.h = (int)div_nn(r2, sq.C[lo]);
    const int r3 = (int)(r2 - (long long)p.h * sq.C[lo]);
    const int nwin = sq.NW[lo];
    p.local = (r3 < cost_unit<KF>() + nwin * COST_WIN) ? max(0, r3 - cost_unit<KF>()) / COST_WIN
                                                        : nwin + (r3 - cost_unit<KF>() - nwin * COST_WIN) / COST_Q;
    if (cost_at(p.ll, p.b, p.h, p.local) < y) advance(p, 1, B, H, sq);
    return p;
  }
  // from the per-sequence arrays: the call's steps and costs, and the number of warps with steps
  __device__ __forceinline__ void totals() {
    S_layer = (long long)H * sq.pre[B];
    S = S_layer * a.n_layers_call;
    C_layer = (long long)H * sq.cpre[B];
    C = C_layer * a.n_layers_call;
    nw = 0;
    if (S > 0) {
      // every range, even a normal-speed one, must span at least the longest step
      nw = max(1LL, min((long long)gridDim.x * NCW, C * SPEED_NORMAL / ((long long)cost_max_step<KF>() * SPEED_FAST)));
      SPtot = speed_before(nw);
    }
  }
  // the step ranges of this CTA's warps, located once: lane j of the producer warp finds the first
  // step of consumer warp j, lane NCW that of the next CTA's first warp (this CTA's end)
  __device__ __forceinline__ void locate(int4* sWpos, long long* sWxs) const {
    if (warp == NCW && lane <= NCW) {
      const long long gwj = (long long)blockIdx.x * NCW + lane;
      Pos p = {0, 0, 0, 0};
      long long x = S;
      if (gwj < nw) {
        p = first_step(gwj);
        x = step_index(p);
      }
      sWpos[lane] = make_int4(p.ll, p.b, p.h, p.local);
      sWxs[lane] = x;
    }
  }
  // This thread's share (index i of the grid's NCW * 32 * gridDim consumer threads) of the record
  // ranges of all units, for the merge kernel (a unit of an empty sequence has none)
  __device__ void unit_info_share(long long i) const {
    for (long long u = i; u < a.n_units; u += (long long)NCW * 32 * gridDim.x) {
      const int h = (int)(u % H), b = (int)((u / H) % B), ll = (int)(u / ((long long)H * B));
      int2 info = make_int2(0, 0);
      if (sq.S[b] > 0) unit_owners(ll, b, h, info.x, info.y);
      a.unit_info[u] = info;
    }
  }
  // [first, last] cost positions of unit u's steps' starts, as owner() arguments
  __device__ __forceinline__ void unit_owners(int ll, int b, int h, int& first, int& count) const {
    first = owner(cost_at(ll, b, h, 0));
    count = owner(cost_at(ll, b, h, sq.S[b] - 1)) - first + 1;
  }

  // ---------------------------------------------------------------- unit set-up
  // issue the loads of unit u's g query vectors (lane holds channels 4*lane..+3 of each)
  __device__ __forceinline__ void fetch_q(int u, float4 (&raw)[MAX_GQA]) {
    const int h = u % H, b = (u / H) % B, ll = u / (H * B);
    const size_t qbase = (((size_t)ll * B + b) * Hq + (size_t)h * g) * D;
#pragma unroll
    for (int hh = 0; hh < MAX_GQA; ++hh) {
      raw[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (hh < g) raw[hh] = load4_in(a.q, qbase + (size_t)hh * D + 4 * lane, a.in_bf16);
    }
  }

  __device__ void load_q(int u, QuantState& st, WinState& ws, int kind) {
    float4 raw[MAX_GQA];
    fetch_q(u, raw);
    build_q(u, raw, st, ws, kind);
  }

  // set up the per-unit state of the window part (kind 0) or the quantised part (kind 1)
  __device__ void build_q(int u, const float4 (&raw)[MAX_GQA], QuantState& st, WinState& ws, int kind) {
    const int h = u % H, ll = u / (H * B);
    const int layer = a.layer0 + ll;
    if (kind == KIND_WINDOW) {
#pragma unroll
      for (int hh = 0; hh < MAX_GQA; ++hh) {
        const float4 x = raw[hh];
        *reinterpret_cast<float4*>(ws.q + hh * D + 4 * lane) =
            make_float4(x.x * LOGIT_SCALE, x.y * LOGIT_SCALE, x.z * LOGIT_SCALE, x.w * LOGIT_SCALE);
        st.acc[hh][0] = st.acc[hh][1] = st.acc[hh][2] = st.acc[hh][3] = 0.f;
      }
      if (lane < 8) ws.ml[lane] = lane < 4 ? -INFINITY : 0.f;
      __syncwarp();
      return;
    }
    float* qs = reinterpret_cast<float*>(smem + SM_Q) + warp * MAX_GQA * D;
    float* qsum = reinterpret_cast<float*>(smem + SM_QSUM) + warp * 16;
    const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
#pragma unroll
    for (int hh = 0; hh < MAX_GQA; ++hh) {
      float y0 = raw[hh].x * sg.x, y1 = raw[hh].y * sg.y, y2 = raw[hh].z * sg.z, y3 = raw[hh].w * sg.w;
      hadamard_warp(y0, y1, y2, y3, lane);
      float sc[4] = {C_WHT * LOGIT_SCALE, C_WHT * LOGIT_SCALE, C_WHT * LOGIT_SCALE, C_WHT * LOGIT_SCALE};
      if (a.sinkhorn) {
        const __half* sig = a.p.sigk + ((size_t)layer * H + h) * D + 4 * lane;
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] *= __half2float(sig[e]);
      }
      y0 *= sc[0];
      y1 *= sc[1];
      y2 *= sc[2];
      y3 *= sc[3];
      *reinterpret_cast<float4*>(qs + hh * D + 4 * lane) = make_float4(y0, y1, y2, y3);
      float s = (y0 + y1) + (y2 + y3);
      s += __shfl_xor_sync(FULL, s, 1);
      s += __shfl_xor_sync(FULL, s, 2);
      s += __shfl_xor_sync(FULL, s, 4);
      if ((lane & 7) == 0) qsum[hh * 4 + (lane >> 3)] = s;
    }
    __syncwarp();
    const int r = lane >> 2, i = lane & 3;
    const int head = r >> 1;
    const bool lo = r & 1;
    const bool hv = head < g;
    const float* qh = qs + head * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      int d0, d1, d2, d3;
      if (KF == KVQ_TQ3_QJL) {
        // codes: k-step kk holds channels 32i + 4kk + {0,1 | 2,3}
        d0 = 32 * i + 4 * kk;
        d1 = d0 + 1;
        d2 = d0 + 2;
        d3 = d0 + 3;
      } else if (KF == KVQ_Q8G32) {
        // Q8: k-step kk holds channels 16kk + {2i, 2i+1 | 2i+8, 2i+9}
        d0 = 16 * kk + 2 * i;
        d1 = d0 + 1;
        d2 = d0 + 8;
        d3 = d0 + 9;
      } else {
        // Q4: k-step (G, e) = (kk >> 1, kk & 1) holds channels 32G + 8i + 4e + {0,2 | 1,3}; the codes
        // arrive scaled by 2^-9, so q~ is scaled by 2^9 (exact)
        const int G = kk >> 1, e = kk & 1;
        d0 = 32 * G + 8 * i + 4 * e;
        d1 = d0 + 2;
        d2 = d0 + 1;
        d3 = d0 + 3;
      }
      const float us = (KF == KVQ_Q4G32) ? CODE_UNSCALE : 1.f;
      const uint32_t v0 = hv ? split_pick(qh[d0] * us, lo) : 0u, v1 = hv ? split_pick(qh[d1] * us, lo) : 0u;
      const uint32_t v2 = hv ? split_pick(qh[d2] * us, lo) : 0u, v3 = hv ? split_pick(qh[d3] * us, lo) : 0u;
      st.qb[kk][0] = v0 | (v1 << 16);
      st.qb[kk][1] = v2 | (v3 << 16);
    }
    // zero-point term as one more k-step: k = group G (0..3), column = head (hi | lo)
    st.zb = (hv && i < 2) ? split_pick(qsum[head * 4 + 2 * i], lo) | (split_pick(qsum[head * 4 + 2 * i + 1], lo) << 16)
                          : 0u;
    if (KF == KVQ_TQ3_QJL) {
      // S q~ for each head (lane computes projections 4*lane .. 4*lane+3 from q~), written over q~
      // once every lane has read its q~ fragments; signs use the codes' k-step mapping: k-step kk
      // holds projections 32i + 4kk + {0,1 | 2,3}
      const float4* stp = reinterpret_cast<const float4*>(a.p.qjl_t) + lane;
      float4 sq[MAX_GQA];
#pragma unroll
      for (int hh = 0; hh < MAX_GQA; ++hh) sq[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int j = 0; j < D; ++j) {
        const float4 s4 = stp[j * (D / 4)];
#pragma unroll
        for (int hh = 0; hh < MAX_GQA; ++hh) {
          const float qj = qs[hh * D + j];
          sq[hh].x += s4.x * qj;
          sq[hh].y += s4.y * qj;
          sq[hh].z += s4.z * qj;
          sq[hh].w += s4.w * qj;
        }
      }
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < MAX_GQA; ++hh) *reinterpret_cast<float4*>(qs + hh * D + 4 * lane) = sq[hh];
      __syncwarp();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int p0 = 32 * i + 4 * kk;
        const uint32_t s0 = hv ? split_pick(qh[p0], lo) : 0u, s1 = hv ? split_pick(qh[p0 + 1], lo) : 0u;
        const uint32_t s2 = hv ? split_pick(qh[p0 + 2], lo) : 0u, s3 = hv ? split_pick(qh[p0 + 3], lo) : 0u;
        st.sb[kk][0] = s0 | (s1 << 16);
        st.sb[kk][1] = s2 | (s3 << 16);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) st.acc[j][0] = st.acc[j][1] = st.acc[j][2] = st.acc[j][3] = 0.f;
    st.zacc[0] = st.zacc[1] = st.zacc[2] = st.zacc[3] = 0.f;
    st.m = -INFINITY;
    st.l = 0.f;
    __syncwarp();
  }

  // ---------------------------------------------------------------- window chunk (raw fp32)
  __device__ void window_step(const uint8_t* stage, int ntok, WinState& ws, QuantState& st) {
    const float* Ks = reinterpret_cast<const float*>(stage);
    const float* Vs = Ks + WCHUNK * D;
    float4 q4[MAX_GQA];
#pragma unroll
    for (int hh = 0; hh < MAX_GQA; ++hh) q4[hh] = *reinterpret_cast<const float4*>(ws.q + hh * D + 4 * lane);
    float part[WCHUNK * MAX_GQA];
#pragma unroll
    for (int t = 0; t < WCHUNK; ++t) {
      const float4 k4 = *reinterpret_cast<const float4*>(Ks + t * D + 4 * lane);
#pragma unroll
      for (int hh = 0; hh < MAX_GQA; ++hh)
        part[4 * t + hh] = q4[hh].x * k4.x + q4[hh].y * k4.y + q4[hh].z * k4.z + q4[hh].w * k4.w;
    }
    // transpose-reduce 16 partial dots over 32 lanes: lanes 2v, 2v+1 end with value v = 4t + hh
#pragma unroll
    for (int o = 16, n = 16; o >= 2; o >>= 1, n >>= 1) {
      const bool up = lane & o;
#pragma unroll
      for (int k = 0; k < n / 2; ++k) {
        const float send = up ? part[k] : part[k + n / 2];
        const float keep = up ? part[k + n / 2] : part[k];
        part[k] = keep + __shfl_xor_sync(FULL, send, o);
      }
    }
    part[0] += __shfl_xor_sync(FULL, part[0], 1);
    const int t = lane >> 3, hh = (lane >> 1) & 3;
    const float lg = (t < ntok && hh < g) ? part[0] : -INFINITY;
    float mc = lg;
    mc = fmaxf(mc, __shfl_xor_sync(FULL, mc, 8));
    mc = fmaxf(mc, __shfl_xor_sync(FULL, mc, 16));
    float alpha[MAX_GQA], mk[MAX_GQA];
    float mown = -INFINITY;
#pragma unroll
    for (int k = 0; k < MAX_GQA; ++k) {
      const float mold = ws.ml[k];
      const float mn = fmaxf(mold, __shfl_sync(FULL, mc, 2 * k));
      alpha[k] = (mn == -INFINITY) ? 1.f : exp2f(mold - mn);
      mk[k] = mn;
      if (hh == k) mown = mn;
    }
    const float p = (lg == -INFINITY) ? 0.f : exp2f(lg - mown);
    float ps = p;
    ps += __shfl_xor_sync(FULL, ps, 8);
    ps += __shfl_xor_sync(FULL, ps, 16);
    float lk[MAX_GQA];
#pragma unroll
    for (int k = 0; k < MAX_GQA; ++k) lk[k] = ws.ml[4 + k] * alpha[k] + __shfl_sync(FULL, ps, 2 * k);
#pragma unroll
    for (int k = 0; k < MAX_GQA; ++k) {
      float4 acc = make_float4(st.acc[k][0], st.acc[k][1], st.acc[k][2], st.acc[k][3]);
      acc.x *= alpha[k];
      acc.y *= alpha[k];
      acc.z *= alpha[k];
      acc.w *= alpha[k];
#pragma unroll
      for (int tt = 0; tt < WCHUNK; ++tt) {
        const float pt = __shfl_sync(FULL, p, 8 * tt + 2 * k);
        if (tt < ntok) {
          const float4 v4 = *reinterpret_cast<const float4*>(Vs + tt * D + 4 * lane);
          acc.x += pt * v4.x;
          acc.y += pt * v4.y;
          acc.z += pt * v4.z;
          acc.w += pt * v4.w;
        }
      }
      st.acc[k][0] = acc.x;
      st.acc[k][1] = acc.y;
      st.acc[k][2] = acc.z;
      st.acc[k][3] = acc.w;
    }
    __syncwarp();
    if (lane < MAX_GQA) {
      ws.ml[lane] = mk[0];
#pragma unroll
      for (int k = 1; k < MAX_GQA; ++k)
        if (lane == k) ws.ml[lane] = mk[k];
    } else if (lane < 2 * MAX_GQA) {
      ws.ml[lane] = lk[0];
#pragma unroll
      for (int k = 1; k < MAX_GQA; ++k)
        if (lane - MAX_GQA == k) ws.ml[lane] = lk[k];
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- quantised half-page
  // regions of a 32-token half-page (bytes): K main at 0, V main at 64*HALF, K meta at 128*HALF,
  // V meta after K meta
  static constexpr int OFF_VMAIN = (KF == KVQ_Q8G32 ? 128 : 64) * HALF;
  static constexpr int OFF_KMETA = OFF_VMAIN + 64 * HALF;
  static constexpr int OFF_VMETA = OFF_KMETA + (KF == KVQ_TQ3_QJL ? 4 : KF == KVQ_Q8G32 ? 8 : 16) * HALF;

  // logits of tokens ta = 16mt + r and tb = ta + 8 for head i (this thread's column pair)
  __device__ __forceinline__ void tile_logits(const uint8_t* stage, int mt, const QuantState& st, float& la,
                                              float& lb) {
    const int r = lane >> 2, i = lane & 3;
    const int ta = 16 * mt + r, tb = ta + 8;
    const uint8_t* kmain = stage;
    const uint8_t* kmeta = stage + OFF_KMETA;
    if (KF == KVQ_Q8G32) {
      // Q8 keys: a token's 16-byte chunks 2i (k-steps 0-3) and 2i + 1 (4-7), swizzled by the token's
      // parity (ta and tb have the parity of r); word kk & 3 of a chunk holds the stored bytes
      // u = c + 128 of this lane's A operands, and a byte permute with 0x64 high bytes makes each
      // pair the exact fp16 values 1024 + u = 1152 + c.  Per group G: acc_G = q~_G . (1152 + c);
      // the offset leaves through the zero-point mma: logit = sum_G d_G acc_G - 1152 sum_G d_G qsum_G.
      const int sw = r & 1;
      const uint4 a0 = *reinterpret_cast<const uint4*>(kmain + ta * 128 + 16 * ((2 * i) ^ sw));
      const uint4 a1 = *reinterpret_cast<const uint4*>(kmain + ta * 128 + 16 * ((2 * i + 1) ^ sw));
      const uint4 b0 = *reinterpret_cast<const uint4*>(kmain + tb * 128 + 16 * ((2 * i) ^ sw));
      const uint4 b1 = *reinterpret_cast<const uint4*>(kmain + tb * 128 + 16 * ((2 * i + 1) ^ sw));
      constexpr uint32_t HI = 0x64646464u;
      float acc[4][4];
#pragma unroll
      for (int G = 0; G < 4; ++G) {
        acc[G][0] = acc[G][1] = acc[G][2] = acc[G][3] = 0.f;
#pragma unroll
        for (int sdx = 0; sdx < 2; ++sdx) {
          const int kk = 2 * G + sdx, w = kk & 3;
          const uint4 ca = kk < 4 ? a0 : a1, cb = kk < 4 ? b0 : b1;
          const uint32_t wa = w == 0 ? ca.x : w == 1 ? ca.y : w == 2 ? ca.z : ca.w;
          const uint32_t wb = w == 0 ? cb.x : w == 1 ? cb.y : w == 2 ? cb.z : cb.w;
          mma16816(acc[G], __byte_perm(wa, HI, 0x4140u), __byte_perm(wb, HI, 0x4140u), __byte_perm(wa, HI, 0x4342u),
                   __byte_perm(wb, HI, 0x4342u), st.qb[kk][0], st.qb[kk][1]);
        }
      }
      const uint2 ma = *reinterpret_cast<const uint2*>(kmeta + ta * 8);
      const uint2 mb = *reinterpret_cast<const uint2*>(kmeta + tb * 8);
      // sum_G d_G qsum_G: A row = token, k = group (lanes i = 0, 1 hold groups (0, 1), (2, 3); lanes
      // i = 2, 3 meet a zero B fragment)
      float zacc[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816(zacc, (i & 1) ? ma.y : ma.x, (i & 1) ? mb.y : mb.x, 0u, 0u, st.zb, 0u);
      const float2 da01 = __half22float2(u2h(ma.x)), da23 = __half22float2(u2h(ma.y));
      const float2 db01 = __half22float2(u2h(mb.x)), db23 = __half22float2(u2h(mb.y));
      constexpr float OFFSET = 1152.0f;
      la = da01.x * (acc[0][0] + acc[0][1]) + da01.y * (acc[1][0] + acc[1][1]) + da23.x * (acc[2][0] + acc[2][1]) +
           da23.y * (acc[3][0] + acc[3][1]) - OFFSET * (zacc[0] + zacc[1]);
      lb = db01.x * (acc[0][2] + acc[0][3]) + db01.y * (acc[1][2] + acc[1][3]) + db23.x * (acc[2][2] + acc[2][3]) +
           db23.y * (acc[3][2] + acc[3][3]) - OFFSET * (zacc[2] + zacc[3]);
    } else if (KF == KVQ_TQ3_QJL) {
      // record byte 16i + 2kk + e of a token = its A operands of k-step kk, slot e (k = 2i, 2i+1 for
      // e = 0, 2i + 8, 2i + 9 for e = 1): two 3-bit codes and two QJL sign bits.  One byte_perm
      // puts the byte above this lane's table offset; the entry's centroid pair and +-1 sign pair
      // are read as two 4-byte loads, so that each lands directly in its mma operand register (an
      // 8-byte load would pair a centroid and a sign register, and the operands would need moves).
      // even and odd k-steps accumulate separately: four independent mma chains instead of two
      float cacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint4 ka = *reinterpret_cast<const uint4*>(kmain + ta * 64 + 16 * i);
      const uint4 kb = *reinterpret_cast<const uint4*>(kmain + tb * 64 + 16 * i);
      const uint32_t lane4 = 4u * lane;
      constexpr int LUT_WIN = (int)DYN_SMEM_WINDOW_BASE + SM_LUT;
      if (lut_base_known) {
        // the table's shared-window address is the constant LUT_WIN: one byte_perm per byte
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int wi = kk >> 1;
          const uint32_t wa = wi == 0 ? ka.x : wi == 1 ? ka.y : wi == 2 ? ka.z : ka.w;
          const uint32_t wb = wi == 0 ? kb.x : wi == 1 ? kb.y : wi == 2 ? kb.z : kb.w;
          uint32_t ca[2], cb[2], sa[2], sb[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            // result bytes: [lane4, record byte 2(kk & 1) + e, 0, 0] = 256 v + 4 lane: the lane's
            // copy of entry v's centroid pair; its sign pair is 128 bytes further
            const uint32_t sel = 0x5504u | ((uint32_t)(2 * (kk & 1) + e) << 4);
            const uint32_t pa = __byte_perm(wa, lane4, sel), pb = __byte_perm(wb, lane4, sel);
            ca[e] = lds_u32_at<LUT_WIN>(pa);
            sa[e] = lds_u32_at<LUT_WIN + 128>(pa);
            cb[e] = lds_u32_at<LUT_WIN>(pb);
            sb[e] = lds_u32_at<LUT_WIN + 128>(pb);
          }
          mma16816(cacc[kk & 1], ca[0], cb[0], ca[1], cb[1], st.qb[kk][0], st.qb[kk][1]);
          mma16816(sacc[kk & 1], sa[0], sb[0], sa[1], sb[1], st.sb[kk][0], st.sb[kk][1]);
        }
      } else {
        const uint32_t lut = smem_addr(smem + SM_LUT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int wi = kk >> 1;
          const uint32_t wa = wi == 0 ? ka.x : wi == 1 ? ka.y : wi == 2 ? ka.z : ka.w;
          const uint32_t wb = wi == 0 ? kb.x : wi == 1 ? kb.y : wi == 2 ? kb.z : kb.w;
          uint32_t ca[2], cb[2], sa[2], sb[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t sel = 0x5504u | ((uint32_t)(2 * (kk & 1) + e) << 4);
            const uint32_t pa = lut + __byte_perm(wa, lane4, sel), pb = lut + __byte_perm(wb, lane4, sel);
            ca[e] = lds_u32(pa);
            sa[e] = lds_u32(pa + 128);
            cb[e] = lds_u32(pb);
            sb[e] = lds_u32(pb + 128);
          }
          mma16816(cacc[kk & 1], ca[0], cb[0], ca[1], cb[1], st.qb[kk][0], st.qb[kk][1]);
          mma16816(sacc[kk & 1], sa[0], sb[0], sa[1], sb[1], st.sb[kk][0], st.sb[kk][1]);
        }
      }
      const __half* nrm = reinterpret_cast<const __half*>(kmeta);
      const float na = __half2float(nrm[ta]), nb = __half2float(nrm[tb]);
      const float ga = __half2float(nrm[HALF + ta]), gb = __half2float(nrm[HALF + tb]);
      const float ca0 = (cacc[0][0] + cacc[1][0]) + (cacc[0][1] + cacc[1][1]);
      const float cb0 = (cacc[0][2] + cacc[1][2]) + (cacc[0][3] + cacc[1][3]);
      const float sa0 = (sacc[0][0] + sacc[1][0]) + (sacc[0][1] + sacc[1][1]);
      const float sb0 = (sacc[0][2] + sacc[1][2]) + (sacc[0][3] + sacc[1][3]);
      la = na * (ca0 + QJL_CONST * ga * sa0);
      lb = nb * (cb0 + QJL_CONST * gb * sb0);
    } else {
      const uint4 ka = *reinterpret_cast<const uint4*>(kmain + ta * 64 + 16 * i);
      const uint4 kb = *reinterpret_cast<const uint4*>(kmain + tb * 64 + 16 * i);
      float acc[4][4];
#pragma unroll
      for (int G = 0; G < 4; ++G) {
        acc[G][0] = acc[G][1] = acc[G][2] = acc[G][3] = 0.f;
        // word G of this thread's 16 bytes = channels 32G + 8i .. +7 of the token
        const uint32_t wa = G == 0 ? ka.x : G == 1 ? ka.y : G == 2 ? ka.z : ka.w;
        const uint32_t wb = G == 0 ? kb.x : G == 1 ? kb.y : G == 2 ? kb.z : kb.w;
        uint32_t al0, al1, ah0, ah1, bl0, bl1, bh0, bh1;
        cvt8(wa, al0, al1, ah0, ah1);
        cvt8(wb, bl0, bl1, bh0, bh1);
        mma16816(acc[G], al0, bl0, ah0, bh0, st.qb[2 * G][0], st.qb[2 * G][1]);
        mma16816(acc[G], al1, bl1, ah1, bh1, st.qb[2 * G + 1][0], st.qb[2 * G + 1][1]);
      }
      const uint4 ma = *reinterpret_cast<const uint4*>(kmeta + ta * 16);
      const uint4 mb = *reinterpret_cast<const uint4*>(kmeta + tb * 16);
      // zero-point term sum_G z_G * sum(q~_G) on the tensor core: A row = token, k = group
      // (this thread's k pair 2i, 2i+1 is zero (G0, G1) for i = 0, (G2, G3) for i = 1; lanes i = 2, 3
      // meet a zero B fragment, so any finite pair does there and no lane needs a second select)
      float zacc[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t zla = (i & 1) ? ma.w : ma.z;
      const uint32_t zlb = (i & 1) ? mb.w : mb.z;
      mma16816(zacc, zla, zlb, 0u, 0u, st.zb, 0u);
      const float2 sa01 = __half22float2(u2h(ma.x)), sa23 = __half22float2(u2h(ma.y));
      const float2 sb01 = __half22float2(u2h(mb.x)), sb23 = __half22float2(u2h(mb.y));
      la = (zacc[0] + zacc[1]) + sa01.x * (acc[0][0] + acc[0][1]) + sa01.y * (acc[1][0] + acc[1][1]) +
           sa23.x * (acc[2][0] + acc[2][1]) + sa23.y * (acc[3][0] + acc[3][1]);
      lb = (zacc[2] + zacc[3]) + sb01.x * (acc[0][2] + acc[0][3]) + sb01.y * (acc[1][2] + acc[1][3]) +
           sb23.x * (acc[2][2] + acc[2][3]) + sb23.y * (acc[3][2] + acc[3][3]);
    }
  }

  // Tail half-page (ntok < 32): zero the scales and zeros (and TQ norms) of the missing tokens in
  // shared memory, so that their -inf logits and zero weights never meet stale values; the fence
  // orders these generic-proxy writes before the next bulk copy into the stage.
  __device__ void sanitize_tail(uint8_t* stage, int ntok) {
    __half* vmeta = reinterpret_cast<__half*>(stage + OFF_VMETA);
    for (int idx = lane; idx < 8 * HALF; idx += 32)
      if ((idx % HALF) >= ntok) vmeta[idx] = __float2half_rn(0.f);
    if (KF == KVQ_TQ3_QJL) {
      __half* nrm = reinterpret_cast<__half*>(stage + OFF_KMETA);
      for (int idx = lane; idx < 2 * HALF; idx += 32)
        if ((idx % HALF) >= ntok) nrm[idx] = __float2half_rn(0.f);
    } else if (KF == KVQ_Q8G32) {
      for (int t = ntok + lane; t < HALF; t += 32)
        *reinterpret_cast<uint2*>(stage + OFF_KMETA + t * 8) = make_uint2(0u, 0u);
    } else {
      for (int t = ntok + lane; t < HALF; t += 32)
        *reinterpret_cast<uint4*>(stage + OFF_KMETA + t * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
  }

  __device__ __forceinline__ void logits_tile(const uint8_t* stage, int mt, int ntok, bool tail, float lmask,
                                              float (&lg)[4], const QuantState& st) {
    const int r = lane >> 2;
    float la, lb;
    tile_logits(stage, mt, st, la, lb);
    const int ta = 16 * mt + r;
    float ma = lmask, mb = lmask;
    if (tail) {
      ma = ta < ntok ? lmask : -INFINITY;
      mb = ta + 8 < ntok ? lmask : -INFINITY;
    }
    la += ma;
    lb += mb;
    lg[2 * mt] = la;      // token 16mt + r
    lg[2 * mt + 1] = lb;  // token 16mt + r + 8
  }

  // P.V of the stage's 32 tokens (two 16-token k-steps).
  // * B column n < 4 carries the high fp16 part of head n's weights and column n + 4 the low part,
  //   so p (and p * scale) enter with ~22 significant bits: the code term and the zero-point term
  //   see the same weights, and their large opposite contributions (zero ~ group minimum) cancel
  //   without the fp16 rounding of p showing through.
  // * The tensor-core accumulator is used only within the stage, starting from zero; the running
  //   sums over the unit are kept with round-to-nearest fp32 adds.  A unit can span tens of
  //   thousands of tokens, and the mma adder's own rounding must not build up a drift in those
  //   large, mutually cancelling sums.
  __device__ __forceinline__ void pv_stage(const uint8_t* stage, bool colok, bool lo, const __half* pcol,
                                           QuantState& st) {
    const int r = lane >> 2, i = lane & 3;
    const uint8_t* vmain = stage + OFF_VMAIN;
    const __half* vscale = reinterpret_cast<const __half*>(stage + OFF_VMETA);
    const __half* vzero = vscale + 4 * HALF;

    // p_hi = fp16(p) and p_lo = fp16(p - p_hi) of this lane's column head, tokens (t0, t0+1), (t0+8, t0+9)
    uint32_t pA[2], pB[2], plA[2], plB[2];
    uint4 vab[2], vcd[2];
    float zt[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int t0 = 16 * mt + 2 * i;
      // a missing head's weights are written as zeros by the softmax (its logits are -inf)
      pA[mt] = *reinterpret_cast<const uint32_t*>(pcol + t0);
      pB[mt] = *reinterpret_cast<const uint32_t*>(pcol + t0 + 8);
      plA[mt] = (colok && lo) ? *reinterpret_cast<const uint32_t*>(pcol + MAX_GQA * HALF + t0) : 0u;
      plB[mt] = (colok && lo) ? *reinterpret_cast<const uint32_t*>(pcol + MAX_GQA * HALF + t0 + 8) : 0u;
      // zero-point term: rows = groups r (< 4), k = tokens: A = zero, B = p_hi | p_lo
      uint32_t zA = 0u, zB = 0u;
      if (r < 4) {
        zA = *reinterpret_cast<const uint32_t*>(vzero + r * HALF + t0);
        zB = *reinterpret_cast<const uint32_t*>(vzero + r * HALF + t0 + 8);
      }
      mma16816(zt, zA, 0u, zB, 0u, lo ? plA[mt] : pA[mt], lo ? plB[mt] : pB[mt]);
      // V codes of tokens (t0, t0+1) and (t0+8, t0+9) for channel row r: one 16-byte block per
      // token pair, word G = [t0 byte0, t1 byte0, t0 byte1, t1 byte1] of group G's channels 32G+4r..+3
      const int p0 = 8 * mt + i;
      const int blk = 16 * ((r + 2 * (p0 & 3)) & 7);
      vab[mt] = *reinterpret_cast<const uint4*>(vmain + p0 * 128 + blk);
      vcd[mt] = *reinterpret_cast<const uint4*>(vmain + (p0 + 4) * 128 + blk);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) st.zacc[e] = __fadd_rn(st.zacc[e], zt[e]);
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int t0 = 16 * mt + 2 * i;
        // B operand for group G: p * scale.  High column: fp16(p_hi s); low column:
        // fp16(p_lo s + (p_hi s - fp16(p_hi s))), the inner residual being exact.  px = p_hi in
        // low columns and 0 in high ones; p_lo = 0 in high ones.
        const uint32_t sA = *reinterpret_cast<const uint32_t*>(vscale + G * HALF + t0);
        const uint32_t sB = *reinterpret_cast<const uint32_t*>(vscale + G * HALF + t0 + 8);
        const uint32_t pxA = lo ? pA[mt] : 0u, pxB = lo ? pB[mt] : 0u;
        const uint32_t bA = h2u(__hfma2(u2h(plA[mt]), u2h(sA),
                                        __hfma2(u2h(pA[mt]), u2h(sA), __hneg2(__hmul2(u2h(pxA), u2h(sA))))));
        const uint32_t bB = h2u(__hfma2(u2h(plB[mt]), u2h(sB),
                                        __hfma2(u2h(pB[mt]), u2h(sB), __hneg2(__hmul2(u2h(pxB), u2h(sB))))));
        const uint4 va = vab[mt], vc = vcd[mt];
        const uint32_t wab = G == 0 ? va.x : G == 1 ? va.y : G == 2 ? va.z : va.w;
        const uint32_t wcd = G == 0 ? vc.x : G == 1 ? vc.y : G == 2 ? vc.z : vc.w;
        uint32_t x0, x2, x1, x3, y0, y2, y1, y3;
        cvt8(wab, x0, x2, x1, x3);  // channel 32G + 4r + {0, 2, 1, 3}, tokens (t0, t0 + 1)
        cvt8(wcd, y0, y2, y1, y3);  // same channels, tokens (t0 + 8, t0 + 9)
        mma16816(c0, x0, x1, y0, y1, bA, bB);
        mma16816(c1, x2, x3, y2, y3, bA, bB);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        st.acc[2 * G][e] = __fadd_rn(st.acc[2 * G][e], c0[e]);
        st.acc[2 * G + 1][e] = __fadd_rn(st.acc[2 * G + 1][e], c1[e]);
      }
    }
  }

  __device__ void quant_step(uint8_t* stage, int ntok, QuantState& st) {
    const int r = lane >> 2, i = lane & 3;
    __half* pw = reinterpret_cast<__half*>(smem + SM_P) + warp * 2 * MAX_GQA * HALF;
    const float lmask = (i < g) ? 0.f : -INFINITY;  // column pair of a missing head: never attended
    const bool tail = ntok < HALF;
    if (tail) sanitize_tail(stage, ntok);

    // ---- logits of the 32 tokens (two 16-token m-tiles)
    float lg[4];  // head i, tokens r, r + 8, r + 16, r + 24
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) logits_tile(stage, mt, ntok, tail, lmask, lg, st);

    // ---- online softmax for head i (rows r = 0..7 share it) with a lazily raised reference: the
    // weights are p = 2^(l - m) for the warp's reference m, which is raised (and the accumulators
    // rescaled) only when a logit exceeds it by more than 2^4; otherwise p <= 16 and no cross-lane
    // max is needed.  Any reference gives the same acc / l; 2^(-inf - m) = 0 handles masked tokens,
    // and a head with nothing valid yet keeps m = -inf (reference 0).
    const float lmax = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
    if (__any_sync(FULL, lmax > st.m + LAZY_RAISE)) {
      float mx = lmax;
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
      const float mnew = fmaxf(st.m, mx);
      const float alpha = (mnew == -INFINITY) ? 1.f : ex2(st.m - mnew);
      st.m = mnew;
      st.l *= alpha;
      // accumulator columns 2i, 2i+1 are heads (2i) & 3, (2i+1) & 3: their alpha lives in lanes
      // (r, (2i) & 3), (r, (2i+1) & 3)
      const float al0 = __shfl_sync(FULL, alpha, (lane & ~3) | ((2 * i) & 3));
      const float al1 = __shfl_sync(FULL, alpha, (lane & ~3) | ((2 * i + 1) & 3));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        st.acc[j][0] *= al0;
        st.acc[j][1] *= al1;
        st.acc[j][2] *= al0;
        st.acc[j][3] *= al1;
      }
      st.zacc[0] *= al0;
      st.zacc[1] *= al1;
      st.zacc[2] *= al0;
      st.zacc[3] *= al1;
    }
    const float mref = (st.m == -INFINITY) ? 0.f : st.m;
    float psum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = 8 * k + r;  // tokens r, r+8, r+16, r+24
      const float pv = ex2(lg[k] - mref);
      psum += pv;
      const __half ph = __float2half_rn(pv);
      pw[i * HALF + t] = ph;
      pw[MAX_GQA * HALF + i * HALF + t] = __float2half_rn(pv - __half2float(ph));
    }
    st.l += psum;
    __syncwarp();

    // ---- P.V: k-step = 16 tokens; this thread's B column is head r & 3 (high part for r < 4, low part
    // for r >= 4), tokens t0, t0+1, +8, +9
    const bool colok = (r & 3) < g, lo = r >= 4;
    const __half* pcol = pw + (r & 3) * HALF;
    pv_stage(stage, colok, lo, pcol, st);
    __syncwarp();
  }

  // ---------------------------------------------------------------- records
  __device__ __forceinline__ float* record(int u, int gw) const { return record_at(a, u, gw); }

  __device__ void write_quant(float* rec, QuantState& st) {
    const int r = lane >> 2, i = lane & 3;
    // undo the 2^-9 of the converted codes and fold in the zero-point term:
    // acc[h][c] = 512 * acc[h][c] + zterm[G(c)][h]
#pragma unroll
    for (int G = 0; G < 4; ++G) {
      const float z0 = __shfl_sync(FULL, st.zacc[0], 4 * G + i);
      const float z1 = __shfl_sync(FULL, st.zacc[1], 4 * G + i);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        st.acc[2 * G + e][0] = st.acc[2 * G + e][0] * CODE_UNSCALE + z0;
        st.acc[2 * G + e][1] = st.acc[2 * G + e][1] * CODE_UNSCALE + z1;
        st.acc[2 * G + e][2] = st.acc[2 * G + e][2] * CODE_UNSCALE + z0;
        st.acc[2 * G + e][3] = st.acc[2 * G + e][3] * CODE_UNSCALE + z1;
      }
    }
    // add the low-part columns 4..7 (lanes i = 2, 3) to the high-part columns 0..3 (lanes i = 0, 1)
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) st.acc[j][e] += __shfl_xor_sync(FULL, st.acc[j][e], 2);
    float l = st.l;
    l += __shfl_xor_sync(FULL, l, 4);
    l += __shfl_xor_sync(FULL, l, 8);
    l += __shfl_xor_sync(FULL, l, 16);
    // heads 2i, 2i+1 in columns; channel of m-tile 2G+e row r is 32G + 4r + 2e, row r+8 adds 1
    const float l0 = __shfl_sync(FULL, l, 0), l1 = __shfl_sync(FULL, l, 1);
    const float l2 = __shfl_sync(FULL, l, 2), l3 = __shfl_sync(FULL, l, 3);
    const bool anyl = l0 > 0.f || l1 > 0.f || l2 > 0.f || l3 > 0.f;
    if (anyl) {
#pragma unroll
      for (int cidx = 0; cidx < 2; ++cidx) {
        const int hh = 2 * i + cidx;
        if (hh < g) {
          float* dst = rec + 16 + hh * D;
#pragma unroll
          for (int G = 0; G < 4; ++G)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c0 = 32 * G + 4 * r + 2 * e;
              dst[c0] = st.acc[2 * G + e][cidx];
              dst[c0 + 1] = st.acc[2 * G + e][2 + cidx];
            }
        }
      }
    }
    st.l = l;  // every lane with head i now has the full sum
  }

  // header: [Qm[4], Ql[4], Wm[4], Wl[4]]
  __device__ void write_header(float* rec, bool hasq, const QuantState& st, bool hasw, const WinState& ws) {
    const int k = lane & 3;
    const float qm = __shfl_sync(FULL, st.m, k);
    const float ql = __shfl_sync(FULL, st.l, k);
    float v;
    if (lane < 4) v = hasq ? qm : -INFINITY;
    else if (lane < 8) v = hasq ? ql : 0.f;
    else if (lane < 12) v = hasw ? ws.ml[k] : -INFINITY;
    else v = hasw ? ws.ml[4 + k] : 0.f;
    if (lane < 16) rec[lane] = v;
  }

  // window accumulator of this warp's part of unit u into its record
  __device__ __forceinline__ void store_window_acc(int u, int gw, const QuantState& st) {
    float* dst = record(u, gw) + 16 + MAX_GQA * D + 4 * lane;
#pragma unroll
    for (int k = 0; k < MAX_GQA; ++k)
      *reinterpret_cast<float4*>(dst + k * D) = make_float4(st.acc[k][0], st.acc[k][1], st.acc[k][2], st.acc[k][3]);
  }

  // Write this warp's record of unit u (read by the merge kernel once this grid has ended).
  __device__ void finish_unit(int u, int gw, int kind, bool hasq, bool hasw, QuantState& st, WinState& ws) {
    float* rec = record(u, gw);
    if (kind == KIND_QUANT) write_quant(rec, st);
    else store_window_acc(u, gw, st);
    write_header(rec, hasq, st, hasw, ws);
  }

};

// Combine the partial records of query head hh of unit u (records cf .. cf + nrec - 1, one per
// warp that streamed part of the unit) in record order and write the head's output.  Latency-bound:
// a round trip to records just written by other SMs took ~2 us (measured inside the merge), so
// the reads are issued together: after the unit's record range, one round trip per CHUNK records
// brings their (m, l) entries (lane j: record j), this lane's channels of their quantised parts
// and, speculatively, of the window parts of the unit's first MERGE_WIN_SPEC records (a unit's
// window chunks are its first steps, so the records holding a window part are a prefix of its
// records).  Records without a part for this head (weight 0) are skipped, whatever their stale
// contents; a window part further on (a warp range shorter than the window) costs one more round
// trip.  A unit without records (empty sequence) gets zeros.
constexpr int MERGE_CHUNK = 16;       // records per round trip of merge_kernel (one warp per head)
constexpr int WIDE_MERGE_CHUNK = 20;  // of merge_wide_kernel's quantised-part warps
constexpr int MERGE_WIN_SPEC = 4;     // leading records whose window part is read speculatively

// Merge records cf + r0 .. cf + r1 - 1 of unit u, query head hh, into the running state of the
// parts selected (QUANT: 0 = quantised, rotated space; WIN: 1 = window): maxima Mk, sums Lk and this
// lane's channels 4 lane .. +3 of the accumulators O, in record order.  A window-only merge stops
// at the first chunk without a window part.
template <int CHUNK, bool QUANT, bool WIN>
__device__ __forceinline__ void merge_records(const DecodeArgs& a, int u, int hh, int lane, int cf, int r0, int r1,
                                              float4 (&O)[2], float (&Mk)[2], float (&Lk)[2]) {
  static_assert(CHUNK <= 32, "one lane per record header");
  for (int base = r0; base < r1; base += CHUNK) {
    const int cnt = min(CHUNK, r1 - base);
    // head hh's (m, l) of the selected parts of record base + lane: header [Qm[4], Ql[4], Wm[4], Wl[4]]
    float hd[4] = {-INFINITY, 0.f, -INFINITY, 0.f};
    if (lane < cnt) {
      const float* hp = record_at(a, u, cf + base + lane);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < 2 ? QUANT : WIN) hd[i] = __ldcg(hp + 4 * i + hh);
    }
    float4 xq[QUANT ? CHUNK : 1], xw[WIN ? MERGE_WIN_SPEC : 1];
    if (QUANT) {
#pragma unroll
      for (int r = 0; r < CHUNK; ++r) {
        const float* rec = record_at(a, u, cf + base + r) + 16 + hh * D + 4 * lane;
        xq[r] = r < cnt ? __ldcg(reinterpret_cast<const float4*>(rec)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (WIN) {
#pragma unroll
      for (int r = 0; r < MERGE_WIN_SPEC; ++r) {
        const float* rec = record_at(a, u, cf + base + r) + 16 + (MAX_GQA + hh) * D + 4 * lane;
        xw[r] = (base + r < MERGE_WIN_SPEC && r < cnt) ? __ldcg(reinterpret_cast<const float4*>(rec))
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float f[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // 0 = quantised part (rotated space), 1 = window part
      if (!(k == 0 ? QUANT : WIN)) continue;
      const float mv = hd[2 * k], lv = hd[2 * k + 1];
      float m = lv > 0.f ? mv : -INFINITY;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      const float mn = fmaxf(Mk[k], m);
      const float sc = (Mk[k] == -INFINITY) ? 0.f : exp2f(Mk[k] - mn);  // rescale earlier chunks
      Lk[k] *= sc;
      O[k] = make_float4(O[k].x * sc, O[k].y * sc, O[k].z * sc, O[k].w * sc);
      Mk[k] = mn;
      f[k] = lv > 0.f ? exp2f(mv - mn) : 0.f;
      float lw = lv * f[k];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) lw += __shfl_xor_sync(FULL, lw, o);
      Lk[k] += lw;
    }
    if (QUANT) {
#pragma unroll
      for (int r = 0; r < CHUNK; ++r) {
        const float fr = __shfl_sync(FULL, f[0], r);
        if (fr > 0.f) {
          O[0].x += fr * xq[r].x;
          O[0].y += fr * xq[r].y;
          O[0].z += fr * xq[r].z;
          O[0].w += fr * xq[r].w;
        }
      }
    }
    if (WIN) {
#pragma unroll
      for (int r = 0; r < MERGE_WIN_SPEC; ++r) {
        const float fr = __shfl_sync(FULL, f[1], r);
        if (base + r < MERGE_WIN_SPEC && fr > 0.f) {
          O[1].x += fr * xw[r].x;
          O[1].y += fr * xw[r].y;
          O[1].z += fr * xw[r].z;
          O[1].w += fr * xw[r].w;
        }
      }
      // window parts beyond the speculatively read records, in record order
      unsigned todo = __ballot_sync(FULL, f[1] > 0.f && base + lane >= MERGE_WIN_SPEC);
      while (todo) {
        const int j = __ffs(todo) - 1;
        todo &= todo - 1;
        const float fr = __shfl_sync(FULL, f[1], j);
        const float4 x = __ldcg(reinterpret_cast<const float4*>(record_at(a, u, cf + base + j) + 16 +
                                                                 (MAX_GQA + hh) * D + 4 * lane));
        O[1].x += fr * x.x;
        O[1].y += fr * x.y;
        O[1].z += fr * x.z;
        O[1].w += fr * x.w;
      }
      // the records with a window part are a prefix: done once the chunk's last record has none
      if (!QUANT && !(__shfl_sync(FULL, hd[3], cnt - 1) > 0.f)) break;
    }
  }
}

// This lane's channels of the rotation signs and of the unit's V balancing scales (ones without
// Sinkhorn), for the output phase: requested early, while the records are read.
__device__ __forceinline__ void merge_constants(const DecodeArgs& a, int u, int lane, float4& sg, float4& sv) {
  const int H = a.Hkv, B = a.batch;
  const int h = u % H, ll = u / (H * B);
  sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
  sv = make_float4(1.f, 1.f, 1.f, 1.f);
  if (a.sinkhorn) {
    const __half2* sig = reinterpret_cast<const __half2*>(a.p.sigv + ((size_t)(a.layer0 + ll) * H + h) * D + 4 * lane);
    const float2 s01 = __half22float2(sig[0]), s23 = __half22float2(sig[1]);
    sv = make_float4(s01.x, s01.y, s23.x, s23.y);
  }
}

// The head's output from the merged state: undo the balancing scale and the rotation of the
// quantised part, combine it with the window part, divide by the sum.
__device__ __forceinline__ void merge_output(const DecodeArgs& a, int u, int hh, int lane, const float4 (&O)[2],
                                             const float (&Mk)[2], const float (&Lk)[2], float4 sg, float4 sv) {
  const int H = a.Hkv, B = a.batch, g = a.g;
  const int h = u % H, b = (u / H) % B, ll = u / (H * B);
  float q0 = O[0].x, q1 = O[0].y, q2 = O[0].z, q3 = O[0].w;
  const bool hq = Lk[0] > 0.f, hw = Lk[1] > 0.f;
  if (hq) {
    // undo the balancing scale and the rotation: v = s . (c H (sigma . y))
    q0 *= sv.x;
    q1 *= sv.y;
    q2 *= sv.z;
    q3 *= sv.w;
    hadamard_warp(q0, q1, q2, q3, lane);
    q0 *= C_WHT * sg.x;
    q1 *= C_WHT * sg.y;
    q2 *= C_WHT * sg.z;
    q3 *= C_WHT * sg.w;
  }
  const float Mt = fmaxf(hq ? Mk[0] : -INFINITY, hw ? Mk[1] : -INFINITY);
  const float f0 = hq ? exp2f(Mk[0] - Mt) : 0.f;
  const float f1 = hw ? exp2f(Mk[1] - Mt) : 0.f;
  const float den = Lk[0] * f0 + Lk[1] * f1;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float4 o;
  o.x = (q0 * f0 + O[1].x * f1) * inv;
  o.y = (q1 * f0 + O[1].y * f1) * inv;
  o.z = (q2 * f0 + O[1].z * f1) * inv;
  o.w = (q3 * f0 + O[1].w * f1) * inv;
  *reinterpret_cast<float4*>(a.out + (((size_t)ll * B + b) * H * g + (size_t)h * g + hh) * D + 4 * lane) = o;
}


// The merge of query head hh of unit u by one warp: its record range, then its records (above).
__device__ void merge_head(const DecodeArgs& a, int u, int hh, int lane) {
  const int2 info = __ldcg(a.unit_info + u);
  float4 sg, sv;
  merge_constants(a, u, lane, sg, sv);
  float4 O[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float Mk[2] = {-INFINITY, -INFINITY}, Lk[2] = {0.f, 0.f};
  merge_records<MERGE_CHUNK, true, true>(a, u, hh, lane, info.x, 0, info.y, O, Mk, Lk);
  merge_output(a, u, hh, lane, O, Mk, Lk, sg, sv);
}

// One warp per (unit, query head).  Launched as a programmatic dependent of decode_kernel; waits
// for the whole grid (its records and record ranges) before reading anything.
__global__ void __launch_bounds__(MERGE_WARPS * 32) merge_kernel(const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // a following decode launched as a programmatic dependent (the next layer's call) may run its
  // set-up now: it writes nothing outside shared memory before its own wait for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long t = (long long)blockIdx.x * MERGE_WARPS + (threadIdx.x >> 5);
  if (t >= (long long)a.n_units * a.g) return;
  merge_head(a, (int)(t / a.g), (int)(t % a.g), lane);
}

// Calls whose units have many records each (a single layer's decode spread over every warp of
// the GPU: hundreds of records per unit): one CTA per (unit, query head), its warps merging
// consecutive slices of the records' quantised parts in parallel (up to WIDE_MERGE_CHUNK records
// each in one round trip) and the last warp the window parts (a prefix of the records); the first
// warp then combines the warps' states in warp order (a fixed order: deterministic; lane j holds
// warp j's maximum and sum, so the weights take one exponential per lane) and writes the output.
__global__ void __launch_bounds__(WIDE_MERGE_WARPS * 32) merge_wide_kernel(const __grid_constant__ DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float4 sO[WIDE_MERGE_WARPS][2][32];
  __shared__ float sM[WIDE_MERGE_WARPS][2], sL[WIDE_MERGE_WARPS][2];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int u = blockIdx.x / a.g, hh = blockIdx.x % a.g;
  const int2 info = __ldcg(a.unit_info + u);
  float4 sg, sv;
  if (w == 0) merge_constants(a, u, lane, sg, sv);
  float4 O[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float Mk[2] = {-INFINITY, -INFINITY}, Lk[2] = {0.f, 0.f};
  constexpr int NQW = WIDE_MERGE_WARPS - 1;  // warps on the quantised parts
  if (w < NQW) {
    const int per = (info.y + NQW - 1) / NQW;
    const int r0 = min(info.y, w * per), r1 = min(info.y, r0 + per);
    merge_records<WIDE_MERGE_CHUNK, true, false>(a, u, hh, lane, info.x, r0, r1, O, Mk, Lk);
  } else {
    merge_records<MERGE_CHUNK, false, true>(a, u, hh, lane, info.x, 0, info.y, O, Mk, Lk);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    sO[w][k][lane] = O[k];
    if (lane == 0) {
      sM[w][k] = Mk[k];
      sL[w][k] = Lk[k];
    }
  }
  __syncthreads();
  if (w != 0) return;
  static_assert(WIDE_MERGE_WARPS <= 32, "one lane per slice");
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float lj = lane < WIDE_MERGE_WARPS ? sL[lane][k] : 0.f;
    const float mj = lj > 0.f ? sM[lane][k] : -INFINITY;
    float M = mj;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    const float fj = lj > 0.f ? exp2f(mj - M) : 0.f;
    float L = lj * fj;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(FULL, L, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < WIDE_MERGE_WARPS; ++j) {
      const float f = __shfl_sync(FULL, fj, j);
      if (f > 0.f) {
        const float4 x = sO[j][k][lane];
        acc.x += f * x.x;
        acc.y += f * x.y;
        acc.z += f * x.z;
        acc.w += f * x.w;
      }
    }
    O[k] = acc;
    Mk[k] = M;
    Lk[k] = L;
  }
  merge_output(a, u, hh, lane, O, Mk, Lk, sg, sv);
}

template <int KF>
__global__ void __launch_bounds__(Geo<KF>::NTHREADS, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
  using GE = Geo<KF>;
  constexpr int NCW = GE::NCW, NSTAGE = GE::NSTAGE, NTHREADS = GE::NTHREADS;
  extern __shared__ __align__(1024) uint8_t smem[];
  Kernel<KF> K(a, smem);
  const int tid = threadIdx.x;
  K.warp = tid >> 5;
  K.lane = tid & 31;
  K.lut_base_known = smem_addr(smem) == DYN_SMEM_WINDOW_BASE;
  K.B = a.batch;
  K.H = a.Hkv;
  K.W = a.W;
  K.g = a.g;
  K.Hq = a.Hkv * a.g;
  const int B = a.batch, H = a.Hkv, W = a.W;
  int* sS = reinterpret_cast<int*>(smem + GE::SM_SEQ);
  int* sPre = sS + (B + 1);
  int* sL = sPre + (B + 1);
  int* sNW = sL + (B + 1);
  int* sC = sNW + (B + 1);
  int* sCpre = sC + (B + 1);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + GE::SM_BARS);
  uint64_t* empty = full + NSTAGE;
  int4* desc = reinterpret_cast<int4*>(smem + GE::SM_DESC);
  int4* sWpos = reinterpret_cast<int4*>(smem + GE::SM_WPOS);
  long long* sWxs = reinterpret_cast<long long*>(smem + GE::SM_WPOS + (NCW + 1) * 16);
  K.sq.S = sS;
  K.sq.pre = sPre;
  K.sq.L = sL;
  K.sq.NW = sNW;
  K.sq.C = sC;
  K.sq.cpre = sCpre;
  // Launched as a programmatic dependent: the previous kernel of the stream may still be running
  // and writing the inputs (the cache, q, the lengths).  Q4G32 and Q8G32 keys: the split of the
  // work is computed before waiting for it, from the lengths as they stand (read through L2, never
  // cached in L1); after the wait the lengths are read again and the split recomputed if any
  // changed.  Nothing else of the inputs is read, and nothing is written outside shared memory,
  // before the wait.  TQ3 keys wait first: with the early split their consumers' code came out
  // 0.4-0.8 % slower (measured), more than the split saves on an all-layer call.  (No early
  // trigger for the merge kernel: its CTAs, resident early, slowed the streaming warps.)
  if constexpr (KF == KVQ_TQ3_QJL) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the TQ3 decode table (2 KB in the cache header) is read once per CTA into the first stage,
    // and expanded to its per-lane copies after the barrier below (the stages are idle until then)
    if (tid < 256) reinterpret_cast<uint2*>(smem + GE::SM_STAGES)[tid] = a.p.cb->lut8[tid];
    for (int b = tid; b < B; b += NTHREADS) {
      int L = a.seq_lens[b];
      if (L < 0 || L > a.max_seq_len) {
        if (blockIdx.x == 0) atomicOr(a.p.status, KVQ_DEV_SEQLEN_RANGE);
        L = 0;
      }
      seq_steps<KF>(b, L, W, sL, sNW, sS, sC);
    }
    __syncthreads();
    if (K.warp == 0) seq_prefix(K.lane, B, sS, sC, sPre, sCpre);
    if (tid >= 32 && tid < 32 + 2 * NSTAGE) {
      // one barrier per thread of warps 1-2 (full[NSTAGE] then empty[NSTAGE], contiguous)
      mbar_init(full + (tid - 32), 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    {
      // entry v: 32 lane copies of its centroid pair, then 32 lane copies of its sign pair
      const uint32_t* src = reinterpret_cast<const uint32_t*>(smem + GE::SM_STAGES);
      uint32_t* lut = reinterpret_cast<uint32_t*>(smem + GE::SM_LUT);
      for (int idx = tid; idx < 256 * 64; idx += NTHREADS) lut[idx] = src[2 * (idx >> 6) + ((idx >> 5) & 1)];
    }
    __syncthreads();
    K.totals();
    if (K.S == 0 || (long long)blockIdx.x * NCW >= K.nw) {
      if (tid < NCW * 32) K.unit_info_share((long long)tid * gridDim.x + blockIdx.x);
      return;
    }
    K.locate(sWpos, sWxs);
  } else {
    if (tid >= 32 && tid < 32 + 2 * NSTAGE) {
      mbar_init(full + (tid - 32), 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // pass 0 (before the wait) computes the split silently; pass 1 (after it) reads the lengths
    // again, reports bad ones, and recomputes the split only if one changed
    for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) asm volatile("griddepcontrol.wait;" ::: "memory");
      bool changed = false;
      for (int b = tid; b < B; b += NTHREADS) {
        int L = __ldcg(a.seq_lens + b);
        if (L < 0 || L > a.max_seq_len) {
          if (pass == 1 && blockIdx.x == 0) atomicOr(a.p.status, KVQ_DEV_SEQLEN_RANGE);
          L = 0;
        }
        if (pass == 0 || L != sL[b]) {
          changed = true;
          seq_steps<KF>(b, L, W, sL, sNW, sS, sC);
        }
      }
      if (!__syncthreads_or(changed)) continue;
      if (K.warp == 0) seq_prefix(K.lane, B, sS, sC, sPre, sCpre);
      __syncthreads();
      K.totals();
      if (K.S > 0 && (long long)blockIdx.x * NCW < K.nw) K.locate(sWpos, sWxs);
    }
  }
  __syncthreads();
  // the record ranges of all units, for the merge kernel: a share per consumer thread of the grid,
  // computed by warps with steps once their first copies are in flight
  const long long info_i = (long long)tid * gridDim.x + blockIdx.x;
  if (K.S == 0 || (long long)blockIdx.x * NCW >= K.nw) {
    if (tid < NCW * 32) K.unit_info_share(info_i);
    return;
  }

  if (K.warp == NCW) {
    // ======================= producer: lane w streams consumer warp w's contiguous step range.
    // The lanes poll their next stage without blocking and start, in the same pass, every copy
    // whose stage has been released, so the warp stays converged; a pass that starts nothing
    // sleeps briefly, and ~1 s without any progress ends the stream with a status bit.
    const int w = K.lane;
    const long long gw = (long long)blockIdx.x * NCW + w;
    int n = 0;
    Pos ps = {0, 0, 0, 0};
    if (w < NCW && gw < K.nw) {
      const int4 p = sWpos[w];
      ps = {p.x, p.y, p.z, p.w};
      n = (int)(sWxs[w + 1] - sWxs[w]);
    }
    int bt_page = -1, bt_phys = 0;  // the last block-table entry read by this lane
    constexpr int NS = GE::NSLOT;
    int k = 0;
    unsigned long long t_idle = 0;
    while (__any_sync(FULL, k < n)) {
      const int slot = w + NCW * (k % NS);
      const bool ready = k < n && (k < NS || mbar_test(empty + slot, ((k / NS) - 1) & 1));
      if (ready) {
        const int u = (ps.ll * B + ps.b) * H + ps.h;
        const int layer = a.layer0 + ps.ll;
        const int L = sL[ps.b];
        const int nwin = W > 0 ? (min(L, W) + WCHUNK - 1) / WCHUNK : 0;
        uint8_t* dst = smem + GE::SM_STAGES + slot * GE::STAGE;
        if (ps.local < nwin) {
          const int s0 = ps.local * WCHUNK;
          const int ntok = min(WCHUNK, min(L, W) - s0);
          desc[slot] = make_int4(u, KIND_WINDOW, ntok, ps.local);
          const size_t ro = ((((size_t)layer * a.max_batch + ps.b) * H + ps.h) * W + s0) * D;
          mbar_arrive_tx(full + slot, 2 * WCHUNK * D * 4);
          bulk_g2s(dst, a.p.ringk + ro, WCHUNK * D * 4, full + slot);
          bulk_g2s(dst + WCHUNK * D * 4, a.p.ringv + ro, WCHUNK * D * 4, full + slot);
        } else {
          const int hp = ps.local - nwin;  // half-page index within the sequence
          const int Lq = W > 0 ? max(0, L - W) : L;
          const int ntok = min(HALF, Lq - hp * HALF);
          const int page = ps.b * a.max_pages_per_seq + (hp >> 1);
          if (page != bt_page) {
            // the cache's own table is the identity: no read
            bt_phys = a.identity_pages ? page : a.block_table[page];
            bt_page = page;
          }
          const int phys = bt_phys;
          if (phys < 0 || phys >= a.L.n_pages) {
            atomicOr(a.p.status, KVQ_DEV_BAD_PAGE);
            desc[slot] = make_int4(u, KIND_QUANT, 0, ps.local);
            mbar_arrive(full + slot);
          } else {
            desc[slot] = make_int4(u, KIND_QUANT, ntok, ps.local);
            const uint8_t* src = a.p.pages +
                                 (((size_t)layer * a.L.n_pages + phys) * H + ps.h) * (size_t)a.L.page_bytes +
                                 (size_t)(hp & 1) * a.L.half_bytes;
            mbar_arrive_tx(full + slot, a.L.half_bytes);
            bulk_g2s(dst, src, a.L.half_bytes, full + slot);
          }
        }
        if (++k < n) advance(ps, 1, B, H, K.sq);
      }
      if (__any_sync(FULL, ready)) {
        t_idle = 0;
      } else {
        const unsigned long long now = globaltimer();
        if (t_idle == 0) t_idle = now;
        if (__any_sync(FULL, now - t_idle > a.wait_ns)) {
          if (w == 0) atomicOr(a.p.status, KVQ_DEV_TIMEOUT);
          break;
        }
        __nanosleep(64);
      }
    }
    // never leave the CTA with a copy still landing in shared memory
    for (int kk = max(0, k - NS); kk < k; ++kk) mbar_wait(full + w + NCW * (kk % NS), (kk / NS) & 1, a.p.status);
    return;
  }

  // ======================= consumers: warp gw processes its steps (see first_step) in order
  const long long gw = (long long)blockIdx.x * NCW + K.warp;
  if (gw >= K.nw) {
    K.unit_info_share(info_i);
    return;
  }
  Pos p0;
  {
    const int4 p = sWpos[K.warp];
    p0 = {p.x, p.y, p.z, p.w};
  }
  const int n = (int)(sWxs[K.warp + 1] - sWxs[K.warp]);
  QuantState st;
  WinState ws;
  ws.q = reinterpret_cast<float*>(smem + GE::SM_Q) + K.warp * MAX_GQA * D;
  ws.ml = reinterpret_cast<float*>(smem + GE::SM_WML) + K.warp * 8;
  int cur = -1, kind = -1;
  bool hasq = false, hasw = false;
  {
    // set up the first unit while the pipeline fills
    const int L0 = sL[p0.b];
    const int nwin0 = W > 0 ? (min(L0, W) + WCHUNK - 1) / WCHUNK : 0;
    cur = (p0.ll * B + p0.b) * H + p0.h;
    kind = p0.local < nwin0 ? KIND_WINDOW : KIND_QUANT;
    if (kind == KIND_WINDOW) {
      hasw = true;
    } else {
      hasq = true;
    }
    K.load_q(cur, st, ws, kind);
  }
  K.unit_info_share(info_i);
  // step k uses slot warp + NCW*(k mod NSLOT), phase k / NSLOT of that slot
  for (int k = 0, j = 0, ph = 0; k < n; ++k) {
    const int slot = K.warp + NCW * j;
    if (!mbar_wait(full + slot, ph, a.p.status)) break;
    if (++j == GE::NSLOT) {
      j = 0;
      ph ^= 1;
    }
    const int4 d = desc[slot];
    if (d.x != cur) {
      float4 raw[MAX_GQA];
      K.fetch_q(d.x, raw);  // in flight while the previous unit's record is published
      K.finish_unit(cur, (int)gw, kind, hasq, hasw, st, ws);
      cur = d.x;
      kind = d.y;
      hasq = kind == KIND_QUANT;
      hasw = kind == KIND_WINDOW;
      K.build_q(cur, raw, st, ws, kind);
    } else if (d.y != kind) {
      if (kind == KIND_WINDOW) K.store_window_acc(cur, (int)gw, st);
      K.load_q(cur, st, ws, d.y);
      kind = d.y;
      if (kind == KIND_WINDOW) hasw = true;
      else hasq = true;
    }
    uint8_t* stage = smem + GE::SM_STAGES + slot * GE::STAGE;
    if (d.z > 0) {
      if (d.y == KIND_WINDOW) K.window_step(stage, d.z, ws, st);
      else K.quant_step(stage, d.z, st);
    }
    __syncwarp();
    if (K.lane == 0) mbar_arrive(empty + slot);
  }
  K.finish_unit(cur, (int)gw, kind, hasq, hasw, st, ws);
}

}  // namespace

int decode_consumer_warps(int k_format) {
  return k_format == KVQ_TQ3_QJL ? Geo<KVQ_TQ3_QJL>::NCW
         : k_format == KVQ_Q8G32 ? Geo<KVQ_Q8G32>::NCW
                                 : Geo<KVQ_Q4G32>::NCW;
}

size_t decode_scratch_bytes(int n_units, int n_ctas, int k_format) {
  // record ranges int2 [n_units], then the partial records (index unit + warp)
  return align256((size_t)n_units * sizeof(int2)) + decode_record_slots(n_units, n_ctas, k_format) * REC_FLOATS * sizeof(float);
}

size_t decode_record_slots(int n_units, int n_ctas, int k_format) {
  return (size_t)n_units + (size_t)n_ctas * decode_consumer_warps(k_format);
}

// largest dynamic shared-memory size granted so far to decode_kernel<KF>, per device: the attribute
// is set again only when a call needs more (no host call per launch, none during stream capture
// once a call of the same or a larger batch has run)
constexpr int MAX_DEVICES = 64;
template <int KF>
std::atomic<int> g_smem_granted[MAX_DEVICES];

template <int KF>
static cudaError_t launch_kf(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = Geo<KF>::SM_SEQ + 6 * (size_t)(a.batch + 1) * sizeof(int);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES || g_smem_granted<KF>[dev].load() < (int)smem) {
    e = cudaFuncSetAttribute(decode_kernel<KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < MAX_DEVICES) {
      int cur = g_smem_granted<KF>[dev].load();
      while (cur < (int)smem && !g_smem_granted<KF>[dev].compare_exchange_weak(cur, (int)smem)) {
      }
    }
  }
  // programmatic dependent launch: the CTAs may be launched while the previous kernel of the
  // stream (typically the append of the step's new tokens) is finishing; each waits for it
  // (griddepcontrol.wait) before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_ctas);
  cfg.blockDim = dim3(Geo<KF>::NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_kernel<KF>, a);
  if (e != cudaSuccess) return e;
  // the merge, as a programmatic dependent of the decode grid: one warp per (unit, query head), or
  // one CTA per (unit, query head) when the units are few and each holds many records (at most
  // about consumer warps / units of them)
  const long long tasks = (long long)a.n_units * a.g;
  const long long recs_per_unit = (long long)a.n_ctas * Geo<KF>::NCW / a.n_units + 2;
  cudaLaunchConfig_t mcfg = cfg;
  mcfg.blockDim = dim3(MERGE_WARPS * 32);
  mcfg.dynamicSmemBytes = 0;
  if (recs_per_unit > WIDE_MERGE_RECORDS) {
    mcfg.gridDim = dim3((unsigned)tasks);
    mcfg.blockDim = dim3(WIDE_MERGE_WARPS * 32);
    return cudaLaunchKernelEx(&mcfg, merge_wide_kernel, a);
  }
  mcfg.gridDim = dim3((unsigned)((tasks + MERGE_WARPS - 1) / MERGE_WARPS));
  return cudaLaunchKernelEx(&mcfg, merge_kernel, a);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  return a.k_format == KVQ_TQ3_QJL ? launch_kf<KVQ_TQ3_QJL>(a, s)
         : a.k_format == KVQ_Q8G32 ? launch_kf<KVQ_Q8G32>(a, s)
                                   : launch_kf<KVQ_Q4G32>(a, s);
}

}  // namespace kvq
