// KVarN calibration kernel: Sinkhorn variance balancing of a rotated calibration block.
//
// [KV] TLDR: Walsh-Hadamard transform, then Sinkhorn variance balancing, before 4-bit.  Reading
// of the unstated details (float32, fixed order): 8 iterations of
//   row step     rho_i   = sqrt(sumsq(X_i) / 128)   (per-lane blocks of 4, then a lane-halving
//                tree), X_i /= rho_i when rho_i > 0;
//   column step  kappa_j = sqrt(S_j / n) with S_j summed over tokens 0..n-1 in order,
//                X_.j /= kappa_j when kappa_j > 0, sigma_j *= kappa_j;
// then sigma_j is stored as fp16.  The append kernel divides the rotated vector by sigma.
//
// One CTA of 1024 threads per (layer, kv-head, K|V); the float working copy of the block lives in
// the caller's scratch buffer (it does not fit in shared memory for 1024 tokens).
#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int THREADS = 1024;
constexpr int ITERS = 8;

__global__ void __launch_bounds__(THREADS, 1) calibrate_kernel(const CalibArgs a) {
  __shared__ float sigma[D];
  __shared__ float kappa[D];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kv = blockIdx.x & 1;
  const int unit = blockIdx.x >> 1;  // (layer_local, head)
  const int h = unit % a.Hkv, ll = unit / a.Hkv;
  const int layer = a.layer0 + ll;
  const int n = a.ntok;
  float* X = a.work + (size_t)blockIdx.x * n * D;
  const void* src = kv ? a.vc : a.kc;

  // rotate every row: y = c * H (s . x)
  const float4 sg = *reinterpret_cast<const float4*>(a.p.signs + 4 * lane);
  for (int row = warp; row < n; row += THREADS / 32) {
    const float4 x = load4_in(src, ((size_t)unit * n + row) * D + 4 * lane, a.in_bf16);
    float y0 = __fmul_rn(x.x, sg.x), y1 = __fmul_rn(x.y, sg.y);
    float y2 = __fmul_rn(x.z, sg.z), y3 = __fmul_rn(x.w, sg.w);
    hadamard_warp(y0, y1, y2, y3, lane);
    *reinterpret_cast<float4*>(X + (size_t)row * D + 4 * lane) =
        make_float4(__fmul_rn(y0, C_WHT), __fmul_rn(y1, C_WHT), __fmul_rn(y2, C_WHT), __fmul_rn(y3, C_WHT));
  }
  if (tid < D) sigma[tid] = 1.0f;
  __syncthreads();

  for (int it = 0; it < ITERS; ++it) {
    for (int row = warp; row < n; row += THREADS / 32) {
      float4* px = reinterpret_cast<float4*>(X + (size_t)row * D + 4 * lane);
      float4 x = *px;
      const float rho = __fsqrt_rn(__fdiv_rn(sumsq_warp(x.x, x.y, x.z, x.w), 128.0f));
      if (rho > 0.0f) {
        x.x = __fdiv_rn(x.x, rho);
        x.y = __fdiv_rn(x.y, rho);
        x.z = __fdiv_rn(x.z, rho);
        x.w = __fdiv_rn(x.w, rho);
        *px = x;
      }
    }
    __syncthreads();
    if (tid < D) {
      float s = 0.0f;
#pragma unroll 8
      for (int t = 0; t < n; ++t) {
        const float v = X[(size_t)t * D + tid];
        s = __fadd_rn(s, __fmul_rn(v, v));
      }
      float k = __fsqrt_rn(__fdiv_rn(s, (float)n));
      if (!(k > 0.0f)) k = 1.0f;
      kappa[tid] = k;
      sigma[tid] = __fmul_rn(sigma[tid], k);
    }
    __syncthreads();
    for (int idx = tid; idx < n * D; idx += THREADS) X[idx] = __fdiv_rn(X[idx], kappa[idx & (D - 1)]);
    __syncthreads();
  }
  if (tid < D) {
    __half* dst = (kv ? a.p.sigv : a.p.sigk) + ((size_t)layer * a.Hkv + h) * D;
    dst[tid] = __float2half_rn(sigma[tid]);
  }
}

}  // namespace

cudaError_t launch_calibrate(const CalibArgs& a, cudaStream_t s) {
  const int blocks = a.n_layers_call * a.Hkv * 2;
  calibrate_kernel<<<blocks, THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
