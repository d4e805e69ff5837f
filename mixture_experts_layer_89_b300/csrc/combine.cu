// Combine: y[t] = sum over kept slots j of w[t,j] * y_perm[row_of[t,j]]  (+ y_shared[t]).
//
// The layer output is the routing-weighted sum of the selected experts' outputs (FLAME-MoE
// summary, sec. 2; the accumulation of the mini-moe tutorial, sec. 3.1 MoELayer), plus the
// always-on shared experts.  A dropped slot (row -1) contributes nothing and the surviving
// weights are not renormalised (OpenMythos article, sec. 3.1, overflow handling).
//
// The expert outputs arrive in fp32 (the projections keep their accumulators), so the layer output
// is rounded once.  One warp per (token, 256-column chunk); fp32 accumulation in slot order, then
// + shared.  All k source rows of a chunk are loaded before any is accumulated so a lane keeps up
// to 2(k+1) independent 16-byte loads in flight.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

// One warp per (token, 256-column chunk), 8 consecutive columns per lane (two 16-byte loads per
// source row), so that a call with few tokens still spreads over many SMs.
template <typename T, int KMAX>
__global__ void __launch_bounds__(256) k_combine(const float* __restrict__ y_perm, const int32_t* __restrict__ row_of,
                                                 const float* __restrict__ topk_w, const float* __restrict__ y_shared,
                                                 T* __restrict__ y, int Tn, int d, int k) {
  pdl_trigger();
  pdl_wait();
  const int nch = (d + 255) / 256;
  const long items = (long)Tn * nch;
  const long warps = (long)gridDim.x * 8;
  const int lane = threadIdx.x & 31;
  for (long it = (long)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += warps) {
    const int t = (int)(it / nch);
    const int c = (int)(it - (long)t * nch) * 256 + lane * 8;
    int rows[KMAX];
    float ws[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = (j < k) ? row_of[(size_t)t * k + j] : -1;
      ws[j] = (j < k) ? topk_w[(size_t)t * k + j] : 0.f;
    }
    if (c >= d) continue;
    float v[KMAX][8];
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (rows[j] >= 0) load8(y_perm + (size_t)rows[j] * d + c, v[j]);
    float sv[8];
    if (y_shared) load8(y_shared + (size_t)t * d + c, sv);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (rows[j] >= 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(ws[j], v[j][i], acc[i]);
      }
    if (y_shared) {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += sv[i];
    }
    store8(y + (size_t)t * d + c, acc);
  }
}

// Any d: one element per lane step (same accumulation order).
template <typename T>
__global__ void __launch_bounds__(256) k_combine_scalar(const float* __restrict__ y_perm,
                                                        const int32_t* __restrict__ row_of,
                                                        const float* __restrict__ topk_w,
                                                        const float* __restrict__ y_shared, T* __restrict__ y, int Tn,
                                                        int d, int k) {
  pdl_trigger();
  pdl_wait();
  const int warps = gridDim.x * 8;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < Tn; t += warps) {
    for (int c = threadIdx.x & 31; c < d; c += 32) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int r = row_of[(size_t)t * k + j];
        if (r >= 0) acc = fmaf(topk_w[(size_t)t * k + j], y_perm[(size_t)r * d + c], acc);
      }
      if (y_shared) acc += y_shared[(size_t)t * d + c];
      y[(size_t)t * d + c] = from_f<T>(acc);
    }
  }
}

template <typename T>
cudaError_t launch_t(const float* y_perm, const int32_t* row_of, const float* topk_w, const float* y_shared, void* y,
                     int Tn, int d, int k, cudaStream_t st) {
  const long items = (long)Tn * ((d + 255) / 256);
  int blocks = (int)((items + 7) / 8);
  if (blocks > 148 * 32) blocks = 148 * 32;
  T* yo = static_cast<T*>(y);
  const dim3 g(blocks), b(256);
  if (d % 8 != 0) return launch_pdl(k_combine_scalar<T>, g, b, 0, st, y_perm, row_of, topk_w, y_shared, yo, Tn, d, k);
  if (k <= 2) return launch_pdl(k_combine<T, 2>, g, b, 0, st, y_perm, row_of, topk_w, y_shared, yo, Tn, d, k);
  if (k <= 4) return launch_pdl(k_combine<T, 4>, g, b, 0, st, y_perm, row_of, topk_w, y_shared, yo, Tn, d, k);
  return launch_pdl(k_combine<T, 8>, g, b, 0, st, y_perm, row_of, topk_w, y_shared, yo, Tn, d, k);
}
}  // namespace

cudaError_t launch_combine(bool bf16, const float* y_perm, const int32_t* row_of, const float* topk_w,
                           const float* y_shared, void* y, int T, int d, int k, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (bf16) return launch_t<__nv_bfloat16>(y_perm, row_of, topk_w, y_shared, y, T, d, k, st);
  return launch_t<float>(y_perm, row_of, topk_w, y_shared, y, T, d, k, st);
}

}  // namespace moe
