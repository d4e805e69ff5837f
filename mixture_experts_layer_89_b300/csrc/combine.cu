// Combine: y[t] = sum over kept slots j of w[t,j] * y_perm[row_of[t,j]]  (+ y_shared[t]).
//
// The layer output is the routing-weighted sum of the selected experts' outputs (FLAME-MoE
// summary, sec. 2; the accumulation of the mini-moe tutorial, sec. 3.1 MoELayer), plus the
// always-on shared experts.  A dropped slot (row -1) contributes nothing and the surviving
// weights are not renormalised (OpenMythos article, sec. 3.1, overflow handling).
//
// One warp per token; each lane moves 16-byte vectors; fp32 accumulation in slot order, one
// rounding at the store.  All k source rows of a chunk are loaded before any is accumulated so a
// lane keeps up to k+1 independent 16-byte loads in flight.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[8]) {
    uint4 q;
    q.x = pack_bf16x2(v[0], v[1]);
    q.y = pack_bf16x2(v[2], v[3]);
    q.z = pack_bf16x2(v[4], v[5]);
    q.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = q;
  }
};

template <typename T, int KMAX>
__global__ void __launch_bounds__(256) k_combine(const T* __restrict__ y_perm, const int32_t* __restrict__ row_of,
                                                 const float* __restrict__ topk_w, const T* __restrict__ y_shared,
                                                 T* __restrict__ y, int Tn, int d, int k) {
  constexpr int N = Vec<T>::N;
  const int warps = gridDim.x * 8;
  const int lane = threadIdx.x & 31;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < Tn; t += warps) {
    int rows[KMAX];
    float ws[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      rows[j] = (j < k) ? row_of[(size_t)t * k + j] : -1;
      ws[j] = (j < k) ? topk_w[(size_t)t * k + j] : 0.f;
    }
    for (int c = lane * N; c < d; c += 32 * N) {
      float acc[N];
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.f;
      float v[KMAX][N];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (rows[j] >= 0) Vec<T>::load(y_perm + (size_t)rows[j] * d + c, v[j]);
      float sv[N];
      if (y_shared) Vec<T>::load(y_shared + (size_t)t * d + c, sv);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (rows[j] >= 0) {
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] = fmaf(ws[j], v[j][i], acc[i]);
        }
      if (y_shared) {
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += sv[i];
      }
      Vec<T>::store(y + (size_t)t * d + c, acc);
    }
  }
}

// Any d: one element per lane step.
template <typename T>
__global__ void __launch_bounds__(256) k_combine_scalar(const T* __restrict__ y_perm,
                                                        const int32_t* __restrict__ row_of,
                                                        const float* __restrict__ topk_w,
                                                        const T* __restrict__ y_shared, T* __restrict__ y, int Tn,
                                                        int d, int k) {
  const int warps = gridDim.x * 8;
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < Tn; t += warps) {
    for (int c = threadIdx.x & 31; c < d; c += 32) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int r = row_of[(size_t)t * k + j];
        if (r >= 0) acc = fmaf(topk_w[(size_t)t * k + j], to_f(y_perm[(size_t)r * d + c]), acc);
      }
      if (y_shared) acc += to_f(y_shared[(size_t)t * d + c]);
      y[(size_t)t * d + c] = from_f<T>(acc);
    }
  }
}

template <typename T>
cudaError_t launch_t(const void* y_perm, const int32_t* row_of, const float* topk_w, const void* y_shared, void* y,
                     int Tn, int d, int k, cudaStream_t st) {
  int blocks = (Tn + 7) / 8;
  if (blocks > 148 * 32) blocks = 148 * 32;
  const T* yp = static_cast<const T*>(y_perm);
  const T* ys = static_cast<const T*>(y_shared);
  T* yo = static_cast<T*>(y);
  if (((size_t)d * sizeof(T)) % 16 != 0) {
    k_combine_scalar<T><<<blocks, 256, 0, st>>>(yp, row_of, topk_w, ys, yo, Tn, d, k);
  } else if (k <= 2) {
    k_combine<T, 2><<<blocks, 256, 0, st>>>(yp, row_of, topk_w, ys, yo, Tn, d, k);
  } else if (k <= 4) {
    k_combine<T, 4><<<blocks, 256, 0, st>>>(yp, row_of, topk_w, ys, yo, Tn, d, k);
  } else {
    k_combine<T, 8><<<blocks, 256, 0, st>>>(yp, row_of, topk_w, ys, yo, Tn, d, k);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_combine(bool bf16, const void* y_perm, const int32_t* row_of, const float* topk_w,
                           const void* y_shared, void* y, int T, int d, int k, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (bf16) return launch_t<__nv_bfloat16>(y_perm, row_of, topk_w, y_shared, y, T, d, k, st);
  return launch_t<float>(y_perm, row_of, topk_w, y_shared, y, T, d, k, st);
}

}  // namespace moe
