// Expert projections on CUDA cores in fp32 -- the path of fp32 layers, whose parity bound
// (relative error 1e-4) rules out the tensor cores' reduced-precision fp32 formats.
//
// Expert FFN forms: GELU(erf) with biases (mini-moe tutorial, sec. 3.1) and SwiGLU (GPT-4 2%
// article, sec. 3.1).  One thread per output element; rows are grouped by expert through the
// device-side offsets, so no count ever returns to the host.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
__device__ __forceinline__ float gelu_erf(float u) { return 0.5f * u * (1.f + erff(u * 0.70710678118654752f)); }
__device__ __forceinline__ float silu(float u) { return u / (1.f + expf(-u)); }

template <typename T, typename TO, int ACT>
__global__ void __launch_bounds__(128) k_proj_simt(const T* __restrict__ A, int64_t lda,
                                                   const int32_t* __restrict__ offsets, int G, int rows_static,
                                                   const T* __restrict__ B0, const T* __restrict__ B1,
                                                   const T* __restrict__ bias, int N, int K, int N_w, int K_w,
                                                   TO* __restrict__ out, int64_t ldc) {
  const int row = blockIdx.x;
  const int n = blockIdx.y * blockDim.x + threadIdx.x;
  if (n >= N) return;
  int g = 0;
  if (offsets) {
    if (row < offsets[0] || row >= offsets[G]) return;  // a problem's rows need not start at row 0
    int lo = 0, hi = G;  // largest g with offsets[g] <= row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (offsets[mid] <= row) lo = mid; else hi = mid;
    }
    g = lo;
  } else if (row >= rows_static) {
    return;
  }
  const int gn = g + n / N_w, nn = n % N_w;
  const T* a = A + (size_t)row * lda;
  float acc0 = 0.f, acc1 = 0.f;
  for (int k0 = 0; k0 < K; k0 += K_w) {
    const int gw = gn + k0 / K_w;
    const T* b0 = B0 + ((size_t)gw * N_w + nn) * K_w;
    const T* b1 = (ACT == ACT_SWIGLU) ? B1 + ((size_t)gw * N_w + nn) * K_w : nullptr;
    const int kl = min(K_w, K - k0);
    for (int kk = 0; kk < kl; ++kk) {
      const float av = to_f(a[k0 + kk]);
      acc0 = fmaf(av, to_f(b0[kk]), acc0);
      if (ACT == ACT_SWIGLU) acc1 = fmaf(av, to_f(b1[kk]), acc1);
    }
  }
  float r;
  if (ACT == ACT_SWIGLU) {
    r = silu(acc0) * acc1;
  } else {
    if (bias) acc0 += to_f(bias[(size_t)gn * N_w + nn]);
    r = (ACT == ACT_GELU) ? gelu_erf(acc0) : acc0;
  }
  out[(size_t)row * ldc + n] = from_f<TO>(r);
}

template <typename T>
cudaError_t launch_t(const Projection& p, cudaStream_t st) {
  const int rows = p.offsets ? p.rows_alloc : p.rows_static;
  if (rows <= 0 || p.N <= 0) return cudaSuccess;
  dim3 grid(rows, (p.N + 127) / 128);
  const T* A = static_cast<const T*>(p.A);
  const T* B0 = static_cast<const T*>(p.B0);
  const T* B1 = static_cast<const T*>(p.B1);
  const T* bias = static_cast<const T*>(p.bias);
  switch (p.act) {
    case ACT_GELU:
      k_proj_simt<T, T, ACT_GELU><<<grid, 128, 0, st>>>(A, p.lda, p.offsets, p.G, p.rows_static, B0, B1, bias, p.N,
                                                        p.K, p.N_w, p.K_w, static_cast<T*>(p.out), p.ldc);
      break;
    case ACT_SWIGLU:
      k_proj_simt<T, T, ACT_SWIGLU><<<grid, 128, 0, st>>>(A, p.lda, p.offsets, p.G, p.rows_static, B0, B1, bias,
                                                          p.N, p.K, p.N_w, p.K_w, static_cast<T*>(p.out), p.ldc);
      break;
    default:
      if (p.out_f32)
        k_proj_simt<T, float, ACT_NONE><<<grid, 128, 0, st>>>(A, p.lda, p.offsets, p.G, p.rows_static, B0, B1, bias,
                                                              p.N, p.K, p.N_w, p.K_w, static_cast<float*>(p.out),
                                                              p.ldc);
      else
        k_proj_simt<T, T, ACT_NONE><<<grid, 128, 0, st>>>(A, p.lda, p.offsets, p.G, p.rows_static, B0, B1, bias, p.N,
                                                          p.K, p.N_w, p.K_w, static_cast<T*>(p.out), p.ldc);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_projection_simt(bool bf16, const Projection& p, cudaStream_t st) {
  return bf16 ? launch_t<__nv_bfloat16>(p, st) : launch_t<float>(p, st);
}

}  // namespace moe
