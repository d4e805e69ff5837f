// 8-bit expert weights: per-row scaled INT8 or E4M3 codes of a stack of weight matrices (the
// mini-moe tutorial's deployment advice: quantise every expert to cut what is stored and loaded).
//
// Logical row r of w [blocks][rows][cols] is row r of every block placed side by side (blocks = 1
// for per-row scales of an expert stack; blocks = S for the shared experts' down projections,
// which act as one [d, S*dff] matrix).  scale_r = max |row| / qmax and code = nearest code of
// w / scale_r, both IEEE float32 divisions, so the decisions are those of any float32
// implementation of the same definition.  One CTA per logical row: a max pass, then the codes.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int QTHREADS = 256;

__device__ __forceinline__ uint8_t code_int8(float q) {
  int v = __float2int_rn(q);  // nearest integer, ties to even
  v = v > 127 ? 127 : (v < -127 ? -127 : v);
  return (uint8_t)(int8_t)v;
}
__device__ __forceinline__ uint8_t code_e4m3(float q) {
  uint16_t r;  // nearest E4M3 value, ties to even, magnitudes above 448 saturate to 448
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(q));
  return (uint8_t)(r & 0xFFu);
}

template <typename T, int FMT>
__global__ void __launch_bounds__(QTHREADS) k_quantize(const T* __restrict__ w, int blocks, int rows, int cols,
                                                       uint8_t* __restrict__ codes, float* __restrict__ scale,
                                                       int32_t* nonfinite) {
  const int r = blockIdx.x;
  const int64_t n = (int64_t)blocks * cols;
  const int64_t bstride = (int64_t)rows * cols;
  auto at = [&](int64_t i) -> int64_t {  // element i of the logical row -> offset in w and codes
    const int64_t b = i / cols;
    return b * bstride + (int64_t)r * cols + (i - b * cols);
  };
  __shared__ float red[QTHREADS / 32];
  __shared__ int bad_sh;
  if (threadIdx.x == 0) bad_sh = 0;
  float m = 0.f;
  int bad = 0;
  for (int64_t i = threadIdx.x; i < n; i += QTHREADS) {
    const float v = to_f(w[at(i)]);
    if (!isfinite(v)) ++bad;
    m = fmaxf(m, fabsf(v));  // (fmaxf drops a NaN operand; such rows are reported, not scaled)
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (bad) atomicAdd(&bad_sh, bad);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < QTHREADS / 32; ++i) amax = fmaxf(amax, red[i]);
  const float qmax = FMT == 1 ? 127.f : 448.f;
  const float s = amax > 0.f ? __fdiv_rn(amax, qmax) : 1.f;
  for (int64_t i = threadIdx.x; i < n; i += QTHREADS) {
    const int64_t o = at(i);
    const float q = __fdiv_rn(to_f(w[o]), s);
    codes[o] = FMT == 1 ? code_int8(q) : code_e4m3(q);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    scale[r] = s;
    if (nonfinite && bad_sh) atomicAdd(nonfinite, bad_sh);
  }
}

template <typename T>
cudaError_t launch_fmt(int fmt, const void* w, int blocks, int rows, int cols, uint8_t* codes, float* scale,
                       int32_t* nonfinite, cudaStream_t st) {
  const T* wt = static_cast<const T*>(w);
  if (fmt == 1)
    k_quantize<T, 1><<<rows, QTHREADS, 0, st>>>(wt, blocks, rows, cols, codes, scale, nonfinite);
  else
    k_quantize<T, 2><<<rows, QTHREADS, 0, st>>>(wt, blocks, rows, cols, codes, scale, nonfinite);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_quantize(bool bf16, int fmt, const void* w, int blocks, int rows, int cols, uint8_t* codes,
                            float* scale, int32_t* nonfinite, cudaStream_t st) {
  if (fmt != 1 && fmt != 2) return cudaErrorInvalidValue;
  if (rows <= 0 || blocks <= 0 || cols <= 0) return cudaSuccess;
  return bf16 ? launch_fmt<__nv_bfloat16>(fmt, w, blocks, rows, cols, codes, scale, nonfinite, st)
              : launch_fmt<float>(fmt, w, blocks, rows, cols, codes, scale, nonfinite, st);
}

}  // namespace moe
