// Backward of the routing half of the layer (a first part of the backward pass: the pages train
// these layers with the load-balance and z-loss terms in the objective, the mini-moe tutorial's
// training loop and the FLAME-MoE summary, sec. 2).
//
//   combine:  y_t = sum over kept slots j of w_tj y_perm[row_of[t, j]]  (+ shared experts)
//             dL/dw_tj = <dy_t, y_perm[row]>   (0 for a dropped slot)
//             dL/dy_perm[row] = w_tj dy_t      (the down-projection's upstream gradient)
//   router:   w = softmax of the k selected logits / tau (the renormalised top-k probabilities), so
//             dz_e = w_e (dw_e - sum_i w_i dw_i) for the selected e; the load-balance loss
//             alpha E sum_e f_e Pbar_e adds P_te (g_e - sum_e' P_te' g_e'), g_e = dlb alpha E f_e / T
//             (f_e = counts_e / (T k); top-k selection and counts pass no gradient); the z-loss
//             beta mean_t lse_t^2 adds dzl 2 beta lse_t P_te / T; everything is divided by tau;
//             then dW_r = dz^T x and dx = dz W_r.
// Every sum runs in a fixed order (results do not depend on scheduling).  fp32 arithmetic on CUDA
// cores: these are small contractions next to the expert GEMMs (E <= 256 columns).
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr float kBad = -3.0e38f;

// One warp per (token, slot): the dot product of dy_t and the slot's fp32 output row (lane-strided,
// then a fixed shuffle tree), and the row's upstream gradient w_tj dy_t.
template <typename T>
__global__ void __launch_bounds__(256) k_combine_bwd(const T* __restrict__ dy, const float* __restrict__ y_perm,
                                                     const int32_t* __restrict__ row_of,
                                                     const float* __restrict__ topk_w, int Tn, int d, int k,
                                                     float* __restrict__ dw, T* __restrict__ dy_perm) {
  const int warp_g = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_g >= Tn * k) return;
  const int t = warp_g / k;
  const int r = row_of[warp_g];
  if (r < 0) {
    if (lane == 0) dw[warp_g] = 0.f;
    return;
  }
  const float w = topk_w[warp_g];
  const T* dyt = dy + (size_t)t * d;
  const float* yr = y_perm + (size_t)r * d;
  T* out = dy_perm + (size_t)r * d;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float g = to_f(dyt[c]);
    s = fmaf(g, yr[c], s);
    out[c] = from_f<T>(w * g);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) dw[warp_g] = s;
}

// Router gradient of the logits, 32 tokens per CTA: the fp32 logits (K in chunks of 64 columns
// through shared memory, every logit accumulated in column order), then one warp per token.
constexpr int BT = 32, BC = 64, BTHREADS = 256;
constexpr int BMAXO = BT * 256 / BTHREADS;

template <typename T>
__global__ void __launch_bounds__(BTHREADS) k_router_dz(const T* __restrict__ x, const T* __restrict__ wr,
                                                        const float* __restrict__ lbias, const int32_t* __restrict__ idx,
                                                        const float* __restrict__ tw, const int32_t* __restrict__ counts,
                                                        const float* __restrict__ dw, int Tn, int d, int E, int k,
                                                        float inv_tau, float lb_coef, float z_coef, float dlb, float dzl,
                                                        float* __restrict__ dz) {
  extern __shared__ float sm[];
  float* xs = sm;                   // [BT][BC+1]
  float* wsm = xs + BT * (BC + 1);  // [E][BC+1]
  float* zs = wsm + E * (BC + 1);   // [BT][E+1]
  float* gp = zs + BT * (E + 1);    // [E]: dlb alpha E f_e / T
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * BT;
  const int nvalid = min(BT, Tn - t0);
  for (int e = tid; e < E; e += BTHREADS)
    gp[e] = dlb * lb_coef * (float)E * ((float)counts[e] / ((float)Tn * (float)k)) / (float)Tn;
  const int nout = BT * E;
  float acc[BMAXO];
#pragma unroll
  for (int j = 0; j < BMAXO; ++j) acc[j] = 0.f;
  for (int c0 = 0; c0 < d; c0 += BC) {
    const int cw = min(BC, d - c0);
    for (int i = tid; i < BT * BC; i += BTHREADS) {
      const int r = i / BC, c = i - r * BC;
      xs[r * (BC + 1) + c] = (r < nvalid && c < cw) ? to_f(x[(size_t)(t0 + r) * d + c0 + c]) : 0.f;
    }
    for (int i = tid; i < E * BC; i += BTHREADS) {
      const int e = i / BC, c = i - e * BC;
      wsm[e * (BC + 1) + c] = c < cw ? to_f(wr[(size_t)e * d + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < BMAXO; ++j) {
      const int o = tid + j * BTHREADS;
      if (o < nout) {
        const int r = o / E, e = o - r * E;
        const float* xr = xs + r * (BC + 1);
        const float* we = wsm + e * (BC + 1);
        float a = acc[j];
#pragma unroll 8
        for (int c = 0; c < BC; ++c) a = fmaf(xr[c], we[c], a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < BMAXO; ++j) {
    const int o = tid + j * BTHREADS;
    if (o < nout) {
      const int r = o / E, e = o - r * E;
      const float z = acc[j] + (lbias ? lbias[e] : 0.f);
      zs[r * (E + 1) + e] = isfinite(z) ? z : kBad;
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < nvalid; r += BTHREADS / 32) {
    const int t = t0 + r;
    const float* zr = zs + r * (E + 1);
    float m = kBad;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, zr[e]);
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += __expf((zr[e] - m) * inv_tau);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv_s = 1.f / s;
    const float lse = m * inv_tau + __logf(s);
    // sum_e P_e g_e (load-balance term) and sum_j w_j dw_j (renormalised top-k)
    float pg = 0.f;
    for (int e = lane; e < E; e += 32) pg = fmaf(__expf((zr[e] - m) * inv_tau) * inv_s, gp[e], pg);
#pragma unroll
    for (int o = 16; o; o >>= 1) pg += __shfl_xor_sync(0xffffffffu, pg, o);
    float wd = 0.f;
    for (int j = 0; j < k; ++j) wd = fmaf(tw[(size_t)t * k + j], dw[(size_t)t * k + j], wd);
    const float zc = dzl * 2.f * z_coef * lse / (float)Tn;
    for (int e = lane; e < E; e += 32) {
      const float p = __expf((zr[e] - m) * inv_tau) * inv_s;
      float g = p * (gp[e] - pg) + zc * p;
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) g += tw[(size_t)t * k + j] * (dw[(size_t)t * k + j] - wd);
      dz[(size_t)t * E + e] = g * inv_tau;
    }
  }
}

// dW_r [E, d] = dz^T x: a CTA per block of 32 experts x 64 columns, the tokens in chunks of 32
// through shared memory, each output summed in token order.
template <typename T>
__global__ void __launch_bounds__(256) k_router_dwr(const float* __restrict__ dz, const T* __restrict__ x, int Tn,
                                                    int d, int E, float* __restrict__ dwr) {
  __shared__ float zsm[32][33];  // [token][expert]
  __shared__ float xsm[32][65];  // [token][column]
  const int e0 = blockIdx.y * 32, c0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  const int el = tid >> 3, cl = (tid & 7) * 8;  // this thread: expert e0 + el, columns c0 + cl .. + 7
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int t0 = 0; t0 < Tn; t0 += 32) {
    for (int i = tid; i < 32 * 32; i += 256) {
      const int tt = i >> 5, e = i & 31;
      zsm[tt][e] = (t0 + tt < Tn && e0 + e < E) ? dz[(size_t)(t0 + tt) * E + e0 + e] : 0.f;
    }
    for (int i = tid; i < 32 * 64; i += 256) {
      const int tt = i >> 6, c = i & 63;
      xsm[tt][c] = (t0 + tt < Tn && c0 + c < d) ? to_f(x[(size_t)(t0 + tt) * d + c0 + c]) : 0.f;
    }
    __syncthreads();
    for (int tt = 0; tt < 32; ++tt) {
      const float g = zsm[tt][el];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, xsm[tt][cl + i], acc[i]);
    }
    __syncthreads();
  }
  if (e0 + el < E) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + cl + i < d) dwr[(size_t)(e0 + el) * d + c0 + cl + i] = acc[i];
  }
}

// dx [T, d] = dz W_r: a CTA per block of 32 tokens x 64 columns, the experts in order.
template <typename T>
__global__ void __launch_bounds__(256) k_router_dx(const float* __restrict__ dz, const T* __restrict__ wr, int Tn,
                                                   int d, int E, float* __restrict__ dx) {
  __shared__ float zsm[32][33];  // [token][expert chunk]
  __shared__ float wsm[32][65];  // [expert chunk][column]
  const int t0 = blockIdx.y * 32, c0 = blockIdx.x * 64;
  const int tid = threadIdx.x;
  const int tl = tid >> 3, cl = (tid & 7) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int e0 = 0; e0 < E; e0 += 32) {
    for (int i = tid; i < 32 * 32; i += 256) {
      const int tt = i >> 5, e = i & 31;
      zsm[tt][e] = (t0 + tt < Tn && e0 + e < E) ? dz[(size_t)(t0 + tt) * E + e0 + e] : 0.f;
    }
    for (int i = tid; i < 32 * 64; i += 256) {
      const int e = i >> 6, c = i & 63;
      wsm[e][c] = (e0 + e < E && c0 + c < d) ? to_f(wr[(size_t)(e0 + e) * d + c0 + c]) : 0.f;
    }
    __syncthreads();
    for (int e = 0; e < 32; ++e) {
      const float g = zsm[tl][e];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, wsm[e][cl + i], acc[i]);
    }
    __syncthreads();
  }
  if (t0 + tl < Tn) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + cl + i < d) dx[(size_t)(t0 + tl) * d + c0 + cl + i] = acc[i];
  }
}

template <typename T>
cudaError_t router_bwd_t(const void* x, const void* wr, const float* lbias, const int32_t* idx, const float* tw,
                         const int32_t* counts, const float* dw, int T_, int d, int E, int k, float inv_tau,
                         float lb_coef, float z_coef, float dlb, float dzl, float* dz, float* dwr, float* dx,
                         cudaStream_t st) {
  const T* xt = static_cast<const T*>(x);
  const T* wt = static_cast<const T*>(wr);
  if (T_ > 0) {
    const size_t smem = sizeof(float) * ((size_t)BT * (BC + 1) + (size_t)E * (BC + 1) + (size_t)BT * (E + 1) + E);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_router_dz<T>), smem);
    if (e != cudaSuccess) return e;
    k_router_dz<T><<<(T_ + BT - 1) / BT, BTHREADS, smem, st>>>(xt, wt, lbias, idx, tw, counts, dw, T_, d, E, k,
                                                               inv_tau, lb_coef, z_coef, dlb, dzl, dz);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_router_dx<T><<<dim3((d + 63) / 64, (T_ + 31) / 32), 256, 0, st>>>(dz, wt, T_, d, E, dx);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_router_dwr<T><<<dim3((d + 63) / 64, (E + 31) / 32), 256, 0, st>>>(dz, xt, T_, d, E, dwr);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_combine_backward(bool bf16, const void* dy, const float* y_perm, const int32_t* row_of,
                                    const float* topk_w, int T, int d, int k, float* dw, void* dy_perm,
                                    cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const size_t threads = (size_t)T * k * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (bf16)
    k_combine_bwd<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(dy), y_perm, row_of, topk_w,
                                                         T, d, k, dw, static_cast<__nv_bfloat16*>(dy_perm));
  else
    k_combine_bwd<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(dy), y_perm, row_of, topk_w, T, d, k, dw,
                                                 static_cast<float*>(dy_perm));
  return cudaGetLastError();
}

cudaError_t launch_router_backward(bool bf16, const void* x, const void* wr, const float* lbias, const int32_t* idx,
                                   const float* tw, const int32_t* counts, const float* dw, int T, int d, int E, int k,
                                   float inv_tau, float lb_coef, float z_coef, float dlb, float dzl, float* dz,
                                   float* dwr, float* dx, cudaStream_t st) {
  if (E < 1 || E > 256 || k < 1 || k > 8 || k > E) return cudaErrorInvalidValue;
  if (bf16)
    return router_bwd_t<__nv_bfloat16>(x, wr, lbias, idx, tw, counts, dw, T, d, E, k, inv_tau, lb_coef, z_coef, dlb,
                                       dzl, dz, dwr, dx, st);
  return router_bwd_t<float>(x, wr, lbias, idx, tw, counts, dw, T, d, E, k, inv_tau, lb_coef, z_coef, dlb, dzl, dz,
                             dwr, dx, st);
}

}  // namespace moe
