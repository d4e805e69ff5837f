// Backward pass of the layer (the pages train these layers with the load-balance and z-loss terms
// in the objective: the mini-moe tutorial's training loop and the FLAME-MoE summary, sec. 2).
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
//   experts:  pre-activations recomputed from the permuted rows; dh = dy_perm W_down; the
//             activation backward (du, dg or da, and h); dx_perm = du W_up + dg W_gate; the weight
//             gradients dW_down = dy_perm^T h, dW_up = du^T x_perm, dW_gate = dg^T x_perm (and the
//             bias sums) per expert; each token's rows added into dx; shared experts over all tokens.
// Every sum runs in a fixed order (results do not depend on scheduling).  bf16 layers run the
// contractions on the tensor cores (the grouped GEMM of gemm_bwd.cu); fp32 layers, and the router
// without its scratch, on CUDA cores through one register-tiled SGEMM in fp32.
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

// C [M, N] fp32 (row-major, ldc) = sum_k A(m, k) B(k, n), on CUDA cores: 128 x 128 output tiles,
// 256 threads with 8 x 8 register tiles (two 4 x 4 quadrants 64 rows / columns apart, so the
// shared-memory reads are conflict-free float4s), K in steps of 8 through shared memory.  Every
// output is accumulated in k order.  A(m, k) = A[m lda + k] (AK: K contiguous) or A[k lda + m];
// B(k, n) = B[k ldb + n] (BN: N contiguous) or B[n ldb + k].
// Grouped form (blockIdx.z = group g, rows of g = [off[g], off[g + 1]) of the permuted rows):
//   rows on M: A and C rows offset by off[g] (A K-contiguous), B offset by g b_stride, M = rows of g;
//   rows on K: A and B rows offset by off[g] (A M-contiguous, B N-contiguous), C offset by
//              g c_stride, K = rows of g.
// beta = 1 adds the product to C instead of overwriting it.
struct GemmGroups {
  const int32_t* off;  // NULL: one plain problem
  int rows_on_k;
  int64_t b_stride, c_stride;
  int beta;
};

template <typename TA, typename TB, bool AK, bool BN>
__global__ void __launch_bounds__(256) k_sgemm(const TA* __restrict__ A, int64_t lda, const TB* __restrict__ B,
                                               int64_t ldb, float* __restrict__ C, int64_t ldc, int M, int N,
                                               int K, const GemmGroups gr) {
  __shared__ __align__(16) float As[8][128];
  __shared__ __align__(16) float Bs[8][128];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * 128, n0 = blockIdx.x * 128;
  if (gr.off) {
    const int g = blockIdx.z;
    const int lo = gr.off[g], hi = gr.off[g + 1];
    if (gr.rows_on_k) {
      K = hi - lo;
      A += (size_t)lo * lda;
      B += (size_t)lo * ldb;
      C += (size_t)g * gr.c_stride;
    } else {
      M = hi - lo;
      A += (size_t)lo * lda;
      C += (size_t)lo * ldc;
      B += (size_t)g * gr.b_stride;
    }
    if (m0 >= M) return;
  }
  const int ty = tid >> 4, tx = tid & 15;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 8) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 1024 elements of each operand tile, 4 per thread
      const int i = tid + q * 256;
      // A tile [128 m][8 k], B tile [8 k][128 n]: index so that consecutive threads read
      // consecutive addresses of the operand's contiguous dimension
      const int am = AK ? (i >> 3) : (i & 127), ak = AK ? (i & 7) : (i >> 7);
      const int gm = m0 + am, gk = k0 + ak;
      As[ak][am] = (gm < M && gk < K) ? to_f(AK ? A[(size_t)gm * lda + gk] : A[(size_t)gk * lda + gm]) : 0.f;
      const int bn = BN ? (i & 127) : (i >> 3), bk = BN ? (i >> 7) : (i & 7);
      const int gn = n0 + bn, gk2 = k0 + bk;
      Bs[bk][bn] = (gn < N && gk2 < K) ? to_f(BN ? B[(size_t)gk2 * ldb + gn] : B[(size_t)gn * ldb + gk2]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (gn < N) C[(size_t)gm * ldc + gn] = gr.beta ? C[(size_t)gm * ldc + gn] + acc[i][j] : acc[i][j];
    }
  }
}

// M: the rows (plain), or a bound on any group's rows (rows on M); G groups (1 when plain).
template <typename TA, typename TB, bool AK, bool BN>
cudaError_t sgemm(const TA* A, int64_t lda, const TB* B, int64_t ldb, float* C, int64_t ldc, int M, int N, int K,
                  cudaStream_t st, const GemmGroups& gr = GemmGroups{nullptr, 0, 0, 0, 0}, int G = 1) {
  if (M <= 0 || N <= 0 || G <= 0) return cudaSuccess;
  k_sgemm<TA, TB, AK, BN><<<dim3((N + 127) / 128, (M + 127) / 128, G), 256, 0, st>>>(A, lda, B, ldb, C, ldc, M, N, K,
                                                                                     gr);
  return cudaGetLastError();
}

// out[i] = sum over the S slices of part[s][i], in slice order (the split-K partials of dW_r).
__global__ void __launch_bounds__(256) k_sum_slices(const float* __restrict__ part, int S, size_t n,
                                                    float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += part[(size_t)q * n + i];
    out[i] = v;
  }
}

// Router gradient of the logits from the fp32 logits z [T, E] (without the logit bias; recomputed
// by the SGEMM above, each in column order): one warp per token.
template <typename T>
__global__ void __launch_bounds__(256) k_router_dz2(const float* zin, const float* __restrict__ lbias,
                                                    const int32_t* __restrict__ idx, const float* __restrict__ tw,
                                                    const int32_t* __restrict__ counts, const float* __restrict__ dw,
                                                    int Tn, int E, int k, float inv_tau, float lb_coef, float z_coef,
                                                    float dlb, float dzl, float* dz) {
  // zin and dz may be the same buffer: each warp reads its token's row before writing it
  __shared__ float gp[256];  // dlb alpha E f_e / T
  for (int e = threadIdx.x; e < E; e += 256)
    gp[e] = dlb * lb_coef * (float)E * ((float)counts[e] / ((float)Tn * (float)k)) / (float)Tn;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= Tn) return;
  float zr[8];
  float m = kBad;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float z = kBad;
    if (e < E) {
      z = zin[(size_t)t * E + e] + (lbias ? lbias[e] : 0.f);
      if (!isfinite(z)) z = kBad;
    }
    zr[i] = z;
    m = fmaxf(m, z);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float p[8], s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    p[i] = lane + 32 * i < E ? __expf((zr[i] - m) * inv_tau) : 0.f;
    s += p[i];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float inv_s = 1.f / s;
  const float lse = m * inv_tau + __logf(s);
  float pg = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    p[i] *= inv_s;
    if (lane + 32 * i < E) pg = fmaf(p[i], gp[lane + 32 * i], pg);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) pg += __shfl_xor_sync(0xffffffffu, pg, o);
  float wd = 0.f;
  for (int j = 0; j < k; ++j) wd = fmaf(tw[(size_t)t * k + j], dw[(size_t)t * k + j], wd);
  const float zc = dzl * 2.f * z_coef * lse / (float)Tn;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e >= E) continue;
    float g = p[i] * (gp[e] - pg) + zc * p[i];
    for (int j = 0; j < k; ++j)
      if (idx[(size_t)t * k + j] == e) g += tw[(size_t)t * k + j] * (dw[(size_t)t * k + j] - wd);
    dz[(size_t)t * E + e] = g * inv_tau;
  }
}

__global__ void k_transpose_pad(const __nv_bfloat16* __restrict__ in, int64_t ldi, int C,
                                const int32_t* __restrict__ off, const int32_t* __restrict__ koff, int G, int rows,
                                __nv_bfloat16* __restrict__ out, int64_t Kp);

// dz [T, E] fp32 -> dzs [T, 2E] bf16: hi = bf16(dz) at column e, lo = bf16(dz - hi) at E + e
// (hi + lo carries 16 significant bits: |dz - hi - lo| <= 2^-17 |dz|).
__global__ void __launch_bounds__(256) k_split_hi_lo(const float* __restrict__ dz, int Tn, int E,
                                                     __nv_bfloat16* __restrict__ dzs) {
  const size_t n = (size_t)Tn * E;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t t = i / E, e = i % E;
    const float v = dz[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    dzs[t * 2 * E + e] = hi;
    dzs[t * 2 * E + E + e] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

// out[i] = the hi and lo halves of dW_r over the S token slices, summed in slice order:
// part [S][2][n] (hi rows first, then lo rows, per slice).
__global__ void __launch_bounds__(256) k_sum_halves(const float* __restrict__ part, int S, size_t n,
                                                    float* __restrict__ out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += part[(size_t)q * 2 * n + i] + part[(size_t)q * 2 * n + n + i];
    out[i] = v;
  }
}

// koff[s] = the first padded token column of slice s of [0, Tp) (multiples of 64), koff[S] = Tp.
__global__ void k_slice_offsets(int Tp, int S, int32_t* __restrict__ koff) {
  const int s = threadIdx.x;
  if (s <= S) koff[s] = (int)((int64_t)(Tp / 64) * s / S) * 64;
}

// bf16 layers with E a multiple of 64 and a scratch: the three contractions on the tensor cores
// (k_gemm_bwd).  The logits are recomputed with fp32 accumulation from the bf16 x and W_r as on
// the CUDA cores; dz enters dW_r = dz^T x and dx = dz W_r as its bf16 hi and lo parts side by side
// along K (so both keep ~2^-17 relative accuracy): dx = [hi | lo] [W_r; W_r] in one contraction
// (W_r read N-major twice), and [hi^T; lo^T] x as a 2E x d product whose halves are summed.
// scratch: status word, dzs [T, 2E] and its transpose [2E, Tp] bf16, x^T [d, Tp] bf16 (Tp = T
// padded to 64), the 2E x d fp32 product.
cudaError_t router_bwd_tc(const __nv_bfloat16* x, const __nv_bfloat16* wr, const float* lbias, const int32_t* idx,
                          const float* tw, const int32_t* counts, const float* dw, int T_, int d, int E, int k,
                          float inv_tau, float lb_coef, float z_coef, float dlb, float dzl, float* dz, float* dwr,
                          float* dx, const RouterBwdScratch& sc, cudaStream_t st) {
  const int Tp = (T_ + 63) & ~63;
  cudaError_t e = cudaMemsetAsync(sc.status, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess)  // z [T, E] = x W_r^T
    e = launch_gemm_bwd_rows_m(x, T_, wr, 1, E, d, nullptr, 1, T_, dz, E, 0, sc.status, st);
  if (e != cudaSuccess) return e;
  k_router_dz2<__nv_bfloat16><<<(T_ + 7) / 8, 256, 0, st>>>(dz, lbias, idx, tw, counts, dw, T_, E, k, inv_tau, lb_coef,
                                                            z_coef, dlb, dzl, dz);
  k_split_hi_lo<<<592, 256, 0, st>>>(dz, T_, E, sc.dzs);
  const dim3 tb(32, 8);
  k_transpose_pad<<<dim3(Tp / 64, (2 * E + 127) / 128), tb, 0, st>>>(sc.dzs, 2 * E, 2 * E, nullptr, nullptr, 1, T_,
                                                                   sc.dzsT, Tp);
  k_transpose_pad<<<dim3(Tp / 64, (d + 127) / 128), tb, 0, st>>>(x, d, d, nullptr, nullptr, 1, T_, sc.xT, Tp);
  // [hi^T; lo^T] x over the tokens, split into S slices of the token columns (groups of the GEMM)
  // so that enough pairs share the few 2E x d output tiles; partials summed in slice order
  const int tiles = ((2 * E + 255) / 256) * ((d + 255) / 256);
  const int S = max(1, min(min(kRouterBwdSlices, 64 / tiles), Tp / 64));
  if (S > 1) {
    k_slice_offsets<<<1, 32, 0, st>>>(Tp, S, sc.koff);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess)  // one slice: a single group of Tp columns, no offsets array
    e = launch_gemm_bwd_rows_k(sc.dzsT, 2 * E, sc.xT, d, Tp, S > 1 ? sc.koff : nullptr, S, Tp, sc.part, d,
                               (int64_t)2 * E * d, 0, sc.status, st);
  if (e != cudaSuccess) return e;
  k_sum_halves<<<592, 256, 0, st>>>(sc.part, S, (size_t)E * d, dwr);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dx = [hi | lo] [W_r; W_r]
  return launch_gemm_bwd_rows_m_nmajor(sc.dzs, T_, wr, wr, E, 1, d, 2 * E, nullptr, 1, T_, dx, d, 0, sc.status, st,
                                       true);
}

template <typename T>
cudaError_t router_bwd_t(const void* x, const void* wr, const float* lbias, const int32_t* idx, const float* tw,
                         const int32_t* counts, const float* dw, int T_, int d, int E, int k, float inv_tau,
                         float lb_coef, float z_coef, float dlb, float dzl, float* dz, float* dwr, float* dx,
                         cudaStream_t st) {
  const T* xt = static_cast<const T*>(x);
  const T* wt = static_cast<const T*>(wr);
  if (T_ > 0) {
    // z [T, E] = x W_r^T into dz (then overwritten by the logits' gradient, token by token)
    cudaError_t e = sgemm<T, T, true, false>(xt, d, wt, d, dz, E, T_, E, d, st);
    if (e != cudaSuccess) return e;
    k_router_dz2<T><<<(T_ + 7) / 8, 256, 0, st>>>(dz, lbias, idx, tw, counts, dw, T_, E, k, inv_tau, lb_coef, z_coef,
                                                  dlb, dzl, dz);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // dW_r = dz^T x: the tokens split into S slices (more CTAs than the E x d output alone gives),
    // the slices' partials in the dx buffer (S E <= T floats per column), summed in slice order
    const int S = T_ >= 8 * E ? 8 : (T_ >= 2 * E ? T_ / E : 1);
    if (S == 1) {
      e = sgemm<float, T, false, true>(dz, E, xt, d, dwr, d, E, d, T_, st);
    } else {
      const int ts = (T_ + S - 1) / S;
      for (int q = 0; q < S && e == cudaSuccess; ++q) {
        const int t0 = q * ts, tn = min(ts, T_ - t0);
        if (tn > 0)
          e = sgemm<float, T, false, true>(dz + (size_t)t0 * E, E, xt + (size_t)t0 * d, d, dx + (size_t)q * E * d, d, E,
                                           d, tn, st);
        else
          e = cudaMemsetAsync(dx + (size_t)q * E * d, 0, sizeof(float) * (size_t)E * d, st);
      }
      if (e == cudaSuccess) {
        k_sum_slices<<<592, 256, 0, st>>>(dx, S, (size_t)E * d, dwr);
        e = cudaGetLastError();
      }
    }
    if (e != cudaSuccess) return e;
    return sgemm<float, T, true, true>(dz, E, wt, d, dx, d, T_, d, E, st);  // dx = dz W_r (overwrites the partials)
  }
  return cudaMemsetAsync(dwr, 0, sizeof(float) * (size_t)E * d, st);
}

// Activation backward, elementwise over the rows of each group (blockIdx.y = group; rows
// [off[g], off[g + 1]), or [0, rows) with off == NULL), in place:
//   SwiGLU: gate and up pre-activations p0 = g, p1 = u and dh -> p0 = dg = dh u silu'(g),
//           p1 = du = dh silu(g), dh = h = silu(g) u;
//   GELU:   pre-activation p0 = a (bias b[g] not yet added) and dh -> p0 = da = dh gelu'(a + b),
//           dh = h = gelu(a + b).
// silu(g) = g sigma(g), silu'(g) = sigma(g) (1 + g (1 - sigma(g))); gelu(a) = a Phi(a),
// gelu'(a) = Phi(a) + a phi(a) with the standard normal CDF Phi and density phi.
__device__ __forceinline__ void swiglu_bwd(float gv, float uv, float up, float& dg, float& du, float& h) {
  const float sg = 1.f / (1.f + expf(-gv));
  const float si = gv * sg;
  dg = up * uv * (sg * (1.f + gv * (1.f - sg)));
  du = up * si;
  h = si * uv;
}
__device__ __forceinline__ void gelu_bwd(float a, float up, float& da, float& h) {
  const float cdf = 0.5f * (1.f + erff(a * 0.70710678118654752f));
  const float pdf = 0.39894228040143268f * expf(-0.5f * a * a);
  da = up * (cdf + a * pdf);
  h = a * cdf;
}

template <int ACT, typename T>
__global__ void __launch_bounds__(256) k_act_bwd(float* __restrict__ p0, float* __restrict__ p1,
                                                 float* __restrict__ dh, const T* __restrict__ bias,
                                                 const int32_t* __restrict__ off, int rows, int dff) {
  const int g = blockIdx.y;
  const int lo = off ? off[g] : 0, hi = off ? off[g + 1] : rows;
  for (int r = lo + (int)blockIdx.x; r < hi; r += gridDim.x) {
    const size_t base = (size_t)r * dff;
    for (int c = threadIdx.x; c < dff; c += blockDim.x) {
      const size_t i = base + c;
      if (ACT == ACT_SWIGLU) {
        swiglu_bwd(p0[i], p1[i], dh[i], p0[i], p1[i], dh[i]);
      } else {
        const float a = p0[i] + (bias ? to_f(bias[(size_t)g * dff + c]) : 0.f);
        gelu_bwd(a, dh[i], p0[i], dh[i]);
      }
    }
  }
}

// The same for bf16 layers, whose next contractions run on the tensor cores: from the fp32
// pre-activations p0 (g, or a without its bias), p1 (u) and dh, the bf16 operands D [rows][ldd]
// (SwiGLU: du at column c and dg at dff + c; GELU: da) and h [rows][dff]; GELU also keeps the fp32
// da in p0 for the bias sums.  Four columns per thread (dff is a multiple of 64).
__device__ __forceinline__ void st_bf16x4(__nv_bfloat16* p, float a, float b, float c, float d) {
  uint2 v;
  v.x = pack_bf16x2(a, b);
  v.y = pack_bf16x2(c, d);
  *reinterpret_cast<uint2*>(p) = v;
}

template <int ACT>
__global__ void __launch_bounds__(256) k_act_bwd_tc(float* __restrict__ p0, const float* __restrict__ p1,
                                                    const float* __restrict__ dh, const __nv_bfloat16* __restrict__ bias,
                                                    const int32_t* __restrict__ off, int rows, int dff,
                                                    __nv_bfloat16* __restrict__ D, int64_t ldd,
                                                    __nv_bfloat16* __restrict__ h) {
  const int g = blockIdx.y;
  const int lo = off ? off[g] : 0, hi = off ? off[g + 1] : rows;
  for (int r = lo + (int)blockIdx.x; r < hi; r += gridDim.x) {
    for (int c = 4 * threadIdx.x; c < dff; c += 4 * blockDim.x) {
      const size_t i = (size_t)r * dff + c;
      const float4 up = *reinterpret_cast<const float4*>(dh + i);
      const float4 x0 = *reinterpret_cast<const float4*>(p0 + i);
      float hv[4];
      if (ACT == ACT_SWIGLU) {
        const float4 x1 = *reinterpret_cast<const float4*>(p1 + i);
        float dg[4], du[4];
        swiglu_bwd(x0.x, x1.x, up.x, dg[0], du[0], hv[0]);
        swiglu_bwd(x0.y, x1.y, up.y, dg[1], du[1], hv[1]);
        swiglu_bwd(x0.z, x1.z, up.z, dg[2], du[2], hv[2]);
        swiglu_bwd(x0.w, x1.w, up.w, dg[3], du[3], hv[3]);
        st_bf16x4(D + (size_t)r * ldd + c, du[0], du[1], du[2], du[3]);
        st_bf16x4(D + (size_t)r * ldd + dff + c, dg[0], dg[1], dg[2], dg[3]);
      } else {
        float b4[4] = {0.f, 0.f, 0.f, 0.f};
        if (bias)
          for (int j = 0; j < 4; ++j) b4[j] = __bfloat162float(bias[(size_t)g * dff + c + j]);
        float4 da;
        gelu_bwd(x0.x + b4[0], up.x, da.x, hv[0]);
        gelu_bwd(x0.y + b4[1], up.y, da.y, hv[1]);
        gelu_bwd(x0.z + b4[2], up.z, da.z, hv[2]);
        gelu_bwd(x0.w + b4[3], up.w, da.w, hv[3]);
        *reinterpret_cast<float4*>(p0 + i) = da;
        st_bf16x4(D + (size_t)r * ldd + c, da.x, da.y, da.z, da.w);
      }
      st_bf16x4(h + i, hv[0], hv[1], hv[2], hv[3]);
    }
  }
}

// koff[g] = sum over g' < g of the rows of g' rounded up to 64: each group's first column in the
// transposed copies that the weight gradients contract over.
__global__ void k_pad_offsets(const int32_t* __restrict__ off, int G, int32_t* __restrict__ koff) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int run = 0;
  koff[0] = 0;
  for (int g = 0; g < G; ++g) {
    run += (off[g + 1] - off[g] + 63) & ~63;
    koff[g + 1] = run;
  }
}

// out [C][Kp]: padded column p of group g (koff[g] <= p < koff[g+1]) holds row off[g] + p - koff[g]
// of in [rows][ldi] while that row is the group's, else zero.  off / koff NULL: one group of `rows`
// rows, padded to a multiple of 64.  A block moves 64 padded columns x 128 channels: 16-byte loads
// of 8 channels of a row (all four issued before the shared-memory writes), bf16 pairs in shared
// memory, 16-byte stores of 8 padded columns of a channel (C, ldi a multiple of 8; Kp of 64; each
// block's 64 columns lie in one group).
__global__ void __launch_bounds__(256) k_transpose_pad(const __nv_bfloat16* __restrict__ in, int64_t ldi, int C,
                                                       const int32_t* __restrict__ off,
                                                       const int32_t* __restrict__ koff, int G, int rows,
                                                       __nv_bfloat16* __restrict__ out, int64_t Kp) {
  __shared__ uint32_t tw[64][65];  // [padded column][channel pair]
  __shared__ int s_r0, s_hi, s_live;
  const int p0 = blockIdx.x * 64, c0 = blockIdx.y * 128;
  const int tid = threadIdx.y * 32 + threadIdx.x;
  if (tid == 0) {
    int live = 0, r0 = 0, hi = 0;
    if (off) {
      if (p0 < koff[G]) {
        int lo = 0, h = G - 1;  // the last group starting at or before p0
        while (lo < h) {
          const int mid = (lo + h + 1) >> 1;
          if (koff[mid] <= p0) lo = mid;
          else h = mid - 1;
        }
        live = 1;
        r0 = off[lo] + (p0 - koff[lo]);
        hi = off[lo + 1];
      }
    } else if (p0 < ((rows + 63) & ~63)) {
      live = 1;
      r0 = p0;
      hi = rows;
    }
    s_live = live;
    s_r0 = r0;
    s_hi = hi;
  }
  __syncthreads();
  if (!s_live) return;
  const int r0 = s_r0, hi = s_hi;
  const int cc = (tid & 15) * 8;  // this thread's 8 channels of a row
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = i * 16 + (tid >> 4), r = r0 + rl;
    v[i] = (r < hi && c0 + cc < C) ? *reinterpret_cast<const uint4*>(in + (size_t)r * ldi + c0 + cc)
                                   : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = i * 16 + (tid >> 4);
    tw[rl][cc / 2 + 0] = v[i].x;
    tw[rl][cc / 2 + 1] = v[i].y;
    tw[rl][cc / 2 + 2] = v[i].z;
    tw[rl][cc / 2 + 3] = v[i].w;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int o = i * 256 + tid;
    const int ch = o >> 3, pc = o & 7;  // channel of the tile, 8-column chunk of the output row
    const int c = c0 + ch;
    if (c >= C) continue;
    const int j = ch >> 1, sh = (ch & 1) * 16;
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) w[q] = (tw[8 * pc + q][j] >> sh) & 0xFFFFu;
    const uint4 pk = make_uint4(w[0] | (w[1] << 16), w[2] | (w[3] << 16), w[4] | (w[5] << 16), w[6] | (w[7] << 16));
    *reinterpret_cast<uint4*>(out + (size_t)c * Kp + p0 + 8 * pc) = pk;
  }
}

// dst [G, n] = the column sums of each group's rows of src [rows, ld] (rows summed in order).
template <typename T>
__global__ void __launch_bounds__(256) k_group_colsum(const T* __restrict__ src, int64_t ld,
                                                      const int32_t* __restrict__ off, int n,
                                                      float* __restrict__ dst) {
  const int g = blockIdx.y, c = blockIdx.x * 256 + threadIdx.x;
  if (c >= n) return;
  float s = 0.f;
  for (int r = off[g]; r < off[g + 1]; ++r) s += to_f(src[(size_t)r * ld + c]);
  dst[(size_t)g * n + c] = s;
}

// dx [T, d] += the input gradients of each token's kept rows, in slot order.
__global__ void __launch_bounds__(256) k_scatter_rows_add(const float* __restrict__ dxp,
                                                          const int32_t* __restrict__ row_of, int k, int d,
                                                          float* __restrict__ dx) {
  const int t = blockIdx.x;
  int rows[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) rows[j] = j < k ? row_of[(size_t)t * k + j] : -1;
  for (int c = threadIdx.x; c < d; c += 256) {
    float v = dx[(size_t)t * d + c];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (rows[j] >= 0) v += dxp[(size_t)rows[j] * d + c];
    dx[(size_t)t * d + c] = v;
  }
}

// The expert FFN backward of one set of rows: G groups of rows (the routed experts over the
// permuted rows, by off) or one plain problem of `rows` rows (a shared expert, off == NULL), the
// weights of group g at g * (dff d).  xr [rows, d] the FFN inputs, dyr [rows, d] the upstream
// gradients of its outputs.  Writes dW_up, dW_gate, dW_down (and the bias gradients) of every
// group, and dxr = du W_up + dg W_gate (beta_dx = 1: added to dxr).  s0, s1, s2 [rows, dff] fp32.
template <typename T>
cudaError_t ffn_bwd_rows(int act, const T* xr, const T* dyr, const int32_t* off, int G, int rows_bound, int d,
                         int dff, const T* wu, const T* wg, const T* wd, const T* bu, float* dwu, float* dwg,
                         float* dwd, float* dbu, float* dbd, float* dxr, int beta_dx, float* s0, float* s1,
                         float* s2, cudaStream_t st) {
  const bool glu = act == ACT_SWIGLU;
  const int64_t wstride = (int64_t)dff * d;
  const GemmGroups on_m{off, 0, wstride, 0, 0}, on_k{off, 1, 0, wstride, 0};
  const GemmGroups on_m_acc{off, 0, wstride, 0, 1};
  const GemmGroups plain{nullptr, 0, 0, 0, 0}, plain_acc{nullptr, 0, 0, 0, 1};
  const bool grouped = off != nullptr;
  // pre-activations (fp32, K = d in order): u or a = xr W_up^T, g = xr W_gate^T; dh = dyr W_down
  float* pu = glu ? s1 : s0;
  cudaError_t e = sgemm<T, T, true, false>(xr, d, wu, d, pu, dff, rows_bound, dff, d, st, grouped ? on_m : plain, G);
  if (e == cudaSuccess && glu)
    e = sgemm<T, T, true, false>(xr, d, wg, d, s0, dff, rows_bound, dff, d, st, grouped ? on_m : plain, G);
  if (e == cudaSuccess)
    e = sgemm<T, T, true, true>(dyr, d, wd, dff, s2, dff, rows_bound, dff, d, st, grouped ? on_m : plain, G);
  if (e != cudaSuccess) return e;
  const dim3 eg(grouped ? 64 : 592, G);
  if (glu)
    k_act_bwd<ACT_SWIGLU, T><<<eg, 256, 0, st>>>(s0, s1, s2, nullptr, off, rows_bound, dff);
  else
    k_act_bwd<ACT_GELU, T><<<eg, 256, 0, st>>>(s0, nullptr, s2, bu, off, rows_bound, dff);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dbu) {  // biases: routed GELU experts only
    k_group_colsum<float><<<dim3((dff + 255) / 256, G), 256, 0, st>>>(s0, dff, off, dff, dbu);
    k_group_colsum<T><<<dim3((d + 255) / 256, G), 256, 0, st>>>(dyr, d, off, d, dbd);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // weight gradients (K = the group's rows, in row order): dW_down = dyr^T h, dW_up = du^T xr,
  // dW_gate = dg^T xr
  const int kr = grouped ? 0 : rows_bound;
  e = sgemm<T, float, false, true>(dyr, d, s2, dff, dwd, dff, d, dff, kr, st, grouped ? on_k : plain, G);
  if (e == cudaSuccess)
    e = sgemm<float, T, false, true>(pu, dff, xr, d, dwu, d, dff, d, kr, st, grouped ? on_k : plain, G);
  if (e == cudaSuccess && glu)
    e = sgemm<float, T, false, true>(s0, dff, xr, d, dwg, d, dff, d, kr, st, grouped ? on_k : plain, G);
  if (e != cudaSuccess) return e;
  // input gradient (K = dff in order): dxr (+)= du W_up, then + dg W_gate
  e = sgemm<float, T, true, true>(pu, dff, wu, d, dxr, d, rows_bound, d, dff, st,
                                  grouped ? (beta_dx ? on_m_acc : on_m) : (beta_dx ? plain_acc : plain), G);
  if (e == cudaSuccess && glu)
    e = sgemm<float, T, true, true>(s0, dff, wg, d, dxr, d, rows_bound, d, dff, st, grouped ? on_m_acc : plain_acc,
                                    G);
  return e;
}

template <typename T>
cudaError_t expert_bwd_t(const ExpertBackward& b, cudaStream_t st) {
  const T* x = static_cast<const T*>(b.x);
  const T* dy = static_cast<const T*>(b.dy);
  cudaError_t e = cudaMemsetAsync(b.status, 0, sizeof(uint32_t), st);  // no bounded waits on this path
  if (e != cudaSuccess) return e;
  if (b.rows_bound > 0) {
    e = ffn_bwd_rows<T>(b.act, static_cast<const T*>(b.x_perm), static_cast<const T*>(b.dy_perm), b.offsets, b.E,
                        b.rows_bound, b.d, b.dff, static_cast<const T*>(b.w_up), static_cast<const T*>(b.w_gate),
                        static_cast<const T*>(b.w_down), static_cast<const T*>(b.b_up), b.dw_up, b.dw_gate,
                        b.dw_down, b.db_up, b.db_down, b.dx_perm, 0, b.s0, b.s1, b.s2, st);
    if (e != cudaSuccess) return e;
    k_scatter_rows_add<<<b.T, 256, 0, st>>>(b.dx_perm, b.row_of, b.k, b.d, b.dx);
    e = cudaGetLastError();
  } else {  // nothing routed: every expert's gradient is zero
    const size_t wsz = sizeof(float) * (size_t)b.E * b.dff * b.d;
    e = cudaMemsetAsync(b.dw_up, 0, wsz, st);
    if (e == cudaSuccess && b.dw_gate) e = cudaMemsetAsync(b.dw_gate, 0, wsz, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.dw_down, 0, wsz, st);
    if (e == cudaSuccess && b.db_up) e = cudaMemsetAsync(b.db_up, 0, sizeof(float) * (size_t)b.E * b.dff, st);
    if (e == cudaSuccess && b.db_down) e = cudaMemsetAsync(b.db_down, 0, sizeof(float) * (size_t)b.E * b.d, st);
  }
  // shared experts: every token, weight 1, added to dx one expert after another
  const size_t sw = (size_t)b.dff * b.d;
  for (int s = 0; s < b.n_shared && e == cudaSuccess; ++s) {
    if (b.T == 0) {
      e = cudaMemsetAsync(b.dws_up + s * sw, 0, sizeof(float) * sw, st);
      if (e == cudaSuccess && b.dws_gate) e = cudaMemsetAsync(b.dws_gate + s * sw, 0, sizeof(float) * sw, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(b.dws_down + s * sw, 0, sizeof(float) * sw, st);
      continue;
    }
    e = ffn_bwd_rows<T>(b.act, x, dy, nullptr, 1, b.T, b.d, b.dff, static_cast<const T*>(b.ws_up) + s * sw,
                        b.ws_gate ? static_cast<const T*>(b.ws_gate) + s * sw : nullptr,
                        static_cast<const T*>(b.ws_down) + s * sw, nullptr, b.dws_up + s * sw,
                        b.dws_gate ? b.dws_gate + s * sw : nullptr, b.dws_down + s * sw, nullptr, nullptr, b.dx, 1,
                        b.s0, b.s1, b.s2, st);
  }
  return e;
}
// bf16 layers: every contraction on the tensor cores (k_gemm_bwd) with fp32 accumulation; the
// operands the backward creates (du, dg or da, h and the transposed copies) are rounded to bf16.
// The weights are read as stored (K-major for the recomputed pre-activations, N-major for dh and
// dx); the weight gradients contract over the rows, so their operands are transposed per expert.
// One FFN backward over G groups of rows (off) or one plain problem of `rows` rows (off == NULL).
cudaError_t ffn_bwd_tc(const ExpertBackward& b, bool glu, const __nv_bfloat16* xr, const __nv_bfloat16* dyr,
                       const int32_t* off, int G, int rows_alloc, int rows, const __nv_bfloat16* wu,
                       const __nv_bfloat16* wg, const __nv_bfloat16* wd, const __nv_bfloat16* bu, float* dwu,
                       float* dwg, float* dwd, float* dbu, float* dbd, float* dxr, int beta_dx, cudaStream_t st) {
  const int d = b.d, f = b.dff, Kd = glu ? 2 * f : f;
  const int Gw = off ? G : 1;
  const dim3 tb(32, 8);
  // pre-activations g (or a) into s0, u into s1 (W [f][d]: K-major as stored); dh = dy W_down into
  // s2 (W_down [d][f] read N-major)
  cudaError_t e = launch_gemm_bwd_rows_m(xr, rows_alloc, glu ? wg : wu, Gw, f, d, off, G, rows, b.s0, f, 0, b.status, st);
  if (e == cudaSuccess && glu)
    e = launch_gemm_bwd_rows_m(xr, rows_alloc, wu, Gw, f, d, off, G, rows, b.s1, f, 0, b.status, st);
  if (e == cudaSuccess)
    e = launch_gemm_bwd_rows_m_nmajor(dyr, rows_alloc, wd, nullptr, d, Gw, f, d, off, G, rows, b.s2, f, 0, b.status,
                                      st, true);
  if (e != cudaSuccess) return e;
  const dim3 eg(off ? 64 : 592, off ? G : 1);
  if (glu)
    k_act_bwd_tc<ACT_SWIGLU><<<eg, 256, 0, st>>>(b.s0, b.s1, b.s2, nullptr, off, rows, f, b.D, Kd, b.h);
  else
    k_act_bwd_tc<ACT_GELU><<<eg, 256, 0, st>>>(b.s0, nullptr, b.s2, bu, off, rows, f, b.D, Kd, b.h);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (dbu) {
    k_group_colsum<float><<<dim3((f + 255) / 256, G), 256, 0, st>>>(b.s0, f, off, f, dbu);
    k_group_colsum<__nv_bfloat16><<<dim3((d + 255) / 256, G), 256, 0, st>>>(dyr, d, off, d, dbd);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // input gradient du W_up + dg W_gate: one contraction over K = Kd of [du | dg], the weights
  // [f][d] read N-major (W_up for k < f, W_gate beyond)
  e = launch_gemm_bwd_rows_m_nmajor(b.D, rows_alloc, wu, glu ? wg : nullptr, f, Gw, d, Kd, off, G, rows, dxr, d,
                                    beta_dx, b.status, st, true);
  if (e != cudaSuccess) return e;
  // weight gradients over each group's rows: transposed copies, each group zero-padded to 64
  const int32_t* koff = nullptr;
  if (off) {
    k_pad_offsets<<<1, 32, 0, st>>>(off, G, b.koff);
    koff = b.koff;
  }
  const int64_t Kp = b.Kp;
  const int pad_cols = off ? (int)Kp : ((rows + 63) & ~63);
  const unsigned px = (unsigned)(pad_cols / 64);
  k_transpose_pad<<<dim3(px, (Kd + 127) / 128), tb, 0, st>>>(b.D, Kd, Kd, off, koff, G, rows, b.DT, Kp);
  k_transpose_pad<<<dim3(px, (f + 127) / 128), tb, 0, st>>>(b.h, f, f, off, koff, G, rows, b.hT, Kp);
  k_transpose_pad<<<dim3(px, (d + 127) / 128), tb, 0, st>>>(xr, d, d, off, koff, G, rows, b.xT, Kp);
  k_transpose_pad<<<dim3(px, (d + 127) / 128), tb, 0, st>>>(dyr, d, d, off, koff, G, rows, b.dyT, Kp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int cols = (rows + 63) & ~63;
  e = launch_gemm_bwd_rows_k(b.dyT, d, b.hT, f, (int)Kp, koff, G, cols, dwd, f, (int64_t)d * f, 0, b.status, st);
  if (e == cudaSuccess)
    e = launch_gemm_bwd_rows_k(b.DT, f, b.xT, d, (int)Kp, koff, G, cols, dwu, d, (int64_t)f * d, 0, b.status, st);
  if (e == cudaSuccess && glu)
    e = launch_gemm_bwd_rows_k(b.DT + (size_t)f * Kp, f, b.xT, d, (int)Kp, koff, G, cols, dwg, d, (int64_t)f * d, 0,
                               b.status, st);
  return e;
}

cudaError_t expert_bwd_tc(const ExpertBackward& b, cudaStream_t st) {
  using bf = __nv_bfloat16;
  const bool glu = b.act == ACT_SWIGLU;
  cudaError_t e = cudaMemsetAsync(b.status, 0, sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  if (b.rows_bound > 0) {
    e = ffn_bwd_tc(b, glu, static_cast<const bf*>(b.x_perm), static_cast<const bf*>(b.dy_perm), b.offsets, b.E,
                   b.rows_alloc, 0, static_cast<const bf*>(b.w_up), static_cast<const bf*>(b.w_gate),
                   static_cast<const bf*>(b.w_down), static_cast<const bf*>(b.b_up), b.dw_up, b.dw_gate, b.dw_down,
                   b.db_up, b.db_down, b.dx_perm, 0, st);
    if (e != cudaSuccess) return e;
    k_scatter_rows_add<<<b.T, 256, 0, st>>>(b.dx_perm, b.row_of, b.k, b.d, b.dx);
    e = cudaGetLastError();
  } else {
    const size_t wsz = sizeof(float) * (size_t)b.E * b.dff * b.d;
    e = cudaMemsetAsync(b.dw_up, 0, wsz, st);
    if (e == cudaSuccess && b.dw_gate) e = cudaMemsetAsync(b.dw_gate, 0, wsz, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.dw_down, 0, wsz, st);
    if (e == cudaSuccess && b.db_up) e = cudaMemsetAsync(b.db_up, 0, sizeof(float) * (size_t)b.E * b.dff, st);
    if (e == cudaSuccess && b.db_down) e = cudaMemsetAsync(b.db_down, 0, sizeof(float) * (size_t)b.E * b.d, st);
  }
  const size_t sw = (size_t)b.dff * b.d;
  for (int s = 0; s < b.n_shared && e == cudaSuccess; ++s) {
    if (b.T == 0) {
      e = cudaMemsetAsync(b.dws_up + s * sw, 0, sizeof(float) * sw, st);
      if (e == cudaSuccess && b.dws_gate) e = cudaMemsetAsync(b.dws_gate + s * sw, 0, sizeof(float) * sw, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(b.dws_down + s * sw, 0, sizeof(float) * sw, st);
      continue;
    }
    e = ffn_bwd_tc(b, glu, static_cast<const bf*>(b.x), static_cast<const bf*>(b.dy), nullptr, 1, b.T, b.T,
                   static_cast<const bf*>(b.ws_up) + s * sw, glu ? static_cast<const bf*>(b.ws_gate) + s * sw : nullptr,
                   static_cast<const bf*>(b.ws_down) + s * sw, nullptr, b.dws_up + s * sw,
                   glu ? b.dws_gate + s * sw : nullptr, b.dws_down + s * sw, nullptr, nullptr, b.dx, 1, st);
  }
  return e;
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
                                   float* dwr, float* dx, const RouterBwdScratch* sc, cudaStream_t st) {
  if (E < 1 || E > 256 || k < 1 || k > 8 || k > E) return cudaErrorInvalidValue;
  if (sc && bf16 && T > 0)
    return router_bwd_tc(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(wr), lbias, idx, tw,
                         counts, dw, T, d, E, k, inv_tau, lb_coef, z_coef, dlb, dzl, dz, dwr, dx, *sc, st);
  if (bf16)
    return router_bwd_t<__nv_bfloat16>(x, wr, lbias, idx, tw, counts, dw, T, d, E, k, inv_tau, lb_coef, z_coef, dlb,
                                       dzl, dz, dwr, dx, st);
  return router_bwd_t<float>(x, wr, lbias, idx, tw, counts, dw, T, d, E, k, inv_tau, lb_coef, z_coef, dlb, dzl, dz,
                             dwr, dx, st);
}

cudaError_t launch_expert_backward(bool bf16, const ExpertBackward& b, cudaStream_t st) {
  if (b.k < 1 || b.k > 8) return cudaErrorInvalidValue;
  return bf16 ? expert_bwd_tc(b, st) : expert_bwd_t<float>(b, st);
}

}  // namespace moe
