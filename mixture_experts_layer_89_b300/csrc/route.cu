// Fused router: logits (fp32 accumulation), softmax, top-k with renormalised weights, per-CTA
// expert histograms and the partial sums the auxiliary losses need.
//
// Follows the router of the mini-moe tutorial, sec. 3.1 (bias-free Linear -> softmax -> top-k ->
// renormalise) and the OpenMythos article, sec. 3.1 (routing pseudo-code, load-balance loss);
// the router z-loss is the one the FLAME-MoE summary, sec. 2, names.
//
// One CTA of 256 threads owns 32 tokens.  Phase 1 is a register-tiled fp32 GEMM over d in chunks
// of 32 staged in shared memory (each thread: 2 tokens x NI experts).  Phase 2 gives each warp
// whole tokens: the E logits of a token are spread over the lanes, max/sum/argmax are warp
// shuffles.  Top-k selects by logit (ties -> lower index), weights = exp(z_j - max) / sum over
// the selected, which equals P_j / sum P_selected.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int RT = kRouteTokens;
constexpr int RDC = 32;
constexpr int RTHREADS = 256;
constexpr float kBadLogit = -3.0e38f;

template <typename T, int NI>
__global__ void __launch_bounds__(RTHREADS)
    k_route(const T* __restrict__ x, const T* __restrict__ wr, const float* __restrict__ lbias, int Tn, int d, int E,
            int k, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ hist,
            float* __restrict__ psum, float* __restrict__ lse2, uint32_t* status, float inv_tau) {
  extern __shared__ float sm[];
  float* xs = sm;                      // [RT][RDC+1]
  float* wsm = xs + RT * (RDC + 1);    // [E][RDC+1]
  float* lg = wsm + E * (RDC + 1);     // [RT][E+1]  logits, then probabilities
  float* lse_s = lg + RT * (E + 1);    // [RT]
  int* hist_s = reinterpret_cast<int*>(lse_s + RT);  // [E]

  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RT;
  const int ty = tid >> 4, tx = tid & 15;
  for (int e = tid; e < E; e += RTHREADS) hist_s[e] = 0;

  float acc0[NI], acc1[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) acc0[i] = acc1[i] = 0.f;

  for (int c0 = 0; c0 < d; c0 += RDC) {
    for (int i = tid; i < RT * RDC; i += RTHREADS) {
      const int r = i / RDC, c = i % RDC, t = t0 + r, dc = c0 + c;
      xs[r * (RDC + 1) + c] = (t < Tn && dc < d) ? to_f(x[(size_t)t * d + dc]) : 0.f;
    }
    for (int i = tid; i < E * RDC; i += RTHREADS) {
      const int e = i / RDC, c = i % RDC, dc = c0 + c;
      wsm[e * (RDC + 1) + c] = dc < d ? to_f(wr[(size_t)e * d + dc]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < RDC; ++c) {
      const float a0 = xs[ty * (RDC + 1) + c];
      const float a1 = xs[(ty + 16) * (RDC + 1) + c];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int e = tx + 16 * i;
        const float w = (e < E) ? wsm[e * (RDC + 1) + c] : 0.f;
        acc0[i] = fmaf(a0, w, acc0[i]);
        acc1[i] = fmaf(a1, w, acc1[i]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = tx + 16 * i;
    if (e < E) {
      const float b = lbias ? lbias[e] : 0.f;
      lg[ty * (E + 1) + e] = acc0[i] + b;
      lg[(ty + 16) * (E + 1) + e] = acc1[i] + b;
    }
  }
  __syncthreads();

  // ---- phase 2: one warp per token
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < RT; r += RTHREADS / 32) {
    const int t = t0 + r;
    if (t >= Tn) continue;
    float v[8];
    bool bad = false;
    float m = kBadLogit;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      float z = kBadLogit;
      if (e < E) {
        z = lg[r * (E + 1) + e];
        if (!isfinite(z)) {
          bad = true;
          z = kBadLogit;
        }
      }
      v[i] = z;
      m = fmaxf(m, z);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < E) s += expf((v[i] - m) * inv_tau);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv_s = 1.f / s;

    uint32_t taken = 0;
    int my_e = 0;
    float my_p = 0.f, selsum = 0.f;
    for (int j = 0; j < k; ++j) {
      float bv = -FLT_MAX;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      const float p = expf((bv - m) * inv_tau);
      selsum += p;
      if (lane == j) {
        my_e = be;
        my_p = p;
      }
    }
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_e;
      topk_w[(size_t)t * k + lane] = my_p / selsum;
      atomicAdd(&hist_s[my_e], 1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) lg[r * (E + 1) + e] = expf((v[i] - m) * inv_tau) * inv_s;
    }
    if (lane == 0) {
      lse_s[r] = m * inv_tau + logf(s);
      if (bad) atomicOr(status, DEV_NONFINITE);
    }
  }
  __syncthreads();

  // ---- per-CTA partials, summed in token order (deterministic)
  const int nvalid = min(RT, Tn - t0);
  for (int e = tid; e < E; e += RTHREADS) {
    float ps = 0.f;
    for (int r = 0; r < nvalid; ++r) ps += lg[r * (E + 1) + e];
    psum[(size_t)blockIdx.x * E + e] = ps;
    hist[(size_t)blockIdx.x * E + e] = hist_s[e];
  }
  if (tid == 0) {
    float l2 = 0.f;
    for (int r = 0; r < nvalid; ++r) l2 += lse_s[r] * lse_s[r];
    lse2[blockIdx.x] = l2;
  }
}

// Sums the per-CTA partials in a fixed order: counts, then both losses (accumulated in double).
__global__ void __launch_bounds__(256) k_route_finalize(const int32_t* __restrict__ hist,
                                                        const float* __restrict__ psum,
                                                        const float* __restrict__ lse2, int nb, int Tn, int E, int k,
                                                        float lb_coef, float z_coef, int32_t* __restrict__ counts,
                                                        float* __restrict__ losses) {
  __shared__ double red[256];
  __shared__ double lbterm[256];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += 256) {
    int c = 0;
    double p = 0.0;
    for (int b = 0; b < nb; ++b) {
      c += hist[(size_t)b * E + e];
      p += (double)psum[(size_t)b * E + e];
    }
    counts[e] = c;
    lbterm[e] = (double)c * p;
  }
  double l = 0.0;
  for (int b = tid; b < nb; b += 256) l += (double)lse2[b];
  red[tid] = l;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  if (tid == 0) {
    double lb = 0.0;
    for (int e = 0; e < E; ++e) lb += lbterm[e];
    if (Tn > 0) {
      // lb = alpha E sum_e (c_e / (T k)) (psum_e / T)
      losses[0] = (float)((double)lb_coef * E * lb / ((double)Tn * k * (double)Tn));
      losses[1] = (float)((double)z_coef * red[0] / (double)Tn);
    } else {
      losses[0] = 0.f;
      losses[1] = 0.f;
    }
  }
}

template <typename T, int NI>
cudaError_t launch_route_t(const void* x, const void* wr, const float* lbias, int Tn, int d, int E, int k,
                           int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2, uint32_t* status,
                           cudaStream_t st, float inv_tau) {
  const size_t smem = sizeof(float) * ((size_t)RT * (RDC + 1) + (size_t)E * (RDC + 1) + (size_t)RT * (E + 1) + RT) +
                      sizeof(int) * (size_t)E;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(k_route<T, NI>), smem);
  if (err != cudaSuccess) return err;
  k_route<T, NI><<<route_blocks(Tn), RTHREADS, smem, st>>>(static_cast<const T*>(x), static_cast<const T*>(wr), lbias,
                                                            Tn, d, E, k, topk_idx, topk_w, hist, psum, lse2, status,
                                                            inv_tau);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_route_dispatch_ni(const void* x, const void* wr, const float* lbias, int Tn, int d, int E, int k,
                                     int32_t* ti, float* tw, int32_t* hist, float* psum, float* lse2, uint32_t* status,
                                     cudaStream_t st, float inv_tau) {
  if (E <= 16) return launch_route_t<T, 1>(x, wr, lbias, Tn, d, E, k, ti, tw, hist, psum, lse2, status, st, inv_tau);
  if (E <= 32) return launch_route_t<T, 2>(x, wr, lbias, Tn, d, E, k, ti, tw, hist, psum, lse2, status, st, inv_tau);
  if (E <= 64) return launch_route_t<T, 4>(x, wr, lbias, Tn, d, E, k, ti, tw, hist, psum, lse2, status, st, inv_tau);
  if (E <= 128) return launch_route_t<T, 8>(x, wr, lbias, Tn, d, E, k, ti, tw, hist, psum, lse2, status, st, inv_tau);
  return launch_route_t<T, 16>(x, wr, lbias, Tn, d, E, k, ti, tw, hist, psum, lse2, status, st, inv_tau);
}
}  // namespace

int route_blocks(int T) { return (T + RT - 1) / RT; }

cudaError_t launch_route(bool bf16, const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                         int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2, uint32_t* status,
                         cudaStream_t st, float inv_tau) {
  if (T <= 0) return cudaSuccess;
  if (bf16)
    return launch_route_dispatch_ni<__nv_bfloat16>(x, wr, lbias, T, d, E, k, topk_idx, topk_w, hist, psum, lse2,
                                                   status, st, inv_tau);
  return launch_route_dispatch_ni<float>(x, wr, lbias, T, d, E, k, topk_idx, topk_w, hist, psum, lse2, status, st,
                                         inv_tau);
}

cudaError_t launch_route_finalize(const int32_t* hist, const float* psum, const float* lse2, int nb, int T, int E,
                                  int k, float lb_coef, float z_coef, int32_t* counts, float* losses,
                                  cudaStream_t st) {
  k_route_finalize<<<1, 256, 0, st>>>(hist, psum, lse2, nb, T, E, k, lb_coef, z_coef, counts, losses);
  return cudaGetLastError();
}

}  // namespace moe
