// Per-expert counts and the two auxiliary losses from the router's per-block partials, in one
// fixed order.  Both the router's last CTA (a router call on its own) and the fused dispatch
// kernel (a whole layer) call this, so the two give bit-identical counts and losses.
//
// The load-balance loss is alpha E sum_e f_e P_e with f_e = c_e / (T k) and P_e the mean router
// probability of expert e (the OpenMythos article, sec. 3.1); the z-loss is beta mean_t lse_t^2
// with the coefficient the FLAME-MoE summary, sec. 2, gives.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kLossParts = 8;

struct LossScratch {
  int lcnt[kLossParts][256];   // per-slice counts
  float lps[kLossParts][256];  // per-slice sums of P
  float lbterm[256];           // c_e * sum_t P_te
  float zsum;
};

// Block slices per expert: a power of two, at most 8, with 2 * parts * E <= 256.
__device__ __forceinline__ int loss_parts(int E) {
  int parts = 1;
  while (parts < kLossParts && 2 * parts * E <= 256) parts <<= 1;
  return parts;
}

template <bool GLOBAL>
__device__ __forceinline__ int load_i(const int32_t* p) {
  return GLOBAL ? __ldcg(p) : *p;
}
template <bool GLOBAL>
__device__ __forceinline__ float load_f(const float* p) {
  return GLOBAL ? __ldcg(p) : *p;
}

// 256 threads.  hist / psum: per-block partials [nb][E] (HIST_GLOBAL, PSUM_GLOBAL: in global memory,
// read through L2; else in shared memory); lse2: per-block sums of lse^2 [nb] in global memory.
// Expert e's blocks are cut into `parts` slices with fixed boundaries; each slice is summed in block
// order, the slices in slice order, the experts lane-strided then by a butterfly; all in fp32 (sums
// of <= 256 expert terms and of the per-block z partials stay within ~1e-5 relative, and B300's
// narrow FP64 pipe made a few dependent FP64 operations cost microseconds).  Writes cnt[e] (shared,
// may be null), counts[e] (global, may be null) and losses[0..1]; ends with __syncthreads.
template <bool HIST_GLOBAL, bool PSUM_GLOBAL>
__device__ void route_losses(const int32_t* hist, const float* psum, const float* lse2, int nb, int E, int k, int T,
                             float lb_coef, float z_coef, int* cnt, int32_t* counts, float* losses, LossScratch& sc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int parts = loss_parts(E);
  {
    const int e = tid % E, part = tid / E;
    if (part < parts) {
      const int b_lo = (int)((long)nb * part / parts), b_hi = (int)((long)nb * (part + 1) / parts);
      int c = 0;
      float ps = 0.f;
      constexpr int U = 8;  // loads in flight per thread
      for (int b0 = b_lo; b0 < b_hi; b0 += U) {
        int hv[U];
        float pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool in = b0 + u < b_hi;
          hv[u] = in ? load_i<HIST_GLOBAL>(hist + (size_t)(b0 + u) * E + e) : 0;
          pv[u] = in ? load_f<PSUM_GLOBAL>(psum + (size_t)(b0 + u) * E + e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          c += hv[u];
          ps += pv[u];
        }
      }
      sc.lps[part][e] = ps;
      sc.lcnt[part][e] = c;
    }
  }
  float l = 0.f;
  if (warp == 1) {
    for (int b = lane; b < nb; b += 32) l += __ldcg(lse2 + b);
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int c = 0;
    float ps = 0.f;
    for (int part = 0; part < parts; ++part) {
      c += sc.lcnt[part][e];
      ps += sc.lps[part][e];
    }
    if (cnt) cnt[e] = c;
    if (counts) counts[e] = c;
    sc.lbterm[e] = (float)c * ps;
  }
  if (warp == 1) {
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) sc.zsum = l;
  }
  __syncthreads();
  if (warp == 0) {
    float lb = 0.f;
    for (int e = lane; e < E; e += 32) lb += sc.lbterm[e];
#pragma unroll
    for (int o = 16; o; o >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, o);
    if (lane == 0) {
      const float Tn = (float)T;
      // lb = alpha E sum_e (c_e / (T k)) (psum_e / T);  zl = beta mean_t lse_t^2
      losses[0] = lb_coef * (float)E * (lb / (Tn * Tn * (float)k));
      losses[1] = z_coef * (sc.zsum / Tn);
    }
  }
  __syncthreads();
}

}  // namespace moe
