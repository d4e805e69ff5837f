// Router of bf16 layers for decode-sized batches (T <= kSmallRouteTokens): the same results as
// the tensor-core router -- top-k indices and renormalised weights, the router's per-block
// partials and, for a router call on its own, counts and both losses (route_losses.cuh) -- for a
// batch too small to fill the tensor-core router's 128-token tile.
//
// The router is the bias-free Linear -> softmax -> top-k -> renormalise of the mini-moe tutorial,
// sec. 3.1 (MoELayer), with the losses of the OpenMythos article, sec. 3.1, and the FLAME-MoE
// summary, sec. 2.  A 128-token tile holding a few tokens leaves the tensor-core router one CTA
// (or one cluster) and a serial epilogue; here every (token, expert) logit is its own warp's fp32
// dot product of two bf16 rows (the products are exact in fp32), with a rigorous bound on its
// rounding error.  Where two of a token's leading k + 1 logits lie within their bounds of each
// other, that token's logits are recomputed with compensated (Neumaier) sums, within a few ulp of
// the exact values, before selecting: the choice and order of the k experts are those of the exact
// logits up to ties closer than that.  One CTA per token computes its logits and selects; the last
// CTA to finish reduces.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "route_losses.cuh"

namespace moe {

namespace {
constexpr float kBad = -3.0e38f;

// One step of Neumaier's compensated summation: s + c carries the running sum.
__device__ __forceinline__ void neumaier(float& s, float& c, float p) {
  const float t = __fadd_rn(s, p);
  c = __fadd_rn(c, fabsf(s) >= fabsf(p) ? __fadd_rn(__fsub_rn(s, t), p) : __fadd_rn(__fsub_rn(p, t), s));
  s = t;
}

// Compensated fp32 dot product of the token's row (shared memory) and a weight row (length d, a
// multiple of 8), one warp; every lane returns the same value.  Eight 16-byte loads per lane of the
// weight row are in flight together.
__device__ __forceinline__ float comp_dot_sx(const uint4* __restrict__ xs, const __nv_bfloat16* __restrict__ b, int d,
                                             int lane) {
  constexpr int U = 8;
  float s = 0.f, c = 0.f;
  for (int base = lane * 8; base < d; base += 256 * U) {
    uint4 bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 256;
      bv[u] = i < d ? __ldg(reinterpret_cast<const uint4*>(b + i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 256;
      const uint4 av = i < d ? xs[i >> 3] : make_uint4(0, 0, 0, 0);
      const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
      const uint32_t bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        neumaier(s, c, __fmul_rn(__uint_as_float(aw[j] << 16), __uint_as_float(bw[j] << 16)));
        neumaier(s, c, __fmul_rn(__uint_as_float(aw[j] & 0xffff0000u), __uint_as_float(bw[j] & 0xffff0000u)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
    const float t = __fadd_rn(s, s2);
    const float bp = __fsub_rn(t, s);
    const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(s2, bp));
    c = __fadd_rn(__fadd_rn(c, c2), err);
    s = t;
  }
  return __fadd_rn(s, c);
}

// Plain fp32 dot product of the token's row (shared memory) and a weight row, and the squared norm
// of the weight row; one warp, every lane returns both.  Each lane sums its d/32 exact bf16 x bf16
// products in order and five shuffle levels add the lanes, so the rounding error is at most
// (d/32 + 6) 2^-24 sum_i |x_i w_i| <= (d/32 + 6) 2^-24 ||x|| ||w|| (recursive summation, then
// Cauchy-Schwarz).
__device__ __forceinline__ float fast_dot_sx(const uint4* __restrict__ xs, const __nv_bfloat16* __restrict__ b, int d,
                                             int lane, float& nw2) {
  constexpr int U = 8;
  float s = 0.f, n = 0.f;
  for (int base = lane * 8; base < d; base += 256 * U) {
    uint4 bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 256;
      bv[u] = i < d ? __ldg(reinterpret_cast<const uint4*>(b + i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 256;
      const uint4 av = i < d ? xs[i >> 3] : make_uint4(0, 0, 0, 0);
      const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
      const uint32_t bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float b0 = __uint_as_float(bw[j] << 16), b1 = __uint_as_float(bw[j] & 0xffff0000u);
        s = fmaf(__uint_as_float(aw[j] << 16), b0, s);
        s = fmaf(__uint_as_float(aw[j] & 0xffff0000u), b1, s);
        n = fmaf(b0, b0, n);
        n = fmaf(b1, b1, n);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    n += __shfl_xor_sync(0xffffffffu, n, o);
  }
  nw2 = n;
  return s;
}

// One CTA per token, 1024 threads: warp w computes the logits of experts w, w + 32, ...; warp 0
// selects the top k (ties to the lower index), normalises the weights and the softmax of z / tau,
// and writes the token's probabilities and lse^2 to the workspace.  The last CTA to finish (a
// counter, zero between calls, reset by that CTA) reduces them in token order into the router's
// one-block partials (expert histogram, sums of P, sum of lse^2) and, with `finalize`, counts and
// losses by route_losses.
__global__ void __launch_bounds__(1024, 1) k_route_small(const __nv_bfloat16* __restrict__ x,
                                                      const __nv_bfloat16* __restrict__ wr,
                                                      const float* __restrict__ lbias, int Tn, int d, int E, int k,
                                                      float inv_tau, float* __restrict__ ptok,
                                                      float* __restrict__ l2tok, uint32_t* done,
                                                      int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                      int32_t* __restrict__ hist, float* __restrict__ psum,
                                                      float* __restrict__ lse2, int finalize,
                                                      int32_t* __restrict__ counts, float* __restrict__ losses,
                                                      float lb_coef, float z_coef, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float zs[256];
  __shared__ float zb[256];  // squared weight-row norms, then the logits' error bounds
  __shared__ float nx2_s;
  __shared__ int redo;
  __shared__ int h[256];
  __shared__ int is_last;
  __shared__ LossScratch sc;
  __shared__ float l2s[kSmallRouteTokens];
  extern __shared__ float pst[];  // last CTA: every token's probabilities [T][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  uint4* xs = reinterpret_cast<uint4*>(pst);  // the token's row (d bf16) before pst holds anything else
  for (int i = tid; i < d / 8; i += 1024) xs[i] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d) + i);
  __syncthreads();
  if (warp == 0) {  // |x|^2 of the token's row, for the logits' error bounds
    float nx = 0.f;
    for (int i = lane; i < d / 8; i += 32) {
      const uint4 a = xs[i];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(aw[j] << 16), hi = __uint_as_float(aw[j] & 0xffff0000u);
        nx = fmaf(lo, lo, fmaf(hi, hi, nx));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) nx += __shfl_xor_sync(0xffffffffu, nx, o);
    if (lane == 0) {
      nx2_s = nx;
      redo = 0;
    }
  }
  for (int e = warp; e < E; e += 32) {
    float nw2;
    const float v = fast_dot_sx(xs, wr + (size_t)e * d, d, lane, nw2);
    if (lane == 0) {
      zs[e] = __fadd_rn(v, lbias ? lbias[e] : 0.f);
      zb[e] = nw2;  // becomes the bound below
    }
  }
  __syncthreads();
  // error bound of each fp32 logit: (d/32 + 8) 2^-24 (||x|| ||w_e|| + |z_e|) (the last term covers
  // the bias addition), with 1 % slack for the rounding of the norms themselves
  const float gamma = (float)(d / 32 + 8) * 5.9604645e-8f * 1.01f;
  for (int e = tid; e < E; e += 1024) zb[e] = gamma * (sqrtf(nx2_s * zb[e]) + fabsf(zs[e]));
  __syncthreads();
  for (int pass = 0; pass < 2; ++pass) {
    if (warp == 0) do {
      float v[8];
      float m = kBad;
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        float zz = -FLT_MAX;
        if (e < E) {
          zz = zs[e];
          if (!isfinite(zz)) {
            bad = true;
            zz = kBad;
          }
        }
        v[i] = zz;
        m = fmaxf(m, zz);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (any_bad && lane == 0) atomicOr(status, DEV_NONFINITE);
      // top-k: k rounds of argmax, ties to the lower expert index
      uint32_t taken = 0;
      int my_e = 0;
      float my_v = 0.f, top = 0.f;
      float lead_v[9];  // the leading k + 1 logits in selection order, and their experts
      int lead_e[9];
      for (int j = 0; j < k + (k < E ? 1 : 0); ++j) {
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
        lead_v[j] = bv;
        lead_e[j] = be;
        if (j == k) break;  // the (k+1)-th: only for the near-tie check
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (j == 0) top = bv;
        if (lane == j) {
          my_e = be;
          my_v = bv;
        }
      }
      if (pass == 0 && !any_bad) {
        // the fp32 logits decide the order of the leading k + 1 only where neighbours lie further
        // apart than their two error bounds; else the token's logits are recomputed compensated
        bool near = false;
        for (int j = 0; j + 1 < k + (k < E ? 1 : 0); ++j)
          near = near || (lead_v[j] - lead_v[j + 1] <= zb[lead_e[j]] + zb[lead_e[j + 1]]);
        if (near) {
          if (lane == 0) redo = 1;
          continue;  // (warp-uniform) the exact pass decides
        }
      }
      // renormalised weights of the k (the softmax over the selected logits / tau)
      float wsum = 0.f;
      for (int j = 0; j < k; ++j) wsum += __expf((__shfl_sync(0xffffffffu, my_v, j) - top) * inv_tau);
      if (lane < k) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = __expf((my_v - top) * inv_tau) * (1.f / wsum);
      }
      // softmax over all E and lse, of z / tau
      float s = 0.f, p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        p[i] = lane + 32 * i < E ? __expf((v[i] - m) * inv_tau) : 0.f;
        s += p[i];
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const float inv_s = 1.f / s;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (lane + 32 * i < E) ptok[(size_t)t * E + lane + 32 * i] = p[i] * inv_s;
      if (lane == 0) {
        const float l = m * inv_tau + __logf(s);
        l2tok[t] = l * l;
      }
    } while (false);
    __syncthreads();
    if (!redo) break;
    for (int e = warp; e < E; e += 32) {  // near ties: the compensated logits decide
      const float v = comp_dot_sx(xs, wr + (size_t)e * d, d, lane);
      if (lane == 0) zs[e] = __fadd_rn(v, lbias ? lbias[e] : 0.f);
    }
    if (tid == 0) redo = 0;
    __syncthreads();
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(done, 1u) == (unsigned)Tn - 1) ? 1 : 0;
  __syncthreads();
  if (!is_last) return;
  // ---- last CTA: every token's results (staged into shared memory by all threads at once), then
  // summed in token order
  __threadfence();
  for (int e = tid; e < 256; e += 1024) h[e] = 0;
  for (int i = tid; i < Tn * E; i += 1024) pst[i] = __ldcg(ptok + i);
  for (int u = tid; u < Tn; u += 1024) l2s[u] = __ldcg(l2tok + u);
  __syncthreads();
  for (int a = tid; a < Tn * k; a += 1024) atomicAdd(&h[__ldcg(topk_idx + a)], 1);  // integers: order-free
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    float ps = 0.f;
    for (int u = 0; u < Tn; ++u) ps += pst[u * E + e];
    psum[e] = ps;
    hist[e] = h[e];
  }
  if (tid == 0) {
    float l2 = 0.f;
    for (int u = 0; u < Tn; ++u) l2 += l2s[u];
    lse2[0] = l2;
    *done = 0;  // ready for the next call
  }
  if (finalize) {
    __threadfence();
    __syncthreads();
    route_losses<true, true>(hist, psum, lse2, 1, E, k, Tn, lb_coef, z_coef, nullptr, counts, losses, sc);
  }
}
}  // namespace

cudaError_t launch_route_small(const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                               float inv_tau, float* ptok, float* l2tok, uint32_t* done, int32_t* topk_idx,
                               float* topk_w, int32_t* hist, float* psum, float* lse2, bool finalize, int32_t* counts,
                               float* losses, float lb_coef, float z_coef, uint32_t* status, cudaStream_t st) {
  if (T < 1 || T > kSmallRouteTokens || E < 1 || E > 256 || k < 1 || k > 8 || k > E || d % 8)
    return cudaErrorInvalidValue;
  // the token's row, then (last CTA) every token's probabilities
  const size_t smem = std::max(sizeof(float) * (size_t)T * E, sizeof(__nv_bfloat16) * (size_t)d);
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(k_route_small), smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_route_small, dim3(T), dim3(1024), smem, st, static_cast<const __nv_bfloat16*>(x),
                    static_cast<const __nv_bfloat16*>(wr), lbias, T, d, E, k, inv_tau, ptok, l2tok, done, topk_idx,
                    topk_w, hist, psum, lse2, finalize ? 1 : 0, counts, losses, lb_coef, z_coef, status);
}

}  // namespace moe
