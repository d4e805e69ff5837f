// Fused router of bf16 layers on the 5th-generation tensor cores: logits z = x W_r^T (+ logit
// bias) with fp32 accumulation, softmax, top-k with renormalised weights, per-expert counts and
// both auxiliary losses, in one launch.
//
// The router is the bias-free Linear -> softmax -> top-k -> renormalise of the mini-moe
// tutorial, sec. 3.1 (MoELayer) and the routing pseudo-code of the OpenMythos article, sec. 3.1;
// the load-balance loss is that article's alpha E sum_e f_e P_e, the z-loss the one the FLAME-MoE
// summary, sec. 2, names.  The logit GEMM is a dense contraction (T x d x E), so it runs on
// tcgen05 with N = E (rounded up to 16) and the whole logit row of 128 tokens in TMEM; it then
// costs one HBM read of x.
//
// CTA = 128 tokens, 256 threads:
//   warp 0     TMA producer: x tile [128 x 64] and W_r tile [Npad x 64] per stage
//   warp 1     MMA issuer: 4 x tcgen05.mma (M=128, N=Npad, K=16) per stage
//   warp 2     TMEM allocator
//   warp 3     copies the logit bias to shared memory
//   warps 4-7  epilogue, thread = token: three passes over its TMEM row
//              (1) top-(k+1) by logit, ties to the lower expert index,
//              (2) softmax denominator; near-tie candidates,
//              (3) probabilities, reduced over the CTA's tokens per expert (fixed order).
// Exactness of the selection: the tensor cores accumulate in fp32 but round differently from a
// sequential sum, so a token whose top-(k+1) logits are closer than a band (a bound on that
// accumulation error, scaled with d and the logits' magnitude) is re-decided from logits
// recomputed with compensated fp32 sums (near fp64 accuracy) for every expert within the band of
// the boundary.  The last CTA to finish (a counter in the workspace) reduces the
// per-CTA partials in a fixed order into counts and losses, so results are deterministic.
#include <float.h>
#include <stdio.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int RM = 128;                 // tokens per CTA (MMA M)
constexpr int RBK = 64;                 // K per stage: one 128-byte swizzle row of bf16
constexpr int RTHREADS = 256;
constexpr int A_TILE = RM * RBK * 2;    // 16 KB
constexpr int SMEM_STAGES_BYTES = 192 * 1024;
constexpr int MAX_STAGES = 8;
constexpr int CMAX = 16;                // near-tie candidates kept per token (more: all experts)
// Near-tie band of a token: a bound on the difference between the tensor cores' fp32 accumulation
// and an exactly rounded sum, |error| <~ (d / 16 MMA steps) x ulp(|partial sums|), taken twice
// over with |partial sums| <= max(1, |logits|); measured errors stay ~10x below it.
constexpr float kBandFloor = 2e-5f;
constexpr float kBadLogit = -3.0e38f;

struct RouteCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int hist[256];
  float bias[256];
  float red[4][256];
  float lse2[4];
  double lbterm[256];
  int npairs;
  uint8_t cand[RM][CMAX];
  float cexact[RM][CMAX];
  uint16_t pairs[RM * CMAX];   // (row << 4) | candidate slot
};

struct RouteArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* wr;
  const float* lbias;
  int T, d, E, k, npad, stages;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* hist;      // [nb][E] per-CTA expert histograms
  float* psum;        // [nb][E] per-CTA sums of P over tokens
  float* lse2;        // [nb]    per-CTA sums of lse^2
  uint32_t* done;     // CTA completion counter (zero between calls)
  int32_t* counts;
  float* losses;
  float lb_coef, z_coef;
  float band_scale;   // 2^-22 * d / 16
  uint32_t* status;
};

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Insert (v, e) into the descending list lv/le of length n (elements arrive in increasing e, so a
// strict comparison leaves an equal earlier element in front: ties go to the lower index).
template <int L>
__device__ __forceinline__ void list_insert(float (&lv)[L], int (&le)[L], int n, float v, int e) {
#pragma unroll
  for (int j = 0; j < L; ++j) {
    if (j < n && v > lv[j]) {
      const float tv = lv[j];
      const int te = le[j];
      lv[j] = v;
      le[j] = e;
      v = tv;
      e = te;
    }
  }
}

// Compensated (Neumaier) fp32 dot product of two bf16 rows of length d (a multiple of 8), one
// warp; bf16 x bf16 products are exact in fp32, so the result is close to the exact sum.  Each lane
// keeps eight 16-byte loads of each row in flight.  Every lane returns the same value.
__device__ __forceinline__ void neumaier_add(float& s, float& c, float p) {
  const float t = __fadd_rn(s, p);
  c = __fadd_rn(c, fabsf(s) >= fabsf(p) ? __fadd_rn(__fsub_rn(s, t), p) : __fadd_rn(__fsub_rn(p, t), s));
  s = t;
}

__device__ __forceinline__ float exact_dot(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ b,
                                           int d, int lane) {
  constexpr int U = 8;
  float s = 0.f, c = 0.f;
  for (int base = lane * 8; base < d; base += 256 * U) {
    uint4 av[U], bv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * 256;
      av[u] = i < d ? __ldg(reinterpret_cast<const uint4*>(a + i)) : make_uint4(0, 0, 0, 0);
      bv[u] = i < d ? __ldg(reinterpret_cast<const uint4*>(b + i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t aw[4] = {av[u].x, av[u].y, av[u].z, av[u].w};
      const uint32_t bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        neumaier_add(s, c, __fmul_rn(__uint_as_float(aw[j] << 16), __uint_as_float(bw[j] << 16)));
        neumaier_add(s, c, __fmul_rn(__uint_as_float(aw[j] & 0xffff0000u), __uint_as_float(bw[j] & 0xffff0000u)));
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

// Sum over the 32 lanes of 32 values per lane: afterwards lane l holds sum over lanes of v[l].
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

template <int KL>  // list length >= k + 1
__global__ void __launch_bounds__(RTHREADS, 1)
    k_route_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const RouteArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = A_TILE + a.npad * RBK * 2;
  RouteCtl* ctl = reinterpret_cast<RouteCtl*>(smem + (size_t)a.stages * stage_bytes);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k;
  const int kblocks = a.d / RBK;
  const int t0 = blockIdx.x * RM;
  uint32_t tmem_cols = 32;
  while ((int)tmem_cols < a.npad) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
    tmem_relinquish();
  }
  if (warp == 3) {
    if (lane == 0) ctl->npairs = 0;
    for (int e = lane; e < 256; e += 32) {
      ctl->bias[e] = (e < E && a.lbias) ? a.lbias[e] : 0.f;
      ctl->hist[e] = 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      // every CTA reads all of W_r: start each at a different k-block so that they do not all ask
      // the same L2 lines for the same tile at the same moment
      const int kb0 = (int)(blockIdx.x % (unsigned)kblocks);
      for (int i = 0; i < kblocks; ++i) {
        const int kb = kb0 + i < kblocks ? kb0 + i : kb0 + i - kblocks;
        if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.status)) {
          aborted = true;
          break;
        }
        const uint32_t fb = smem_u32(&ctl->full[s]);
        mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
        armed |= 1u << s;
        armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
        uint8_t* sa = smem + (size_t)s * stage_bytes;
        tma_load_2d(smem_u32(sa), &tmX, fb, kb * RBK, t0);
        tma_load_2d(smem_u32(sa + A_TILE), &tmW, fb, kb * RBK, 0);
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (aborted) {
        for (int i = 0; i < a.stages; ++i)
          if ((armed >> i) & 1u) drain(smem_u32(&ctl->full[i]), (armed_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(RM, a.npad);
      int s = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t sb = sa + A_TILE;
#pragma unroll
        for (int kk = 0; kk < RBK / 16; ++kk)
          umma_bf16(tmem_base, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), idesc, (kb | kk) != 0);
        umma_commit(smem_u32(&ctl->empty[s]));
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      umma_commit(smem_u32(&ctl->mma_done));
      drain(smem_u32(&ctl->mma_done), 0);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    const int r = q * 32 + lane;          // row of the tile = TMEM lane
    const int t = t0 + r;
    const bool valid = t < a.T;
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(smem_u32(&ctl->mma_done), 0, abort_flag, a.status) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    tc_fence_after();
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
    const int nl = min(k + 1, E);         // list entries in use

    // ---- pass 1: top-(k+1) by logit
    float lv[KL];
    int le[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      lv[j] = -FLT_MAX;
      le[j] = 0x7fffffff;
    }
    bool bad = false;
    if (ok) {
      for (int c0 = 0; c0 < E; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(trow + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c0 + i;
          if (e < E) {
            float z = __fadd_rn(__uint_as_float(v[i]), ctl->bias[e]);
            if (!isfinite(z)) {
              bad = true;
              z = kBadLogit;
            }
            list_insert(lv, le, nl, z, e);
          }
        }
      }
    }
    const float m = lv[0];
    float last = lv[0];  // smallest list entry in use (the list is sorted)
#pragma unroll
    for (int j = 1; j < KL; ++j)
      if (j < nl) last = fminf(last, lv[j]);
    const float band = fmaxf(kBandFloor, a.band_scale * fmaxf(1.f, fmaxf(fabsf(m), fabsf(last))));
    bool flagged = false;
#pragma unroll
    for (int j = 0; j + 1 < KL; ++j)
      if (j + 1 < nl && lv[j] - lv[j + 1] < band) flagged = true;
    flagged = flagged && valid && ok && !bad;

    // ---- pass 2: softmax denominator; near-tie candidates of flagged tokens
    const float thr = last - band;
    float s = 0.f;
    int nc = 0;
    if (ok) {
      for (int c0 = 0; c0 < E; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(trow + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c0 + i;
          if (e < E) {
            float z = __fadd_rn(__uint_as_float(v[i]), ctl->bias[e]);
            if (!isfinite(z)) z = kBadLogit;
            s += __expf(z - m);
            if (flagged && z >= thr) {
              if (nc < CMAX) ctl->cand[r][nc] = (uint8_t)e;
              ++nc;
            }
          }
        }
      }
    }

    // ---- exact re-decision of flagged tokens.  The (token, candidate) pairs of the CTA are shared
    // out over the 4 epilogue warps (one warp per dot product); a token with more than CMAX
    // candidates (degenerate inputs, e.g. a row of zeros) is re-decided over all experts by its own
    // warp.
    const bool few = flagged && nc <= CMAX;
    if (few) {
      const int p0 = atomicAdd(&ctl->npairs, nc);
      for (int c = 0; c < nc; ++c) ctl->pairs[p0 + c] = (uint16_t)((r << 4) | c);
    }
    epi_bar();
    const int np = ctl->npairs;
    for (int pi = q; pi < np; pi += 4) {
      const int pr = ctl->pairs[pi] >> 4, pc = ctl->pairs[pi] & 15;
      const int e = ctl->cand[pr][pc];
      float z = exact_dot(a.x + (size_t)(t0 + pr) * a.d, a.wr + (size_t)e * a.d, a.d, lane);
      z = __fadd_rn(z, ctl->bias[e]);
      if (lane == 0) ctl->cexact[pr][pc] = isfinite(z) ? z : kBadLogit;
    }
    epi_bar();
    if (few) {
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        lv[j] = -FLT_MAX;
        le[j] = 0x7fffffff;
      }
      for (int c = 0; c < nc; ++c) list_insert(lv, le, nl, ctl->cexact[r][c], (int)ctl->cand[r][c]);
    }
    unsigned fl = __ballot_sync(0xffffffffu, flagged && !few);
    while (fl) {
      const int f = __ffs(fl) - 1;
      fl &= fl - 1;
      const int tf = t0 + q * 32 + f;
      if (lane == f) {
#pragma unroll
        for (int j = 0; j < KL; ++j) {
          lv[j] = -FLT_MAX;
          le[j] = 0x7fffffff;
        }
      }
      for (int e = 0; e < E; ++e) {
        float z = exact_dot(a.x + (size_t)tf * a.d, a.wr + (size_t)e * a.d, a.d, lane);
        z = __fadd_rn(z, ctl->bias[e]);
        if (!isfinite(z)) z = kBadLogit;
        if (lane == f) list_insert(lv, le, nl, z, e);
      }
    }

    // ---- outputs of the token: indices, renormalised weights, histogram
    const float inv_s = 1.f / s;
    float lse = 0.f;
    if (valid && ok) {
      float wsum = 0.f;
      float p[KL];
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        p[j] = (j < k) ? __expf(lv[j] - lv[0]) : 0.f;
        wsum += p[j];
      }
      const float inv_w = 1.f / wsum;
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        if (j < k) {
          a.topk_idx[(size_t)t * k + j] = le[j];
          a.topk_w[(size_t)t * k + j] = p[j] * inv_w;
          atomicAdd(&ctl->hist[le[j]], 1);
        }
      }
      lse = m + __logf(s);
      if (bad) atomicOr(a.status, DEV_NONFINITE);
    }

    // ---- pass 3: P = exp(z - m) / s, summed over the CTA's tokens per expert
    if (ok) {
      for (int c0 = 0; c0 < E; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(trow + c0, v);
        tmem_wait_ld();
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float z = __fadd_rn(__uint_as_float(v[i]), ctl->bias[min(c0 + i, 255)]);
          if (!isfinite(z)) z = kBadLogit;
          pv[i] = (valid && c0 + i < E) ? __expf(z - m) * inv_s : 0.f;
        }
        const float colsum = warp_transpose_sum(pv, lane);
        if (c0 + lane < E) ctl->red[q][c0 + lane] = colsum;
      }
    }
    float l2 = valid ? lse * lse : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) l2 += __shfl_xor_sync(0xffffffffu, l2, o);
    if (lane == 0) ctl->lse2[q] = l2;
    epi_bar();

    // ---- per-CTA partials, then the last CTA reduces all of them
    const int te = threadIdx.x - 128;
    for (int e = te; e < E; e += 128) {
      a.psum[(size_t)blockIdx.x * E + e] = ((ctl->red[0][e] + ctl->red[1][e]) + ctl->red[2][e]) + ctl->red[3][e];
      a.hist[(size_t)blockIdx.x * E + e] = ctl->hist[e];
    }
    if (te == 0) a.lse2[blockIdx.x] = ((ctl->lse2[0] + ctl->lse2[1]) + ctl->lse2[2]) + ctl->lse2[3];
    __threadfence();
    epi_bar();
    if (te == 0) ctl->is_last = (atomicAdd(a.done, 1u) == gridDim.x - 1) ? 1 : 0;
    epi_bar();
    if (ctl->is_last) {
      __threadfence();
      const int nb = gridDim.x;
      // one thread per expert; partials are loaded 16 at a time (independent loads in flight) and
      // summed in block order, so the result does not depend on which CTA finished last
      constexpr int U = 16;
      for (int e = te; e < E; e += 128) {
        int cnt = 0;
        double ps = 0.0;
        for (int b0 = 0; b0 < nb; b0 += U) {
          int hv[U];
          float pv[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const bool in = b0 + u < nb;
            hv[u] = in ? __ldcg(a.hist + (size_t)(b0 + u) * E + e) : 0;
            pv[u] = in ? __ldcg(a.psum + (size_t)(b0 + u) * E + e) : 0.f;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            cnt += hv[u];
            ps += (double)pv[u];
          }
        }
        a.counts[e] = cnt;
        ctl->lbterm[e] = (double)cnt * ps;
      }
      double l = 0.0;
      if (te < 32) {
        for (int b = te; b < nb; b += 32) l += (double)__ldcg(a.lse2 + b);
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      }
      epi_bar();
      if (te == 0) {
        double lb = 0.0;
        for (int e = 0; e < E; ++e) lb += ctl->lbterm[e];
        const double Tn = (double)a.T;
        // lb = alpha E sum_e (c_e / (T k)) (psum_e / T);  zl = beta mean_t lse_t^2
        a.losses[0] = (float)((double)a.lb_coef * E * lb / (Tn * k * Tn));
        a.losses[1] = (float)((double)a.z_coef * l / Tn);
        *a.done = 0;  // ready for the next call
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

template <int KL>
cudaError_t launch_kl(const CUtensorMap& mx, const CUtensorMap& mw, const RouteArgs& a, int nb, size_t smem,
                      cudaStream_t st) {
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(k_route_tc<KL>), smem);
  if (err != cudaSuccess) return err;
  k_route_tc<KL><<<nb, RTHREADS, smem, st>>>(mx, mw, a);
  return cudaGetLastError();
}
}  // namespace

int route_tc_blocks(int T) { return (T + RM - 1) / RM; }

cudaError_t launch_route_tc(const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                            int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2, uint32_t* done,
                            int32_t* counts, float* losses, float lb_coef, float z_coef, uint32_t* status,
                            cudaStream_t st) {
  if (T <= 0) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)E, st);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(losses, 0, 2 * sizeof(float), st);
  }
  if (d % RBK || E < 1 || E > 256 || k < 1 || k > 8 || k > E) return cudaErrorInvalidValue;
  const int npad = ((E < 16 ? 16 : E) + 15) / 16 * 16;
  CUtensorMap mx, mw;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)T};
    const cuuint64_t str[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {RBK, RM};
    if (!make_tmap_bf16(&mx, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)E};
    const cuuint64_t str[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {RBK, (cuuint32_t)npad};
    if (!make_tmap_bf16(&mw, wr, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int stage_bytes = A_TILE + npad * RBK * 2;
  int stages = SMEM_STAGES_BYTES / stage_bytes;
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  const size_t smem = (size_t)stages * stage_bytes + sizeof(RouteCtl) + 1024;
  RouteArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.wr = static_cast<const __nv_bfloat16*>(wr);
  a.lbias = lbias;
  a.T = T; a.d = d; a.E = E; a.k = k; a.npad = npad; a.stages = stages;
  a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.hist = hist; a.psum = psum; a.lse2 = lse2; a.done = done;
  a.counts = counts; a.losses = losses; a.lb_coef = lb_coef; a.z_coef = z_coef;
  a.band_scale = ldexpf((float)d / 16.f, -22);
  a.status = status;
  const int nb = route_tc_blocks(T);
  cudaError_t err;
  if (k + 1 <= 3) err = launch_kl<3>(mx, mw, a, nb, smem, st);
  else if (k + 1 <= 5) err = launch_kl<5>(mx, mw, a, nb, smem, st);
  else err = launch_kl<9>(mx, mw, a, nb, smem, st);
  return err;
}

}  // namespace moe
