// Fused router of bf16 layers on the 5th-generation tensor cores: logits z = x W_r^T (+ logit
// bias) with fp32 accumulation, softmax, top-k with renormalised weights, per-expert counts and
// both auxiliary losses, in one launch.
//
// The router is the bias-free Linear -> softmax -> top-k -> renormalise of the mini-moe
// tutorial, sec. 3.1 (MoELayer) and the routing pseudo-code of the OpenMythos article, sec. 3.1;
// the load-balance loss is that article's alpha E sum_e f_e P_e, the z-loss the one the FLAME-MoE
// summary, sec. 2, names.  The logit GEMM is a dense contraction (T x d x E), so it runs on
// tcgen05 with N = E (rounded up to 16) and the whole logit row of 128 tokens in TMEM.
//
// Tile = 128 tokens, 256 threads per CTA.  Main loop:
//   warp 0     TMA producer: x tile [rows x 64] and W_r tile [Npad x 64] per stage
//   warp 1     MMA issuer: 4 x tcgen05.mma (M=128, N=Npad, K=16) per stage
//   warp 2     TMEM allocator;   warp 3   logit bias and counters
// With few tiles, a cluster of up to 8 CTAs shares a tile, each over a slice of the k-blocks;
// rank 0 adds the partial logits (distributed shared memory, rank order) and continues alone.
// Epilogue, all 8 warps, the pipeline buffers reused as scratch:
//   A  TMEM -> shared memory (warp w reads TMEM lane quarter w % 4)
//   B  thread per (token, expert half): sorted top-(k+1) insertion lists, ties to the lower
//      expert index, merged per token; near-tie candidates; softmax denominators
//   C  exact re-decision of near ties: the tensor cores accumulate in fp32 but round differently
//      from a sequential sum, so a token whose leading k+1 logits lie closer than a bound on that
//      accumulation error is re-decided from compensated fp32 (Neumaier) dot products of every
//      expert within the band, shared out over the warps
//   D  outputs per token; per-tile expert histogram, sums of P and of lse^2
// The per-tile partials are then reduced in tile order into counts and losses (route_losses.cuh):
// by the last tile's CTA (a counter in the workspace) for a router call on its own, or, inside a
// whole layer, by the dispatch and gather kernels.  Results do not depend on scheduling.
#include <float.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "route_losses.cuh"

namespace moe {

namespace {
constexpr int RM = 128;                 // tokens per CTA (MMA M)
constexpr int RBK = 64;                 // K per stage: one 128-byte swizzle row of bf16
constexpr int RTHREADS = 256;
constexpr int RWARPS = RTHREADS / 32;
constexpr int A_TILE = RM * RBK * 2;    // 16 KB
constexpr int SMEM_STAGES_BYTES = 192 * 1024;
constexpr int MAX_STAGES = 16;
constexpr int KLMAX = 9;                // top-(k+1) list, k <= 8
constexpr int CMAX = 16;                // near-tie candidates kept per token (more: all experts)
// Near-tie band of a token: a bound on the difference between the tensor cores' fp32 accumulation
// and an exactly rounded sum, |error| <~ (d / 16 MMA steps) x ulp(|partial sums|), taken twice
// over with |partial sums| <= max(1, |logits|); measured errors stay ~10x below it.
constexpr float kBandFloor = 2e-5f;
constexpr float kBadLogit = -3.0e38f;

enum : int { F_FEW = 2, F_ALL = 4, F_BAD = 8 };


struct RouteCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
  int npairs;
  int hist[256];
  float bias[256];
  float lse[RM];
  float mx[RM];       // top (tensor-core) logit of each token
  float sinv[RM];     // 1 / softmax denominator (0 for rows past T)
  float spart[2][RM]; // denominators of the two expert halves
  int flags[RM];
  int ncand[RM];
  float lse2w[RWARPS];
  LossScratch ls;     // last CTA: slices of the per-block partials
};

// Epilogue scratch laid over the pipeline buffers once the main loop is done.
constexpr int PPARTS = 8;  // row (or block) slices of the per-expert column sums
struct EpiScratch {
  float* Z;          // [RM][E+1] logits, then exp(z - max)
  float* tlv;        // [2][RM][KLMAX] top lists of the two expert halves (merged list in half 0)
  int* tle;          // [2][RM][KLMAX]
  float* cexact;     // [RM][CMAX] recomputed logits of near-tie candidates
  float* ppart;      // [PPARTS][256] partial column sums
  uint16_t* pairs;   // [RM*CMAX] (row << 4) | candidate slot
  uint8_t* cand;     // [RM][CMAX] candidate experts, ascending
};
__host__ __device__ inline size_t epi_scratch_bytes(int E) {
  return (size_t)RM * (E + 1) * 4 + 2 * (size_t)RM * KLMAX * 8 + (size_t)RM * CMAX * 4 + (size_t)PPARTS * 256 * 4 +
         (size_t)RM * CMAX * (2 + 1);
}
__device__ inline EpiScratch epi_scratch(uint8_t* base, int E) {
  EpiScratch s;
  s.Z = reinterpret_cast<float*>(base);
  s.tlv = s.Z + (size_t)RM * (E + 1);
  s.tle = reinterpret_cast<int*>(s.tlv + 2 * RM * KLMAX);
  s.cexact = reinterpret_cast<float*>(s.tle + 2 * RM * KLMAX);
  s.ppart = s.cexact + RM * CMAX;
  s.pairs = reinterpret_cast<uint16_t*>(s.ppart + PPARTS * 256);
  s.cand = reinterpret_cast<uint8_t*>(s.pairs + RM * CMAX);
  return s;
}

struct RouteArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* wr;
  const float* lbias;
  int T, d, E, k, npad, stages;
  int region;  // bytes before RouteCtl: the stages, or the epilogue scratch if that is larger
  int finalize;  // 1: the last CTA computes counts and losses (and the dispatch scan with pbase)
  int split;     // CTAs per tile (a cluster), each over a slice of the k-blocks
  int pofs;      // split > 1: byte offset of the partial logits [128][E] in the pipeline buffers
  int xrows;  // rows of the x box: 128, or fewer (a multiple of 8) when the layer has fewer tokens
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
  float inv_tau;      // 1 / router temperature (softmax, weights and lse of z / tau; top-k on z)
  // dispatch scan fused into the last CTA (pbase == NULL: not done here): per-block rank bases
  // [nb][E], kept counts [E], offsets [E+1], dropped assignments; cap = capacity (INT_MAX dropless)
  int cap;
  int32_t* pbase;
  int32_t* kept;
  int32_t* offsets;
  int32_t* drops;
  uint32_t* status;
};

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

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

template <int KL>  // list length >= k + 1
__global__ void __launch_bounds__(RTHREADS, 1)
    k_route_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const RouteArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // a stage holds the x rows of the tile (xrows x 128 bytes) and W_r (npad x 128 bytes); with fewer
  // than 128 tokens the MMA's A rows past xrows read the following bytes of shared memory (still
  // inside the allocation: RouteCtl follows the stages) and give logits that are never used
  const int a_bytes = a.xrows * RBK * 2;
  const int stage_bytes = a_bytes + a.npad * RBK * 2;
  RouteCtl* ctl = reinterpret_cast<RouteCtl*>(smem + (size_t)a.region);
  volatile int* abort_flag = &ctl->abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k;
  const int kblocks = a.d / RBK;
  // split > 1: a cluster of `split` CTAs shares one tile, each CTA accumulating its own slice of
  // the k-blocks; the cluster's rank 0 sums the partial logits and does the rest alone
  const int split = a.split;
  const int crank = split > 1 ? (int)cluster_ctarank() : 0;
  const int tile = (int)blockIdx.x / split;
  const int ntiles = (int)gridDim.x / split;
  const int kb_lo = kblocks * crank / split, kb_hi = kblocks * (crank + 1) / split;
  const int t0 = tile * RM;
  const int nvalid = min(RM, a.T - t0);  // rows of the tile that are tokens
  uint32_t tmem_cols = 32;
  while ((int)tmem_cols < a.npad) tmem_cols <<= 1;
  pdl_trigger();

  if (tid == 0) {
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
  // the set-up above overlaps the previous kernel's tail; x, the logit bias and every output buffer
  // belong to earlier kernels from here on
  pdl_wait();
  if (warp == 3) {
    if (lane == 0) ctl->npairs = 0;
    for (int e = lane; e < 256; e += 32) {
      ctl->bias[e] = (e < E && a.lbias) ? a.lbias[e] : 0.f;
      ctl->hist[e] = 0;
    }
    for (int r = lane; r < RM; r += 32) ctl->flags[r] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  // ------------------------------------------------------------------ main loop
  // every wait below drains this CTA's own copies and MMAs when it gives up, so the limit may be
  // shortened through the workspace (moe_set_wait_limit)
  const unsigned long long wlimit = (warp < 2 && lane == 0) ? wait_limit_ns(a.status) : kWaitLimitNs;
  if (warp == 0 && lane == 0) {
    int s = 0;
    uint32_t ph = 0, armed = 0, armed_ph = 0;
    bool aborted = false;
    // every CTA reads all of W_r: start each at a different k-block so that they do not all ask
    // the same L2 lines for the same tile at the same moment
    const int nk = kb_hi - kb_lo;
    const int kb0 = (int)(tile % (unsigned)nk);
    for (int i = 0; i < nk; ++i) {
      const int kb = kb_lo + (kb0 + i < nk ? kb0 + i : kb0 + i - nk);
      if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, a.status, wlimit)) {
        aborted = true;
        break;
      }
      const uint32_t fb = smem_u32(&ctl->full[s]);
      // fewer than 128 tokens: only their rows of x are loaded; the MMA rows past them read stale
      // shared memory and produce logits that are never used
      mbar_arrive_expect_tx(fb, (uint32_t)((a.xrows + a.npad) * RBK * 2));
      armed |= 1u << s;
      armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
      uint8_t* sa = smem + (size_t)s * stage_bytes;
      tma_load_2d(smem_u32(sa), &tmX, fb, kb * RBK, t0);
      tma_load_2d(smem_u32(sa + a_bytes), &tmW, fb, kb * RBK, 0);
      if (++s == a.stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (aborted) {
      for (int i = 0; i < a.stages; ++i)
        if ((armed >> i) & 1u) drain(smem_u32(&ctl->full[i]), (armed_ph >> i) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = umma_idesc_bf16(RM, a.npad);
    int s = 0;
    uint32_t ph = 0;
    for (int kb = 0; kb < kb_hi - kb_lo; ++kb) {
      if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, a.status, wlimit)) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
      const uint32_t sb = sa + a_bytes;
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
    drain(smem_u32(&ctl->mma_done), 0);  // every MMA has completed: the logits are in TMEM
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const EpiScratch S = epi_scratch(smem, E);  // the pipeline buffers are free from here on
  const int ZP = E + 1;                       // padded row pitch: conflict-free column accesses

  // ------------------------------------------------------------------ A: TMEM -> shared memory
  if (split > 1) {
    // raw partial logits of this CTA's k-blocks, rows [0, nvalid), pitch E, at the end of the
    // pipeline buffers (after the epilogue scratch); rank 0 adds the others' (same offset in each
    // CTA of the cluster) in rank order, 16 bytes at a time, then the bias
    float* P = reinterpret_cast<float*>(smem + a.pofs);
    {
      const int q = warp & 3, r = q * 32 + lane;
      const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
      for (int c0 = (warp >> 2) * 32; c0 < E; c0 += 64) {
        uint32_t v[32];
        tmem_ld32(trow + c0, v);
        tmem_wait_ld();
        if (r < nvalid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            if (c0 + i < E)
              *reinterpret_cast<float4*>(P + r * E + c0 + i) =
                  make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                              __uint_as_float(v[i + 3]));
        }
      }
    }
    tc_fence_before();
    cluster_sync_all();  // every partial is in its CTA's shared memory
    if (crank == 0) {
      const int e4n = E >> 2;
      for (int i = tid; i < nvalid * e4n; i += RTHREADS) {
        const int r = i / e4n, e = (i - r * e4n) * 4;
        const uint32_t off = smem_u32(P + r * E + e);
        float4 z = *reinterpret_cast<const float4*>(P + r * E + e);
        float4 rem[7];
#pragma unroll
        for (int c = 1; c < 8; ++c)
          if (c < split) rem[c - 1] = ld_shared_cluster_f32x4(mapa_rank(off, (uint32_t)c));
#pragma unroll
        for (int c = 1; c < 8; ++c) {
          if (c < split) {
            z.x = __fadd_rn(z.x, rem[c - 1].x);
            z.y = __fadd_rn(z.y, rem[c - 1].y);
            z.z = __fadd_rn(z.z, rem[c - 1].z);
            z.w = __fadd_rn(z.w, rem[c - 1].w);
          }
        }
        const float zz[4] = {z.x, z.y, z.z, z.w};
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float zj = __fadd_rn(zz[j], ctl->bias[e + j]);
          if (!isfinite(zj)) {
            zj = kBadLogit;
            bad = true;
          }
          S.Z[r * ZP + e + j] = zj;
        }
        if (bad) atomicOr(&ctl->flags[r], F_BAD);
      }
    }
    cluster_sync_all();  // rank 0 has read every partial: the other CTAs may leave
    if (crank != 0) {
      __syncthreads();
      if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
      }
      return;
    }
  } else {
    const int q = warp & 3, r = q * 32 + lane;
    const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
    bool bad = false;
    for (int c0 = (warp >> 2) * 32; c0 < E; c0 += 64) {
      uint32_t v[32];
      tmem_ld32(trow + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (c0 + i < E) {
          float z = __fadd_rn(__uint_as_float(v[i]), ctl->bias[c0 + i]);
          if (!isfinite(z)) {
            bad = true;
            z = kBadLogit;
          }
          S.Z[r * ZP + c0 + i] = z;
        }
      }
    }
    if (bad) atomicOr(&ctl->flags[r], F_BAD);
  }
  tc_fence_before();
  __syncthreads();

  // ------------------------------------------------------------------ B: top-(k+1) per token
  // Thread per (token, expert half): a sorted insertion list over the half's experts in increasing
  // index (measured faster here than warp-cooperative argmax rounds, whose shuffle round trips
  // dominate), then the lower half's thread merges the upper half's list into its own.
  const int nl = min(k + 1, E);
  const int ehalf = (E + 1) >> 1;
  {
    const int h = tid >> 7, r = tid & (RM - 1);
    float lv[KL];
    int le[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      lv[j] = -FLT_MAX;
      le[j] = 0x7fffffff;
    }
    const int e_hi = r < nvalid ? (h ? E : ehalf) : 0;  // rows past T: no list
    for (int e = h ? ehalf : 0; e < e_hi; ++e) list_insert(lv, le, nl, S.Z[r * ZP + e], e);
    float* tv = S.tlv + (size_t)(h * RM + r) * KLMAX;
    int* te = S.tle + (size_t)(h * RM + r) * KLMAX;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      tv[j] = lv[j];
      te[j] = le[j];
    }
  }
  __syncthreads();
  if (tid < RM) {
    const int r = tid;
    float lv[KL];
    int le[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      lv[j] = S.tlv[r * KLMAX + j];
      le[j] = S.tle[r * KLMAX + j];
    }
    // the upper half's experts all have higher indices: insert them in their list order
#pragma unroll
    for (int j = 0; j < KL; ++j)
      if (j < nl && S.tle[(RM + r) * KLMAX + j] != 0x7fffffff)
        list_insert(lv, le, nl, S.tlv[(RM + r) * KLMAX + j], S.tle[(RM + r) * KLMAX + j]);
    const float m = lv[0];
    float last = lv[0];
#pragma unroll
    for (int j = 1; j < KL; ++j)
      if (j < nl) last = fminf(last, lv[j]);
    const float band = fmaxf(kBandFloor, a.band_scale * fmaxf(1.f, fmaxf(fabsf(m), fabsf(last))));
    bool flagged = false;
#pragma unroll
    for (int j = 0; j + 1 < KL; ++j)
      if (j + 1 < nl && lv[j] - lv[j + 1] < band) flagged = true;
    flagged = flagged && (t0 + r < a.T) && !(ctl->flags[r] & F_BAD);
    int nc = 0;
    if (flagged) {  // near-tie candidates: every expert within the band of the (k+1)-th logit
      const float thr = last - band;
      for (int e = 0; e < E; ++e) {
        if (S.Z[r * ZP + e] >= thr) {
          if (nc < CMAX) S.cand[r * CMAX + nc] = (uint8_t)e;
          ++nc;
        }
      }
      if (nc <= CMAX) {
        const int p0 = atomicAdd(&ctl->npairs, nc);
        for (int c = 0; c < nc; ++c) S.pairs[p0 + c] = (uint16_t)((r << 4) | c);
        ctl->flags[r] |= F_FEW;
      } else {
        ctl->flags[r] |= F_ALL;
      }
    }
    ctl->ncand[r] = nc;
    ctl->mx[r] = m;
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      S.tlv[r * KLMAX + j] = lv[j];
      S.tle[r * KLMAX + j] = le[j];
    }
  }
  __syncthreads();
  {  // softmax denominators, per expert half; Z becomes exp(z - max)
    const int h = tid >> 7, r = tid & (RM - 1);
    const float m = ctl->mx[r];
    float s0 = 0.f, s1 = 0.f;
    const int e_lo = h ? ehalf : 0, e_hi = h ? E : ehalf;
    if (r >= nvalid) {  // rows past T: no token, nothing to normalise
      s0 = 1.f;
    } else {
    int e = e_lo;
    for (; e + 1 < e_hi; e += 2) {
      const float p0 = __expf((S.Z[r * ZP + e] - m) * a.inv_tau), p1 = __expf((S.Z[r * ZP + e + 1] - m) * a.inv_tau);
      S.Z[r * ZP + e] = p0;
      S.Z[r * ZP + e + 1] = p1;
      s0 += p0;
      s1 += p1;
    }
    if (e < e_hi) {
      const float p0 = __expf((S.Z[r * ZP + e] - m) * a.inv_tau);
      S.Z[r * ZP + e] = p0;
      s0 += p0;
    }
    }
    ctl->spart[h][r] = s0 + s1;
  }
  __syncthreads();
  if (tid < RM) {
    const int r = tid;
    const float s = ctl->spart[0][r] + ctl->spart[1][r];
    const bool valid = t0 + r < a.T;
    ctl->sinv[r] = valid ? 1.f / s : 0.f;
    ctl->lse[r] = valid ? ctl->mx[r] * a.inv_tau + __logf(s) : 0.f;
  }

  // ------------------------------------------------------------------ C: exact re-decision of near ties
  {
    const int np = ctl->npairs;
    for (int pi = warp; pi < np; pi += RWARPS) {
      const int pr = S.pairs[pi] >> 4, pc = S.pairs[pi] & 15;
      const int e = S.cand[pr * CMAX + pc];
      float z = exact_dot(a.x + (size_t)(t0 + pr) * a.d, a.wr + (size_t)e * a.d, a.d, lane);
      z = __fadd_rn(z, ctl->bias[e]);
      if (lane == 0) S.cexact[pr * CMAX + pc] = isfinite(z) ? z : kBadLogit;
    }
    // tokens with more candidates than CMAX (degenerate inputs, e.g. a row of zeros): all experts
    for (int r = warp; r < RM; r += RWARPS) {
      if (!(ctl->flags[r] & F_ALL)) continue;
      float lv[KL];
      int le[KL];
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        lv[j] = -FLT_MAX;
        le[j] = 0x7fffffff;
      }
      for (int e = 0; e < E; ++e) {
        float z = exact_dot(a.x + (size_t)(t0 + r) * a.d, a.wr + (size_t)e * a.d, a.d, lane);
        z = __fadd_rn(z, ctl->bias[e]);
        if (!isfinite(z)) z = kBadLogit;
        list_insert(lv, le, nl, z, e);
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < KL; ++j) {
          S.tlv[r * KLMAX + j] = lv[j];
          S.tle[r * KLMAX + j] = le[j];
        }
      }
    }
  }
  __syncthreads();

  // ------------------------------------------------------------------ D: outputs and per-CTA partials
  if (tid < RM) {
    const int r = tid, t = t0 + r;
    const int fl = ctl->flags[r];
    float lv[KL];
    int le[KL];
#pragma unroll
    for (int j = 0; j < KL; ++j) {
      lv[j] = S.tlv[r * KLMAX + j];
      le[j] = S.tle[r * KLMAX + j];
    }
    if (fl & F_FEW) {
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        lv[j] = -FLT_MAX;
        le[j] = 0x7fffffff;
      }
      const int nc = ctl->ncand[r];
      for (int c = 0; c < nc; ++c) list_insert(lv, le, nl, S.cexact[r * CMAX + c], (int)S.cand[r * CMAX + c]);
    }
    float l2 = 0.f;
    if (t < a.T) {
      float wsum = 0.f;
#pragma unroll
      for (int j = 0; j < KL; ++j) wsum += (j < k) ? __expf((lv[j] - lv[0]) * a.inv_tau) : 0.f;
      const float inv_w = 1.f / wsum;
#pragma unroll
      for (int j = 0; j < KL; ++j) {
        if (j < k) {
          a.topk_idx[(size_t)t * k + j] = le[j];
          a.topk_w[(size_t)t * k + j] = __expf((lv[j] - lv[0]) * a.inv_tau) * inv_w;
          atomicAdd(&ctl->hist[le[j]], 1);
        }
      }
      if (fl & F_BAD) atomicOr(a.status, DEV_NONFINITE);
      l2 = ctl->lse[r] * ctl->lse[r];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) l2 += __shfl_xor_sync(0xffffffffu, l2, o);
    if (lane == 0) ctl->lse2w[warp] = l2;
  }
  // per-expert sums of P = exp(z - max) / denominator over the CTA's tokens: row slices, then the
  // slices in order
  int parts = 1;  // a power of two (so it divides RM), with parts * E <= RTHREADS
  while (parts < PPARTS && 2 * parts * E <= RTHREADS) parts <<= 1;
  {
    const int e = tid % E, part = tid / E;
    if (part < parts) {
      const int rows = RM / parts;
      const int r_hi = min((part + 1) * rows, nvalid);  // rows past T hold no token
      float ps = 0.f;
      for (int r = part * rows; r < r_hi; ++r) ps = fmaf(S.Z[r * ZP + e], ctl->sinv[r], ps);
      S.ppart[part * 256 + e] = ps;
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += RTHREADS) {
    float ps = 0.f;
    for (int part = 0; part < parts; ++part) ps += S.ppart[part * 256 + e];
    a.psum[(size_t)tile * E + e] = ps;
    a.hist[(size_t)tile * E + e] = ctl->hist[e];
  }
  if (tid == 0) a.lse2[tile] = ((ctl->lse2w[0] + ctl->lse2w[1]) + ctl->lse2w[2]) + ctl->lse2w[3];
  if (a.finalize) {  // the last CTA to get here reduces every CTA's partials
    __threadfence();
    __syncthreads();
    if (tid == 0) ctl->is_last = (atomicAdd(a.done, 1u) == (unsigned)ntiles - 1) ? 1 : 0;
  } else if (tid == 0) {
    ctl->is_last = 0;  // the fused dispatch kernel reduces them
  }
  __syncthreads();

  // ------------------------------------------------------------------ last CTA: counts and losses
  if (ctl->is_last) {
    __threadfence();
    const int nb = ntiles;
    route_losses<true, true>(a.hist, a.psum, a.lse2, nb, E, k, a.T, a.lb_coef, a.z_coef, ctl->hist, a.counts,
                             a.losses, ctl->ls);
    if (a.pbase) {
      // dispatch scan: each expert's exclusive scan over the blocks (the block's rank base), one
      // slice per thread starting from the earlier slices' counts; kept counts under the capacity;
      // offsets over experts; drops
      const int parts = loss_parts(E);
      const int e = tid % E, part = tid / E;
      if (part < parts) {
        const int b_lo = (int)((long)nb * part / parts), b_hi = (int)((long)nb * (part + 1) / parts);
        int run = 0;
        for (int q = 0; q < part; ++q) run += ctl->ls.lcnt[q][e];
        for (int bb = b_lo; bb < b_hi; ++bb) {
          const int h = __ldcg(a.hist + (size_t)bb * E + e);
          a.pbase[(size_t)bb * E + e] = run;
          run += h;
        }
      }
      for (int ee = tid; ee < E; ee += RTHREADS) {
        const int kp = min(ctl->hist[ee], a.cap);
        a.kept[ee] = kp;
        ctl->hist[ee] = kp;
      }
      __syncthreads();
      if (warp == 2) {  // exclusive scan of the kept counts over experts, 8 per lane
        int v[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ee = lane * 8 + i;
          v[i] = ee < E ? ctl->hist[ee] : 0;
          sum += v[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ee = lane * 8 + i;
          run += v[i];
          if (ee < E) a.offsets[ee + 1] = run;
        }
        if (lane == 0) a.offsets[0] = 0;
        if (lane == 31) *a.drops = a.T * k - incl;
      }
    }
    if (tid == 0) *a.done = 0;  // ready for the next call
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// Whether at least one cluster of `split` CTAs of this kernel (with `smem` bytes each) can be
// resident; asked once per (kernel, device, smem, split) and remembered.
template <typename K>
bool clusters_fit_query(K kern, const cudaLaunchConfig_t& cfg) {
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  return n >= 1;
}
struct FitEntry {
  const void* k;
  int dev;
  size_t smem;
  int split;
  bool fit;
};
std::mutex g_fit_mu;
FitEntry g_fit[64];
int g_nfit = 0;

template <int KL>
bool clusters_fit_kl(size_t smem, int split, const cudaLaunchConfig_t& cfg) {
  const void* key = reinterpret_cast<const void*>(k_route_tc<KL>);
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_fit_mu);
  for (int i = 0; i < g_nfit; ++i)
    if (g_fit[i].k == key && g_fit[i].dev == dev && g_fit[i].smem == smem && g_fit[i].split == split) return g_fit[i].fit;
  const bool fit = clusters_fit_query(k_route_tc<KL>, cfg);
  if (g_nfit < 64) g_fit[g_nfit++] = FitEntry{key, dev, smem, split, fit};
  return fit;
}

template <int KL>
cudaError_t launch_kl(const CUtensorMap& mx, const CUtensorMap& mw, RouteArgs a, int nb, size_t smem, int max_split,
                      cudaStream_t st) {
  auto clusters_fit = [&](const void*, size_t sm, int sp, const cudaLaunchConfig_t& c) {
    return clusters_fit_kl<KL>(sm, sp, c);
  };
  auto kern = k_route_tc<KL>;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  // Few tiles: split each tile's k-blocks over a cluster of up to 8 CTAs (one CTA per SM), so that
  // more SMs pull x and W_r; the split shrinks until the clusters fit the GPU.
  int nsm = 148;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  }
  int split = 1;
  while (split < max_split && (long)nb * split * 2 <= nsm && split * 2 <= a.d / RBK) split <<= 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(RTHREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  for (; split > 1; split >>= 1) {
    attr[1].val.clusterDim.x = split;
    cfg.gridDim = dim3((unsigned)(nb * split), 1, 1);
    cfg.numAttrs = 2;
    if (clusters_fit(reinterpret_cast<const void*>(kern), smem, split, cfg)) break;
  }
  a.split = split;
  cfg.gridDim = dim3((unsigned)(nb * split), 1, 1);
  if (split > 1) {
    attr[1].val.clusterDim.x = split;
    cfg.numAttrs = 2;
  } else {
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, mx, mw, a);
}
}  // namespace

int route_tc_blocks(int T) { return (T + RM - 1) / RM; }

// Bytes of the pipeline buffers for E experts and tiles of 128 tokens (the last CTA stages the
// per-block partials there).
static long route_stage_region(int E) {
  const int npad = ((E < 16 ? 16 : E) + 15) / 16 * 16;
  const int stage_bytes = A_TILE + npad * RBK * 2;
  const int stages = SMEM_STAGES_BYTES / stage_bytes < MAX_STAGES ? SMEM_STAGES_BYTES / stage_bytes : MAX_STAGES;
  return (long)stages * stage_bytes;
}

bool route_tc_fuses_scan(int T, int E) {
  return T > 0 && E >= 1 && E <= 256 && 8L * route_tc_blocks(T) * E <= route_stage_region(E);
}

cudaError_t launch_route_tc(const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                            int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2, uint32_t* done,
                            int32_t* counts, float* losses, float lb_coef, float z_coef, uint32_t* status,
                            cudaStream_t st, const RouteScan* scan, bool finalize, float inv_tau) {
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
    const cuuint32_t box[2] = {RBK, (cuuint32_t)(T < RM ? (T + 7) / 8 * 8 : RM)};
    if (!make_tmap_bf16(&mx, x, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)E};
    const cuuint64_t str[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {RBK, (cuuint32_t)npad};
    if (!make_tmap_bf16(&mw, wr, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  const int xrows = T < RM ? (T + 7) / 8 * 8 : RM;  // a multiple of 8: whole 1024-byte swizzle atoms
  const int stage_bytes = xrows * RBK * 2 + npad * RBK * 2;
  int stages = SMEM_STAGES_BYTES / stage_bytes;
  if (stages > MAX_STAGES) stages = MAX_STAGES;
  size_t region = (size_t)stages * stage_bytes;
  if (region < epi_scratch_bytes(E)) region = (epi_scratch_bytes(E) + 1023) / 1024 * 1024;  // few tokens, many experts
  const size_t smem = region + sizeof(RouteCtl) + 1024;
  RouteArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.wr = static_cast<const __nv_bfloat16*>(wr);
  a.lbias = lbias;
  a.T = T; a.d = d; a.E = E; a.k = k; a.npad = npad; a.stages = stages; a.region = (int)region;
  a.xrows = xrows;
  a.topk_idx = topk_idx; a.topk_w = topk_w;
  a.hist = hist; a.psum = psum; a.lse2 = lse2; a.done = done;
  a.counts = counts; a.losses = losses; a.lb_coef = lb_coef; a.z_coef = z_coef;
  a.band_scale = ldexpf((float)d / 16.f, -22);
  a.inv_tau = inv_tau;
  a.status = status;
  a.finalize = finalize ? 1 : 0;
  const bool fuse = finalize && scan && route_tc_fuses_scan(T, E);
  a.cap = fuse ? scan->cap : 0;
  a.pbase = fuse ? scan->pbase : nullptr;
  a.kept = fuse ? scan->kept : nullptr;
  a.offsets = fuse ? scan->offsets : nullptr;
  a.drops = fuse ? scan->drops : nullptr;
  const int nb = route_tc_blocks(T);
  cudaError_t err;
  // split-K over a cluster needs E % 4 == 0 and room for the partials after the epilogue scratch;
  // a partial tile (T < 128) takes up to 8 CTAs, full tiles up to 4 (rank 0 sums 128 rows)
  const size_t pbytes = (size_t)RM * E * 4;
  int max_split = (E % 4 == 0 && region >= pbytes && (region - pbytes) / 1024 * 1024 >= epi_scratch_bytes(E))
                      ? (T < RM ? 8 : 4)
                      : 1;
  a.pofs = (int)((region - pbytes) / 1024 * 1024);
  if (k + 1 <= 3) err = launch_kl<3>(mx, mw, a, nb, smem, max_split, st);
  else if (k + 1 <= 5) err = launch_kl<5>(mx, mw, a, nb, smem, max_split, st);
  else err = launch_kl<9>(mx, mw, a, nb, smem, max_split, st);
  return err;
}

}  // namespace moe
