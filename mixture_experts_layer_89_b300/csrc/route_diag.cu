// Routing diagnostics beyond the layer itself: the router entropy and the two other balance-loss
// forms the pages give, from the router's logits.
//
//   entropy      H_t = -sum_e P_te ln P_te = lse_t - sum_e P_te z'_te  (z' = z / tau)   -- the
//                routing-collapse signal the Naive-N0.5-Flash article, sec. 4, and the GPT-4 2%
//                article's troubleshooting tips watch (low: confident or collapsed, ln E: uniform)
//   squared form lb_coef E sum_e Pbar_e^2                                -- mini-moe tutorial, sec. 3.1
//   KL form      lb_coef (sum_e (1/E)(ln(1/E) - ln(Pbar_e + 1e-8)) + sum_e (f_e - 1/E)^2)
//                                                                        -- GPT-4 2% article, sec. 4.2
//   Switch form  lb_coef E sum_e f_e Pbar_e (the layer's own load-balance loss, OpenMythos sec. 3.1)
// with Pbar_e = mean_t P_te and f_e = counts_e / (T k) from the top-k of the raw logits.
//
// The logits are recomputed here in fp32 on CUDA cores (32 tokens per CTA, the K dimension in
// 64-column chunks through shared memory, each logit accumulated in a fixed order), so the call
// depends on nothing but its inputs.  Per-CTA partials (sums of P per expert, top-k counts, sum of
// H) are reduced in block order by one more CTA: the results do not depend on scheduling.
#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int DT = 32;        // tokens per CTA
constexpr int DC = 64;        // K columns per chunk
constexpr int DTHREADS = 256;
constexpr int MAXO = DT * 256 / DTHREADS;  // logits per thread at E = 256
constexpr float kBad = -3.0e38f;

size_t diag_smem(int E) {
  return sizeof(float) * ((size_t)DT * (DC + 1) + (size_t)E * (DC + 1) + (size_t)DT * (E + 1) + DT) + sizeof(int) * E;
}

template <typename T>
__global__ void __launch_bounds__(DTHREADS)
    k_route_diag(const T* __restrict__ x, const T* __restrict__ wr, const float* __restrict__ lbias, int Tn, int d,
                 int E, int k, float inv_tau, float* __restrict__ ent_tok, float* __restrict__ psum,
                 int32_t* __restrict__ cnt, float* __restrict__ hsum, uint32_t* status) {
  extern __shared__ float sm[];
  float* xs = sm;                     // [DT][DC+1]
  float* wsm = xs + DT * (DC + 1);    // [E][DC+1]
  float* zs = wsm + E * (DC + 1);     // [DT][E+1]: logits, then probabilities
  float* hs = zs + DT * (E + 1);      // [DT] entropies
  int* cs = reinterpret_cast<int*>(hs + DT);  // [E] top-k counts of the CTA
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * DT;
  const int nvalid = min(DT, Tn - t0);
  for (int e = tid; e < E; e += DTHREADS) cs[e] = 0;

  // ---- logits: output o = (token o / E, expert o % E), accumulated over K in order
  const int nout = DT * E;
  float acc[MAXO];
#pragma unroll
  for (int j = 0; j < MAXO; ++j) acc[j] = 0.f;
  for (int c0 = 0; c0 < d; c0 += DC) {
    const int cw = min(DC, d - c0);
    for (int i = tid; i < DT * DC; i += DTHREADS) {
      const int r = i / DC, c = i - r * DC;
      xs[r * (DC + 1) + c] = (r < nvalid && c < cw) ? to_f(x[(size_t)(t0 + r) * d + c0 + c]) : 0.f;
    }
    for (int i = tid; i < E * DC; i += DTHREADS) {
      const int e = i / DC, c = i - e * DC;
      wsm[e * (DC + 1) + c] = c < cw ? to_f(wr[(size_t)e * d + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < MAXO; ++j) {
      const int o = tid + j * DTHREADS;
      if (o < nout) {
        const int r = o / E, e = o - r * E;
        const float* xr = xs + r * (DC + 1);
        const float* we = wsm + e * (DC + 1);
        float a = acc[j];
#pragma unroll 8
        for (int c = 0; c < DC; ++c) a = fmaf(xr[c], we[c], a);
        acc[j] = a;
      }
    }
    __syncthreads();
  }
  bool bad = false;
#pragma unroll
  for (int j = 0; j < MAXO; ++j) {
    const int o = tid + j * DTHREADS;
    if (o < nout) {
      const int r = o / E, e = o - r * E;
      float z = acc[j] + (lbias ? lbias[e] : 0.f);
      if (r < nvalid && !isfinite(z)) {
        bad = true;
        z = kBad;
      }
      zs[r * (E + 1) + e] = z;
    }
  }
  if (bad) atomicOr(status, DEV_NONFINITE);
  __syncthreads();

  // ---- per token (one warp each): top-k counts on z, then softmax of z / tau and the entropy
  const int warp = tid >> 5, lane = tid & 31;
  for (int r = warp; r < nvalid; r += DTHREADS / 32) {
    float* zr = zs + r * (E + 1);
    float v[8];
    float m = kBad;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? zr[e] : -FLT_MAX;
      m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {  // k rounds of argmax, ties to the lower index
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
      if (lane == 0) atomicAdd(&cs[be], 1);
    }
    float s1 = 0.f, s2 = 0.f, p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      const float u = (v[i] - m) * inv_tau;
      p[i] = e < E ? __expf(u) : 0.f;
      s1 += p[i];
      s2 = e < E ? fmaf(p[i], u, s2) : s2;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    const float inv = 1.f / s1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E) zr[e] = p[i] * inv;
    }
    if (lane == 0) {
      const float h = __logf(s1) - s2 * inv;  // lse - sum P z' with both taken relative to the max
      hs[r] = h;
      if (ent_tok) ent_tok[t0 + r] = h;
    }
  }
  __syncthreads();

  // ---- per-CTA partials, each summed in token order
  for (int e = tid; e < E; e += DTHREADS) {
    float ps = 0.f;
    for (int r = 0; r < nvalid; ++r) ps += zs[r * (E + 1) + e];
    psum[(size_t)blockIdx.x * E + e] = ps;
    cnt[(size_t)blockIdx.x * E + e] = cs[e];
  }
  if (tid == 0) {
    float h = 0.f;
    for (int r = 0; r < nvalid; ++r) h += hs[r];
    hsum[blockIdx.x] = h;
  }
}

// One CTA: the partials of nb blocks in block order, then the four diagnostics.
__global__ void __launch_bounds__(256) k_route_diag_final(const float* __restrict__ psum,
                                                          const int32_t* __restrict__ cnt,
                                                          const float* __restrict__ hsum, int nb, int Tn, int E,
                                                          int k, float lb_coef, float* __restrict__ diag) {
  __shared__ double pbar[256];
  __shared__ double freq[256];
  __shared__ double hpart[256];
  const int tid = threadIdx.x;
  for (int e = tid; e < 256; e += 256) {
    double ps = 0.0;
    long long c = 0;
    if (e < E) {
      for (int b = 0; b < nb; ++b) {
        ps += (double)psum[(size_t)b * E + e];
        c += cnt[(size_t)b * E + e];
      }
    }
    pbar[e] = e < E && Tn > 0 ? ps / Tn : 0.0;
    freq[e] = e < E && Tn > 0 ? (double)c / ((double)Tn * k) : 0.0;
  }
  {  // a contiguous slice of blocks per thread, then the slices in order
    const int per = (nb + 255) / 256;
    double h = 0.0;
    for (int b = tid * per; b < min(nb, (tid + 1) * per); ++b) h += (double)hsum[b];
    hpart[tid] = h;
  }
  __syncthreads();
  if (tid == 0) {
    if (Tn <= 0) {
      diag[0] = diag[1] = diag[2] = diag[3] = 0.f;
      return;
    }
    double h = 0.0, sq = 0.0, kl = 0.0, fr = 0.0, sw = 0.0;
    for (int i = 0; i < 256; ++i) h += hpart[i];
    const double u = 1.0 / E;
    for (int e = 0; e < E; ++e) {
      sq += pbar[e] * pbar[e];
      kl += u * (log(u) - log(pbar[e] + 1e-8));
      fr += (freq[e] - u) * (freq[e] - u);
      sw += freq[e] * pbar[e];
    }
    diag[0] = (float)(h / Tn);
    diag[1] = (float)(lb_coef * E * sq);
    diag[2] = (float)(lb_coef * (kl + fr));
    diag[3] = (float)(lb_coef * E * sw);
  }
}

template <typename T>
cudaError_t launch_t(const void* x, const void* wr, const float* lbias, int Tn, int d, int E, int k, float inv_tau,
                     float lb_coef, float* diag, float* ent_tok, float* psum, int32_t* cnt, float* hsum,
                     uint32_t* status, cudaStream_t st) {
  const int nb = (Tn + DT - 1) / DT;
  if (nb > 0) {
    const size_t smem = diag_smem(E);
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_route_diag<T>), smem);
    if (e != cudaSuccess) return e;
    k_route_diag<T><<<nb, DTHREADS, smem, st>>>(static_cast<const T*>(x), static_cast<const T*>(wr), lbias, Tn, d,
                                                E, k, inv_tau, ent_tok, psum, cnt, hsum, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  k_route_diag_final<<<1, 256, 0, st>>>(psum, cnt, hsum, nb, Tn, E, k, lb_coef, diag);
  return cudaGetLastError();
}
}  // namespace

int route_diag_blocks(int T) { return (T + DT - 1) / DT; }

cudaError_t launch_route_diag(bool bf16, const void* x, const void* wr, const float* lbias, int T, int d, int E,
                              int k, float inv_tau, float lb_coef, float* diag, float* ent_tok, float* psum,
                              int32_t* cnt, float* hsum, uint32_t* status, cudaStream_t st) {
  if (E < 1 || E > 256 || k < 1 || k > 8 || k > E) return cudaErrorInvalidValue;
  if (bf16)
    return launch_t<__nv_bfloat16>(x, wr, lbias, T, d, E, k, inv_tau, lb_coef, diag, ent_tok, psum, cnt, hsum, status,
                                   st);
  return launch_t<float>(x, wr, lbias, T, d, E, k, inv_tau, lb_coef, diag, ent_tok, psum, cnt, hsum, status, st);
}

}  // namespace moe
