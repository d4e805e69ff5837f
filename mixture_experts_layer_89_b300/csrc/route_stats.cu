// Routing statistics: expert co-activation counts, load imbalance and the dropped fraction, from
// the router's top-k indices and the dispatch's offsets.
//
// How often two experts are chosen for the same token, and how unevenly the experts are loaded,
// are the routing behaviours the FLAME-MoE summary (co-activation of experts) and the
// Naive-N0.5-Flash article, sec. 4 (load balance, capacity overflow) discuss.
//
// coact[i][j] (i != j) counts the tokens whose k experts include both i and j; coact[i][i] counts
// the tokens that chose i.  Integer atomics only, so the result does not depend on scheduling.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int ST = 128;  // tokens per CTA

// E <= kCoactSmemE: the CTA accumulates its tokens' pairs in a shared E x E matrix and adds the
// non-zero entries to the global one; else straight into the global matrix.
constexpr int kCoactSmemE = 128;

__global__ void __launch_bounds__(256) k_coact(const int32_t* __restrict__ topk_idx, int Tn, int E, int k,
                                               int32_t* __restrict__ coact, uint32_t* status) {
  extern __shared__ int C[];  // [E][E] when E <= kCoactSmemE
  const bool shared = E <= kCoactSmemE;
  const int tid = threadIdx.x;
  if (shared)
    for (int i = tid; i < E * E; i += 256) C[i] = 0;
  __syncthreads();
  const int t = blockIdx.x * ST + tid;
  if (tid < ST && t < Tn) {
    int e[8];
    bool ok = true;
    for (int j = 0; j < k; ++j) {
      e[j] = topk_idx[(size_t)t * k + j];
      if (e[j] < 0 || e[j] >= E) ok = false;
    }
    if (!ok) {
      atomicOr(status, DEV_BADINDEX);
    } else {
      for (int a = 0; a < k; ++a)
        for (int b = 0; b < k; ++b) {
          const int idx = e[a] * E + e[b];
          if (shared)
            atomicAdd(&C[idx], 1);
          else
            atomicAdd(&coact[idx], 1);
        }
    }
  }
  __syncthreads();
  if (shared)
    for (int i = tid; i < E * E; i += 256)
      if (C[i]) atomicAdd(&coact[i], C[i]);
}

// stats[0] = max_e coact[e][e] / (T k / E); stats[1] = (T k - offsets[E]) / (T k).
__global__ void __launch_bounds__(256) k_route_stats_final(const int32_t* __restrict__ coact,
                                                           const int32_t* __restrict__ offsets, int Tn, int E,
                                                           int k, float* __restrict__ stats) {
  __shared__ int mx[256];
  const int tid = threadIdx.x;
  int m = 0;
  for (int e = tid; e < E; e += 256) m = max(m, coact[(size_t)e * E + e]);
  mx[tid] = m;
  __syncthreads();
  for (int s = 128; s; s >>= 1) {
    if (tid < s) mx[tid] = max(mx[tid], mx[tid + s]);
    __syncthreads();
  }
  if (tid == 0) {
    const float tk = (float)Tn * (float)k;
    stats[0] = tk > 0.f ? (float)mx[0] * (float)E / tk : 0.f;
    stats[1] = (tk > 0.f && offsets) ? (tk - (float)offsets[E]) / tk : 0.f;
  }
}
}  // namespace

cudaError_t launch_route_stats(const int32_t* topk_idx, const int32_t* offsets, int T, int E, int k, int32_t* coact,
                               float* stats, uint32_t* status, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(coact, 0, sizeof(int32_t) * (size_t)E * E, st);
  if (err != cudaSuccess) return err;
  if (T > 0) {
    const size_t smem = E <= kCoactSmemE ? sizeof(int) * (size_t)E * E : 0;
    err = ensure_smem_attr(reinterpret_cast<const void*>(k_coact), smem);
    if (err != cudaSuccess) return err;
    k_coact<<<(T + ST - 1) / ST, 256, smem, st>>>(topk_idx, T, E, k, coact, status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  k_route_stats_final<<<1, 256, 0, st>>>(coact, offsets, T, E, k, stats);
  return cudaGetLastError();
}

}  // namespace moe
