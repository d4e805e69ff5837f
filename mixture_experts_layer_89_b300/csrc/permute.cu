// Dispatch: build the expert-sorted layout of the routed (token, slot) assignments with the
// capacity applied in token order, and gather the token rows into it.
//
// Grouping tokens by target expert before one large matmul per expert is the inference advice of
// the Naive-N0.5-Flash article, sec. 4.2; the flatten-and-reorder formulation and the capacity
// C = cf * tokens / E with overflow dropped are the OpenMythos article, sec. 3.1.
//
// Deterministic, atomics-free ordering: (1) each CTA of 64 tokens histograms its assignments per
// expert; (2) one CTA scans the histograms per expert over CTAs (the rank base of every CTA),
// applies the capacity and scans the kept counts over experts (offsets); (3) each CTA walks its
// assignments in token order with one warp, ranking equal experts inside a 32-wide chunk with
// __match_any_sync, and writes row_of / tok_of; (4) a row-parallel copy gathers x into x_perm.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int PT = kPermTokens;

__global__ void __launch_bounds__(256) k_perm_hist(const int32_t* __restrict__ topk_idx, int Tn, int E, int k,
                                                   int32_t* __restrict__ phist, uint32_t* status) {
  __shared__ int h[256];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += 256) h[e] = 0;
  __syncthreads();
  const long a0 = (long)blockIdx.x * PT * k;
  const long a1 = min(a0 + (long)PT * k, (long)Tn * k);
  for (long a = a0 + tid; a < a1; a += 256) {
    const int e = topk_idx[a];
    if (e < 0 || e >= E) {
      atomicOr(status, DEV_BADINDEX);
      continue;
    }
    atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) phist[(size_t)blockIdx.x * E + e] = h[e];
}

// One CTA: per-expert scan over the dispatch CTAs, capacity, exclusive scan over experts.
__global__ void __launch_bounds__(256) k_perm_scan(const int32_t* __restrict__ phist, int npb,
                                                   const int32_t* __restrict__ counts, int E, int Tk, int cap,
                                                   int32_t* __restrict__ pbase, int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ kept, int32_t* __restrict__ drops,
                                                   uint32_t* status) {
  __shared__ int ks[256];
  const int tid = threadIdx.x;
  int kp = 0;
  if (tid < E) {
    int run = 0;
    for (int b = 0; b < npb; ++b) {
      pbase[(size_t)b * E + tid] = run;
      run += phist[(size_t)b * E + tid];
    }
    if (counts && counts[tid] != run) atomicOr(status, DEV_BADCOUNTS);
    kp = min(run, cap);
    kept[tid] = kp;
  }
  ks[tid] = kp;
  __syncthreads();
  // inclusive Hillis-Steele scan over 256 entries
  for (int s = 1; s < 256; s <<= 1) {
    const int v = (tid >= s) ? ks[tid - s] : 0;
    __syncthreads();
    ks[tid] += v;
    __syncthreads();
  }
  if (tid < E) offsets[tid + 1] = ks[tid];
  if (tid == 0) {
    offsets[0] = 0;
    if (drops) *drops = Tk - ks[E - 1];
  }
}

// Ranks of each CTA's assignments in token order -> row_of, tok_of.
__global__ void __launch_bounds__(32) k_perm_rank(const int32_t* __restrict__ topk_idx,
                                                  const int32_t* __restrict__ pbase,
                                                  const int32_t* __restrict__ offsets, int Tn, int E, int k, int cap,
                                                  int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of) {
  __shared__ int run[256];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) run[e] = pbase[(size_t)blockIdx.x * E + e];
  __syncwarp();
  const long a0 = (long)blockIdx.x * PT * k;
  const long a1 = min(a0 + (long)PT * k, (long)Tn * k);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long c0 = a0; c0 < a1; c0 += 32) {
    const long a = c0 + lane;
    const bool valid = a < a1;
    int e = valid ? topk_idx[a] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int row = -1;
    if (e >= 0) {
      const int r = run[e] + __popc(peers & lt_mask);
      if (r < cap) row = offsets[e] + r;
    }
    __syncwarp();
    if (e >= 0 && (__ffs(peers) - 1) == lane) run[e] += __popc(peers);
    __syncwarp();
    if (valid) {
      row_of[a] = row;
      if (row >= 0) tok_of[row] = (int)(a / k);
    }
  }
}

// x_perm[r] = x[tok_of[r]] for r < n_rows (device count); one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ tok_of,
                                                     const int32_t* __restrict__ n_rows_dev, int max_rows,
                                                     int row_vecs, uint4* __restrict__ x_perm) {
  const int n_rows = min(*n_rows_dev, max_rows);
  const int warps = gridDim.x * 8;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const int t = tok_of[r];
    const uint4* src = x + (size_t)t * row_vecs;
    uint4* dst = x_perm + (size_t)r * row_vecs;
    for (int c = threadIdx.x & 31; c < row_vecs; c += 32) dst[c] = src[c];
  }
}

// Scalar fallback of the gather for rows whose byte length is not a multiple of 16.
template <typename T>
__global__ void __launch_bounds__(256) k_gather_rows_scalar(const T* __restrict__ x,
                                                            const int32_t* __restrict__ tok_of,
                                                            const int32_t* __restrict__ n_rows_dev, int max_rows,
                                                            int d, T* __restrict__ x_perm) {
  const int n_rows = min(*n_rows_dev, max_rows);
  const int warps = gridDim.x * 8;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const int t = tok_of[r];
    for (int c = threadIdx.x & 31; c < d; c += 32) x_perm[(size_t)r * d + c] = x[(size_t)t * d + c];
  }
}
}  // namespace

int perm_blocks(int T) { return (T + PT - 1) / PT; }

cudaError_t launch_perm_hist(const int32_t* topk_idx, int T, int E, int k, int32_t* phist, uint32_t* status,
                             cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  k_perm_hist<<<perm_blocks(T), 256, 0, st>>>(topk_idx, T, E, k, phist, status);
  return cudaGetLastError();
}

cudaError_t launch_perm_scan(const int32_t* phist, int npb, const int32_t* counts, int E, int Tk, int cap,
                             int32_t* pbase, int32_t* offsets, int32_t* kept, int32_t* drops, uint32_t* status,
                             cudaStream_t st) {
  k_perm_scan<<<1, 256, 0, st>>>(phist, npb, counts, E, Tk, cap, pbase, offsets, kept, drops, status);
  return cudaGetLastError();
}

cudaError_t launch_perm_rank(const int32_t* topk_idx, const int32_t* pbase, const int32_t* offsets, int T, int E,
                             int k, int cap, int32_t* row_of, int32_t* tok_of, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  k_perm_rank<<<perm_blocks(T), 32, 0, st>>>(topk_idx, pbase, offsets, T, E, k, cap, row_of, tok_of);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(bool bf16, const void* x, const int32_t* tok_of, const int32_t* n_rows_dev,
                               int max_rows, int d, void* x_perm, cudaStream_t st) {
  if (max_rows <= 0) return cudaSuccess;
  const size_t row_bytes = (size_t)d * (bf16 ? 2 : 4);
  int blocks = (max_rows + 7) / 8;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (row_bytes % 16 == 0) {
    k_gather_rows<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x), tok_of, n_rows_dev, max_rows,
                                          (int)(row_bytes / 16), static_cast<uint4*>(x_perm));
  } else if (bf16) {
    k_gather_rows_scalar<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), tok_of,
                                                                n_rows_dev, max_rows, d,
                                                                static_cast<__nv_bfloat16*>(x_perm));
  } else {
    k_gather_rows_scalar<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(x), tok_of, n_rows_dev, max_rows,
                                                        d, static_cast<float*>(x_perm));
  }
  return cudaGetLastError();
}

}  // namespace moe
