// Dispatch: build the expert-sorted layout of the routed (token, slot) assignments with the
// capacity applied in token order, and gather the token rows into it.
//
// Grouping tokens by target expert before one large matmul per expert is the inference advice of
// the Naive-N0.5-Flash article, sec. 4.2; the flatten-and-reorder formulation and the capacity
// C = cf * tokens / E with overflow dropped are the OpenMythos article, sec. 3.1.
//
// Deterministic, atomics-free ordering over blocks of 128 tokens: (1) a per-block histogram of the
// assignments per expert (for bf16 layers the router already writes it); (2) an exclusive scan of
// each expert's histogram over blocks gives every block its rank base, the capacity gives the kept
// counts and a scan over experts the offsets (for bf16 layers the router's last CTA does this);
// (3) one kernel per block ranks its assignments in token order (one warp, equal experts inside a
// 32-wide chunk ranked with __match_any_sync) and writes row_of / tok_of; (4) a row-parallel copy
// gathers x into x_perm.
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

// One CTA: per-expert exclusive scan over the blocks (16 loads in flight per thread), capacity,
// exclusive scan over experts.
__global__ void __launch_bounds__(256) k_perm_scan(const int32_t* __restrict__ phist, int npb,
                                                   const int32_t* __restrict__ counts, int E, int Tk, int cap,
                                                   int32_t* __restrict__ pbase, int32_t* __restrict__ offsets,
                                                   int32_t* __restrict__ kept, int32_t* __restrict__ drops,
                                                   uint32_t* status) {
  __shared__ int ks[256];
  const int tid = threadIdx.x;
  int kp = 0;
  if (tid < E) {
    constexpr int U = 16;
    int run = 0;
    for (int b0 = 0; b0 < npb; b0 += U) {
      int hv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) hv[u] = b0 + u < npb ? phist[(size_t)(b0 + u) * E + tid] : 0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (b0 + u < npb) pbase[(size_t)(b0 + u) * E + tid] = run;
        run += hv[u];
      }
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

// One CTA per block of PT tokens: the block's assignments ranked in token order (warp 0; equal
// experts inside a 32-wide chunk ranked with __match_any_sync), then row_of / tok_of.
template <int KMAX>
__global__ void __launch_bounds__(256) k_dispatch(const int32_t* __restrict__ topk_idx,
                                                  const int32_t* __restrict__ pbase,
                                                  const int32_t* __restrict__ offsets, int Tn, int E, int k, int cap,
                                                  int32_t* __restrict__ row_of, int32_t* __restrict__ tok_of,
                                                  uint32_t* status) {
  __shared__ int run[256];
  __shared__ int eidx[PT * KMAX];
  __shared__ int rows[PT * KMAX];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * PT;
  const int nt = min(PT, Tn - t0), na = nt * k;
  for (int e = tid; e < E; e += 256) run[e] = pbase[(size_t)blockIdx.x * E + e];
  for (int i = tid; i < na; i += 256) {
    int e = topk_idx[(size_t)t0 * k + i];
    if (e < 0 || e >= E) {
      atomicOr(status, DEV_BADINDEX);
      e = -1;
    }
    eidx[i] = e;
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c0 = 0; c0 < na; c0 += 32) {
      const int a = c0 + lane;
      const int e = a < na ? eidx[a] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      int row = -1;
      if (e >= 0) {
        const int r = run[e] + __popc(peers & lt_mask);
        if (r < cap) row = offsets[e] + r;
      }
      __syncwarp();
      if (e >= 0 && (__ffs(peers) - 1) == lane) run[e] += __popc(peers);
      __syncwarp();
      if (a < na) rows[a] = row;
    }
  }
  __syncthreads();
  for (int i = tid; i < na; i += 256) {
    const int row = rows[i];
    row_of[(size_t)t0 * k + i] = row;
    if (row >= 0) tok_of[row] = t0 + i / k;
  }
}

// x_perm[r] = x[tok_of[r]] for r < n_rows (device count); one warp per row, 16-byte vectors, a
// grid far larger than the SM count so that many loads are in flight.  The rows are written with
// streaming (evict-first) stores so that they do not push x, which every one of its k rows
// re-reads, out of L2.
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ tok_of,
                                                     const int32_t* __restrict__ n_rows_dev, int max_rows,
                                                     int row_vecs, uint4* __restrict__ x_perm) {
  const int n_rows = min(*n_rows_dev, max_rows);
  const int warps = gridDim.x * 8;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const int t = tok_of[r];
    const uint4* src = x + (size_t)t * row_vecs;
    uint4* dst = x_perm + (size_t)r * row_vecs;
    for (int c = threadIdx.x & 31; c < row_vecs; c += 32) __stcs(dst + c, src[c]);
  }
}

// Scalar row copy for rows whose byte length is not a multiple of 16: x_perm[r] = x[tok_of[r]].
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

int dispatch_launches(bool with_rows, int d, int elt_bytes) {
  (void)d;
  (void)elt_bytes;
  return with_rows ? 2 : 1;
}

cudaError_t launch_dispatch(bool bf16, const int32_t* topk_idx, const int32_t* pbase, const int32_t* offsets, int T,
                            int E, int k, int cap, const void* x, int d, int32_t* row_of, int32_t* tok_of,
                            void* x_perm, int max_rows, uint32_t* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int nb = perm_blocks(T);
  if (k <= 2)
    k_dispatch<2><<<nb, 256, 0, st>>>(topk_idx, pbase, offsets, T, E, k, cap, row_of, tok_of, status);
  else if (k <= 4)
    k_dispatch<4><<<nb, 256, 0, st>>>(topk_idx, pbase, offsets, T, E, k, cap, row_of, tok_of, status);
  else
    k_dispatch<8><<<nb, 256, 0, st>>>(topk_idx, pbase, offsets, T, E, k, cap, row_of, tok_of, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !x_perm || max_rows <= 0) return e;
  const size_t row_bytes = (size_t)d * (bf16 ? 2 : 4);
  int blocks = (max_rows + 7) / 8;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (row_bytes % 16 == 0)
    k_gather_rows<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(x), tok_of, offsets + E, max_rows,
                                          (int)(row_bytes / 16), static_cast<uint4*>(x_perm));
  else if (bf16)
    k_gather_rows_scalar<__nv_bfloat16><<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), tok_of,
                                                                offsets + E, max_rows, d,
                                                                static_cast<__nv_bfloat16*>(x_perm));
  else
    k_gather_rows_scalar<float><<<blocks, 256, 0, st>>>(static_cast<const float*>(x), tok_of, offsets + E, max_rows,
                                                        d, static_cast<float*>(x_perm));
  return cudaGetLastError();
}

}  // namespace moe
