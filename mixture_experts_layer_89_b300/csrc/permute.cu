// Dispatch: build the expert-sorted layout of the routed (token, slot) assignments with the
// capacity applied in token order, and gather the token rows into it.
//
// Grouping tokens by target expert before one large matmul per expert is the inference advice of
// the Naive-N0.5-Flash article, sec. 4.2; the flatten-and-reorder formulation and the capacity
// C = cf * tokens / E with overflow dropped are the OpenMythos article, sec. 3.1.
//
// Deterministic, atomics-free ordering over blocks of 128 tokens: (1) a per-block histogram of the
// assignments per expert; (2) an exclusive scan of each expert's histogram over blocks gives every
// block its rank base, the capacity gives the kept counts and a scan over experts the offsets;
// (3) one CTA per block ranks its assignments in token order (one warp, equal experts inside a
// 32-wide chunk ranked with __match_any_sync) and writes row_of / tok_of; (4) a row-parallel copy
// gathers x into x_perm.  Inside a bf16 layer the router writes the per-block histograms (1) and
// k_dispatch_fused derives (2) per CTA before ranking (3); moe_permute on its own and fp32 layers
// run k_perm_hist, k_perm_scan and k_dispatch.
#include "common.cuh"
#include "kernels.h"
#include "route_losses.cuh"

namespace moe {

namespace {
constexpr int PT = kPermTokens;

// Ranks one block's assignments in token order from the per-expert rank bases in run[] (warp 0;
// equal experts inside a 32-wide chunk ranked with __match_any_sync); row = offsets[e] + rank while
// the rank is under the capacity, else -1 (dropped).
__device__ __forceinline__ void rank_block(const int* eidx, int na, int* run, const int* offs, int cap, int* rows) {
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < na; c0 += 32) {
    const int a = c0 + lane;
    const int e = a < na ? eidx[a] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int row = -1;
    if (e >= 0) {
      const int r = run[e] + __popc(peers & lt_mask);
      if (r < cap) row = offs[e] + r;
    }
    __syncwarp();
    if (e >= 0 && (__ffs(peers) - 1) == lane) run[e] += __popc(peers);
    __syncwarp();
    if (a < na) rows[a] = row;
  }
}


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
  const int tid = threadIdx.x, warp = tid >> 5;
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
  if (warp == 0) rank_block(eidx, na, run, offsets, cap, rows);
  __syncthreads();
  for (int i = tid; i < na; i += 256) {
    const int row = rows[i];
    row_of[(size_t)t0 * k + i] = row;
    if (row >= 0) tok_of[row] = t0 + i / k;
  }
}

// Per-block histograms staged by the fused dispatch: at most this many (blocks x experts) ints.
constexpr int kDispatchScanInts = 16384;

struct DispatchFusedArgs {
  const int32_t* topk_idx;
  const int32_t* hist;  // [nb][E] router per-block expert histograms
  const float* psum;    // [nb][E] router per-block sums of P
  const float* lse2;    // [nb]
  int T, E, k, cap;
  float lb_coef, z_coef;
  int32_t* counts;
  float* losses;
  int32_t* offsets;
  int32_t* kept;
  int32_t* drops;
  int32_t* row_of;
  int32_t* tok_of;
  uint32_t* status;
};

// One CTA per block of PT tokens.  Every CTA stages all per-block histograms in shared memory and
// derives what the router's last CTA would otherwise compute for it: its rank base per expert
// (the sum over the earlier blocks), the kept counts under the capacity and the offsets (exclusive
// scan over experts).  CTA 0 also writes offsets, kept, drops, and the counts and losses (the same
// reduction, in the same order, as the router's last CTA).
template <int KMAX>
__global__ void __launch_bounds__(256) k_dispatch_fused(const DispatchFusedArgs a) {
  extern __shared__ int H[];  // [nb][E]
  __shared__ int run[256];
  __shared__ int kp_s[256];
  __shared__ int offs[257];
  __shared__ int eidx[PT * KMAX];
  __shared__ int rows[PT * KMAX];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, nb = gridDim.x, E = a.E, k = a.k;
  const int n = nb * E;
  const int t0 = b * PT;
  const int nt = min(PT, a.T - t0), na = nt * k;
  pdl_trigger();
  pdl_wait();
  {
    constexpr int U = 16;  // independent loads in flight per thread
    for (int i0 = tid; i0 < n; i0 += 256 * U) {
      int hv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * 256;
        hv[u] = i < n ? __ldg(a.hist + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * 256;
        if (i < n) H[i] = hv[u];
      }
    }
  }
  for (int i = tid; i < na; i += 256) {
    int e = a.topk_idx[(size_t)t0 * k + i];
    if (e < 0 || e >= E) {
      atomicOr(a.status, DEV_BADINDEX);
      e = -1;
    }
    eidx[i] = e;
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int base = 0, tot = 0;
    for (int bb = 0; bb < nb; ++bb) {
      const int h = H[bb * E + e];
      base += bb < b ? h : 0;
      tot += h;
    }
    run[e] = base;
    kp_s[e] = min(tot, a.cap);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the kept counts over experts, 8 per lane
    int v[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      v[i] = e < E ? kp_s[e] : 0;
      sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int r = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) offs[e] = r;
      r += v[i];
    }
    if (lane == 31) offs[E] = incl;
  }
  __syncthreads();
  if (warp == 0) rank_block(eidx, na, run, offs, a.cap, rows);
  __syncthreads();
  for (int i = tid; i < na; i += 256) {
    const int row = rows[i];
    a.row_of[(size_t)t0 * k + i] = row;
    if (row >= 0) a.tok_of[row] = t0 + i / k;
  }
  if (b == 0) {
    for (int e = tid; e <= E; e += 256) a.offsets[e] = offs[e];
    for (int e = tid; e < E; e += 256) a.kept[e] = kp_s[e];
    if (tid == 0) *a.drops = a.T * k - offs[E];
  }
}

// Counts and losses of a layer whose router left them to the dispatch: reduced by block 0 of the
// row gather (thousands of blocks), off the critical path of the dispatch ranks.
struct LossArgs {
  const int32_t* hist;
  const float* psum;
  const float* lse2;
  int nb, E, k, T;
  float lb_coef, z_coef;
  int32_t* counts;
  float* losses;
};

// x_perm[r] = x[tok_of[r]] for r < n_rows (device count); one warp per row, 16-byte vectors, a
// grid far larger than the SM count so that many loads are in flight.  The rows are written with
// streaming (evict-first) stores so that they do not push x, which every one of its k rows
// re-reads, out of L2.
template <bool LOSSES>
__global__ void __launch_bounds__(256) k_gather_rows(const uint4* __restrict__ x, const int32_t* __restrict__ tok_of,
                                                     const int32_t* __restrict__ n_rows_dev, int max_rows,
                                                     int row_vecs, uint4* __restrict__ x_perm, const LossArgs la) {
  pdl_trigger();
  pdl_wait();
  if constexpr (LOSSES) {
    __shared__ LossScratch sc;
    if (blockIdx.x == 0)
      route_losses<true, true>(la.hist, la.psum, la.lse2, la.nb, la.E, la.k, la.T, la.lb_coef, la.z_coef, nullptr,
                               la.counts, la.losses, sc);
  }
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
  pdl_trigger();
  pdl_wait();
  const int n_rows = min(*n_rows_dev, max_rows);
  const int warps = gridDim.x * 8;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const int t = tok_of[r];
    for (int c = threadIdx.x & 31; c < d; c += 32) x_perm[(size_t)r * d + c] = x[(size_t)t * d + c];
  }
}

// Backup expert (a routing variant: the mini-moe tutorial, sec. 6, routes tokens over an expert's
// capacity to a backup expert instead of dropping them).  The assignments the capacity drops take
// rows offsets[E] .. offsets[E] + drops - 1 of the expert-sorted layout, in (token, slot) order, and
// keep their routing weight.  k_backup_count: dropped assignments per block of PT tokens.
__global__ void __launch_bounds__(256) k_backup_count(const int32_t* __restrict__ row_of, int Tn, int k,
                                                      int32_t* __restrict__ bcount) {
  pdl_trigger();
  pdl_wait();
  __shared__ int c;
  if (threadIdx.x == 0) c = 0;
  __syncthreads();
  const long a0 = (long)blockIdx.x * PT * k;
  const long a1 = min(a0 + (long)PT * k, (long)Tn * k);
  int local = 0;
  for (long a = a0 + threadIdx.x; a < a1; a += 256) local += row_of[a] < 0 ? 1 : 0;
  atomicAdd(&c, local);  // integers: the total does not depend on the order
  __syncthreads();
  if (threadIdx.x == 0) bcount[blockIdx.x] = c;
}

// One CTA per block: its base (the earlier blocks' counts), the ranks of its dropped assignments in
// (token, slot) order (warp 0, ballots over 32-wide chunks), row_of / tok_of, and the token rows
// copied into x_perm.  CTA 0 also writes the backup expert's row range {offsets[E], offsets[E] + all}.
template <typename T>
__global__ void __launch_bounds__(256) k_backup_place(const int32_t* __restrict__ bcount, int nb,
                                                      const int32_t* __restrict__ kept_rows, int Tn, int k, int d,
                                                      const T* __restrict__ x, int32_t* __restrict__ row_of,
                                                      int32_t* __restrict__ tok_of, T* __restrict__ x_perm,
                                                      int32_t* __restrict__ backup_offs) {
  pdl_trigger();
  pdl_wait();
  __shared__ int red[256];
  __shared__ int rows[PT * 8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a_kept = *kept_rows;
  int before = 0, all = 0;
  for (int b = tid; b < nb; b += 256) {
    const int c = bcount[b];
    all += c;
    if (b < (int)blockIdx.x) before += c;
  }
  red[tid] = before;
  __syncthreads();
  for (int sh = 128; sh; sh >>= 1) {
    if (tid < sh) red[tid] += red[tid + sh];
    __syncthreads();
  }
  const int base = a_kept + red[0];
  __syncthreads();
  if (blockIdx.x == 0) {
    red[tid] = all;
    __syncthreads();
    for (int sh = 128; sh; sh >>= 1) {
      if (tid < sh) red[tid] += red[tid + sh];
      __syncthreads();
    }
    if (tid == 0) {
      backup_offs[0] = a_kept;
      backup_offs[1] = a_kept + red[0];
    }
  }
  const long a0 = (long)blockIdx.x * PT * k;
  const int na = (int)(min(a0 + (long)PT * k, (long)Tn * k) - a0);
  if (warp == 0) {
    int run = 0;
    for (int c0 = 0; c0 < na; c0 += 32) {
      const int a = c0 + lane;
      const bool dropped = a < na && row_of[a0 + a] < 0;
      const unsigned bal = __ballot_sync(0xffffffffu, dropped);
      const int row = dropped ? base + run + __popc(bal & ((1u << lane) - 1u)) : -1;
      run += __popc(bal);
      if (a < na) rows[a] = row;
      if (dropped) {
        row_of[a0 + a] = row;
        tok_of[row] = (int)((a0 + a) / k);
      }
    }
  }
  __syncthreads();
  for (int a = warp; a < na; a += 8) {  // one warp per backup row
    const int row = rows[a];
    if (row < 0) continue;
    const T* src = x + (size_t)((a0 + a) / k) * d;
    T* dst = x_perm + (size_t)row * d;
    for (int c = lane; c < d; c += 32) dst[c] = src[c];
  }
}
}  // namespace

int perm_blocks(int T) { return (T + PT - 1) / PT; }

cudaError_t launch_backup_dispatch(bool bf16, const int32_t* kept_rows, int T, int k, int d, const void* x,
                                   int32_t* row_of, int32_t* tok_of, void* x_perm, int32_t* bcount,
                                   int32_t* backup_offs, cudaStream_t st) {
  if (T <= 0 || k > 8) return T <= 0 ? cudaSuccess : cudaErrorInvalidValue;
  const int nb = perm_blocks(T);
  cudaError_t e = launch_pdl(k_backup_count, dim3(nb), dim3(256), 0, st, static_cast<const int32_t*>(row_of), T, k,
                             bcount);
  if (e != cudaSuccess) return e;
  if (bf16)
    return launch_pdl(k_backup_place<__nv_bfloat16>, dim3(nb), dim3(256), 0, st, static_cast<const int32_t*>(bcount),
                      nb, kept_rows, T, k, d, static_cast<const __nv_bfloat16*>(x), row_of, tok_of,
                      static_cast<__nv_bfloat16*>(x_perm), backup_offs);
  return launch_pdl(k_backup_place<float>, dim3(nb), dim3(256), 0, st, static_cast<const int32_t*>(bcount), nb,
                    kept_rows, T, k, d, static_cast<const float*>(x), row_of, tok_of, static_cast<float*>(x_perm),
                    backup_offs);
}

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

bool dispatch_fuses_scan(int T, int E) {
  return T > 0 && E >= 1 && E <= 256 && (long)perm_blocks(T) * E <= kDispatchScanInts;
}

namespace {
template <int KMAX>
cudaError_t launch_fused_k(const DispatchFusedArgs& a, int nb, cudaStream_t st) {
  const size_t smem = sizeof(int) * (size_t)nb * a.E;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(k_dispatch_fused<KMAX>), smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(k_dispatch_fused<KMAX>, dim3(nb), dim3(256), smem, st, a);
}

cudaError_t launch_gather(bool bf16, const void* x, int d, const int32_t* tok_of, const int32_t* n_rows, void* x_perm,
                          int max_rows, cudaStream_t st, const LossArgs* la = nullptr) {
  const size_t row_bytes = (size_t)d * (bf16 ? 2 : 4);
  int blocks = (max_rows + 7) / 8;
  if (blocks > 148 * 32) blocks = 148 * 32;
  if (la && row_bytes % 16 != 0) return cudaErrorInvalidValue;
  const dim3 g(blocks), b(256);
  if (la)
    return launch_pdl(k_gather_rows<true>, g, b, 0, st, static_cast<const uint4*>(x), tok_of, n_rows, max_rows,
                      (int)(row_bytes / 16), static_cast<uint4*>(x_perm), *la);
  if (row_bytes % 16 == 0)
    return launch_pdl(k_gather_rows<false>, g, b, 0, st, static_cast<const uint4*>(x), tok_of, n_rows, max_rows,
                      (int)(row_bytes / 16), static_cast<uint4*>(x_perm), LossArgs{});
  if (bf16)
    return launch_pdl(k_gather_rows_scalar<__nv_bfloat16>, g, b, 0, st, static_cast<const __nv_bfloat16*>(x), tok_of,
                      n_rows, max_rows, d, static_cast<__nv_bfloat16*>(x_perm));
  return launch_pdl(k_gather_rows_scalar<float>, g, b, 0, st, static_cast<const float*>(x), tok_of, n_rows, max_rows,
                    d, static_cast<float*>(x_perm));
}
}  // namespace

cudaError_t launch_dispatch_fused(bool bf16, const int32_t* topk_idx, const int32_t* hist, const float* psum,
                                  const float* lse2, int T, int E, int k, int cap, float lb_coef, float z_coef,
                                  const void* x, int d, int32_t* counts, float* losses, int32_t* offsets,
                                  int32_t* kept, int32_t* drops, int32_t* row_of, int32_t* tok_of, void* x_perm,
                                  int max_rows, uint32_t* status, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (!dispatch_fuses_scan(T, E) || k < 1 || k > 8 || !x_perm || ((size_t)d * (bf16 ? 2 : 4)) % 16 != 0)
    return cudaErrorInvalidValue;
  DispatchFusedArgs a;
  a.topk_idx = topk_idx; a.hist = hist; a.psum = psum; a.lse2 = lse2;
  a.T = T; a.E = E; a.k = k; a.cap = cap; a.lb_coef = lb_coef; a.z_coef = z_coef;
  a.counts = counts; a.losses = losses; a.offsets = offsets; a.kept = kept; a.drops = drops;
  a.row_of = row_of; a.tok_of = tok_of; a.status = status;
  const int nb = perm_blocks(T);
  cudaError_t e;
  if (k <= 2) e = launch_fused_k<2>(a, nb, st);
  else if (k <= 4) e = launch_fused_k<4>(a, nb, st);
  else e = launch_fused_k<8>(a, nb, st);
  if (e != cudaSuccess) return e;
  LossArgs la;
  la.hist = hist; la.psum = psum; la.lse2 = lse2; la.nb = nb; la.E = E; la.k = k; la.T = T;
  la.lb_coef = lb_coef; la.z_coef = z_coef; la.counts = counts; la.losses = losses;
  // the gather's block 0 reduces the losses, so it runs even when no row can be kept
  return launch_gather(bf16, x, d, tok_of, offsets + E, x_perm, max_rows > 0 ? max_rows : 1, st, &la);
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
  return launch_gather(bf16, x, d, tok_of, offsets + E, x_perm, max_rows, st);
}

}  // namespace moe
