// Grouped bf16 GEMM on the 5th-generation tensor cores for the backward pass of the expert FFNs:
//
//   C[m, n] (+)= sum_k A[m, k] B[n, k]      A, B bf16 (A K-major); fp32 accumulators and output
//
// in two grouped forms (group g < G <= 256):
//   rows on M (input gradients, recomputed pre-activations): group g owns rows [off[g], off[g+1])
//     of A [rows, K] and of C [rows, ldc]; its B is B[g] of B [G][N][K]; K is fixed.
//   rows on K (weight gradients): group g owns the columns [off[g], off[g+1]) of A [M][Kp] and of
//     B [N][Kp] (the group's rows of the layer, transposed, each group zero-padded to a multiple
//     of 64 columns); its C is C + g c_stride, [M, N] with ldc.
// A NULL offset array means one group: rows [0, rows) (rows on M) or columns [0, rows) (on K).
// Rows on M may also read B N-major, straight from the weights as stored: B_g(n, k) at
// [g][k][n] of one tensor for k < ksplit and of a second one (at k - ksplit) beyond, so that
// dh = dy W_down and dx = du W_up + dg W_gate need no transposed copy of the weights.
//
// Persistent 2-SM pairs (a cluster of two CTAs, one per SM, issuing tcgen05.mma with
// cta_group::2): a pair owns a 256 x 256 output tile, each CTA 128 rows of it.  Per 64-deep K step
// each CTA holds its 128 rows of A and its 128-row half of B (32 KB, written by TMA with the
// 128-byte swizzle), so the operand stream per SM is 2/3 of what one SM alone would need for a
// 128 x 256 tile.  The pairs walk the tiles of all groups in order.  In each CTA warp 0 loads the
// stages (both CTAs' copies complete on the leader's barrier); the leader's warp 1 issues the MMAs
// (M = 256, N = 256, K = 16) into one of two TMEM accumulators (2 x 256 columns in each CTA) and
// its commits reach both CTAs; warps 2-5 of each CTA drain its own 128 rows of the other
// accumulator into C (32 x 32 blocks staged in shared memory for coalesced or TMA stores) while
// the next tile accumulates.  Each output is one accumulation in k order, so results do not depend
// on scheduling.  Every wait is bounded: on a time-out the kernel records DEV_TIMEOUT in the status
// word, lets its copies and MMAs in flight land, frees its tensor memory and returns.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int GB_BM = 128;   // rows of C per CTA (256 per pair)
constexpr int GB_BN = 256;   // columns of C per tile (each CTA holds half of B's 256 rows)
constexpr int GB_BK = 64, GB_STAGES = 6, GB_MAXG = 256;
constexpr int GB_A_BYTES = GB_BM * GB_BK * 2;        // 16 KB
constexpr int GB_B_BYTES = (GB_BN / 2) * GB_BK * 2;  // 16 KB
constexpr int GB_STAGE_BYTES = GB_A_BYTES + GB_B_BYTES;
constexpr int GB_THREADS = 192;
constexpr uint32_t GB_TMEM_COLS = 2 * GB_BN;
constexpr int GB_EPI_BYTES = 4 * 32 * 32 * 4;  // one 32 x 32 fp32 staging block per epilogue warp
constexpr size_t GB_SMEM = (size_t)GB_STAGES * GB_STAGE_BYTES + GB_EPI_BYTES + 1024;  // + alignment slack
static_assert(GB_STAGE_BYTES % 1024 == 0 && GB_A_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(GB_SMEM <= 227 * 1024 - 4096, "stages fit the shared memory of one CTA");
static_assert(GB_MAXG <= 32 * 8, "eight groups per lane in the tile count");

struct GbCtl {
  uint64_t full[GB_STAGES], empty[GB_STAGES], tfull[2], tempty[2], mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int pre[GB_MAXG + 1];  // tiles of the groups before g
  int lo[GB_MAXG + 1];   // the group boundaries
};

struct GbArgs {
  int rows_on_k;
  int b_mn, ksplit;  // rows on M: B N-major (map_b for k < ksplit, map_b2 beyond)
  const int32_t* off;  // [G + 1] or NULL (one group of `rows`)
  int G, rows;
  int M, N, K;  // rows on M: N and K; rows on K: M and N
  float* C;
  int64_t ldc, c_stride;
  int beta;
  uint32_t* status;
};

__device__ __forceinline__ void gb_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

struct GbTile {
  int g, m0, n0, mrows, kb, k0;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GB_THREADS, 1)
    k_gemm_bwd(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_b2, const __grid_constant__ CUtensorMap map_c,
               const GbArgs a) {
  extern __shared__ uint8_t gb_raw[];
  __shared__ GbCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gb_raw) + 1023) & ~(uintptr_t)1023);
  float* epi = reinterpret_cast<float*>(smem + (size_t)GB_STAGES * GB_STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  constexpr uint16_t kPair = 0x3;
  volatile int* abort_flag = &ctl.abort_flag;
  const int G = a.off ? a.G : 1;
  const int nt = (a.N + GB_BN - 1) / GB_BN;
  if (threadIdx.x == 0) {
    for (int s = 0; s < GB_STAGES; ++s) {
      mbar_init(smem_u32(&ctl.full[s]), 1);  // the leader's arrive_expect_tx (both CTAs' bytes)
      mbar_init(smem_u32(&ctl.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl.tfull[b]), 1);
      mbar_init(smem_u32(&ctl.tempty[b]), 8);  // one arrive per epilogue warp of the pair
    }
    mbar_init(smem_u32(&ctl.mma_done), 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b);
    if (a.b_mn && a.ksplit < a.K) tma_prefetch_desc(&map_b2);
  }
  if (warp == 2) {  // both CTAs of the pair allocate together and receive the same address
    tmem_alloc_cg2(smem_u32(&ctl.tmem_base), GB_TMEM_COLS);
    tmem_relinquish_cg2();
  }
  if (warp == 3) {  // tiles per group and their exclusive prefix; lane owns groups [8 lane, 8 lane + 8)
    int cnt[8], local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      cnt[i] = 0;
      if (g < G) {
        const int lo = a.off ? a.off[g] : 0;
        const int hi = a.off ? a.off[g + 1] : a.rows;
        ctl.lo[g] = lo;
        if (g == G - 1) ctl.lo[G] = hi;
        const int span = a.rows_on_k ? a.M : (hi > lo ? hi - lo : 0);
        cnt[i] = (span + 2 * GB_BM - 1) / (2 * GB_BM) * nt;
        local += cnt[i];
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      if (g < G) ctl.pre[g] = run;
      run += cnt[i];
    }
    if (lane == 31) ctl.pre[G] = incl;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.pre[G];
  const int pair = (int)blockIdx.x >> 1, npairs = (int)gridDim.x >> 1;

  // this CTA's part of tile u: its 128 rows of the pair's 256, the pair's 256 columns
  auto decode = [&](int u) {
    int lo = 0, hi = G - 1;  // the last group whose first tile is at or before u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ctl.pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    GbTile t;
    t.g = lo;
    const int r = u - ctl.pre[lo];
    const int mt = r / nt;
    t.n0 = (r % nt) * GB_BN;
    const int glo = ctl.lo[lo], ghi = ctl.lo[lo + 1];
    if (a.rows_on_k) {
      t.m0 = mt * 2 * GB_BM + (int)crank * GB_BM;
      t.mrows = max(0, min(GB_BM, a.M - t.m0));
      t.k0 = glo;
      t.kb = (ghi - glo) / GB_BK;
    } else {
      t.m0 = glo + mt * 2 * GB_BM + (int)crank * GB_BM;
      t.mrows = max(0, min(GB_BM, ghi - t.m0));
      t.k0 = 0;
      t.kb = a.K / GB_BK;
    }
    return t;
  };

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      for (int u = pair; u < total && !aborted; u += npairs) {
        const GbTile t = decode(u);
        const int nb = t.n0 + (int)crank * (GB_BN / 2);  // this CTA's half of B
        for (int kb = 0; kb < t.kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl.empty[s]), ph ^ 1u, abort_flag, a.status)) {
            aborted = true;
            break;
          }
          const uint32_t sa = smem_u32(smem + (size_t)s * GB_STAGE_BYTES), sb = sa + GB_A_BYTES;
          const uint32_t fb = smem_u32(&ctl.full[s]);
          const uint32_t lb = mapa_rank(fb, 0);
          if (leader) {
            mbar_arrive_expect_tx(fb, 2u * GB_STAGE_BYTES);
            armed |= 1u << s;
            armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          }
          const int kc = t.k0 + kb * GB_BK;
          tma_load_2d_cg2(sa, &map_a, lb, kc, t.m0);
          if (a.rows_on_k) {
            tma_load_2d_cg2(sb, &map_b, lb, kc, nb);
          } else if (a.b_mn) {  // two boxes of 64 n by 64 k, 8 KB apart
            const bool lo_half = kc < a.ksplit;
            const CUtensorMap* mb = lo_half ? &map_b : &map_b2;
            const int kl = lo_half ? kc : kc - a.ksplit;
#pragma unroll
            for (int j = 0; j < GB_BN / 2 / 64; ++j) tma_load_3d_cg2(sb + j * 8192, mb, lb, nb + 64 * j, kl, t.g);
          } else {
            tma_load_3d_cg2(sb, &map_b, lb, kc, nb, t.g);
          }
          if (++s == GB_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted && leader)  // both CTAs' armed copies land (or the wait runs out) before leaving
        for (int i = 0; i < GB_STAGES; ++i)
          if ((armed >> i) & 1u) gb_drain(smem_u32(&ctl.full[i]), (armed_ph >> i) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool aborted = false;
      const uint32_t idesc = umma_idesc_bf16(2 * GB_BM, GB_BN) | (a.b_mn ? (1u << 16) : 0u);  // bit 16: B MN-major
      for (int u = pair; u < total && !aborted; u += npairs, ++it) {
        const GbTile t = decode(u);
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&ctl.tempty[acc]), aph ^ 1u, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * GB_BN);
        for (int kb = 0; kb < t.kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl.full[s]), ph, abort_flag, a.status)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * GB_STAGE_BYTES), sb = sa + GB_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < GB_BK / 16; ++kk) {
            // K-major: 16 k are 32 bytes along a row; N-major: 16 k are 16 rows of 128 bytes
            const uint64_t bdesc = a.b_mn ? sdesc_mn_sw128(sb + kk * 2048, 8192) : sdesc_k_sw128(sb + kk * 32);
            umma_bf16_cg2(d_tmem, sdesc_k_sw128(sa + kk * 32), bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_cg2_mc(smem_u32(&ctl.empty[s]), kPair);  // both CTAs' copies of the stage are free
          if (++s == GB_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        if (t.kb > 0) {
          umma_commit_cg2_mc(smem_u32(&ctl.tfull[acc]), kPair);  // both CTAs' accumulators are full
        } else {  // nothing to sum: both epilogues write zeros
          mbar_arrive_cluster(mapa_rank(smem_u32(&ctl.tfull[acc]), 0));
          mbar_arrive_cluster(mapa_rank(smem_u32(&ctl.tfull[acc]), 1));
        }
      }
      umma_commit_cg2_mc(smem_u32(&ctl.mma_done), kPair);
      gb_drain(smem_u32(&ctl.mma_done), 0);
    }
  } else {
    const int q = warp & 3;  // this warp reads TMEM lanes 32 q .. 32 q + 31 (its CTA's tile rows)
    int it = 0;
    for (int u = pair; u < total; u += npairs, ++it) {
      const GbTile t = decode(u);
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(&ctl.tfull[acc]), aph, abort_flag, a.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      // each 32 x 32 block goes through shared memory (16-byte chunks XOR-swizzled by row, so both
      // the row-wise writes and the column-wise reads are conflict-free): lane = row on the way
      // in, then 8 lanes per 128-byte row segment on the way out (coalesced stores)
      float* cbase = a.C + (a.rows_on_k ? (size_t)t.g * a.c_stride : 0) + (size_t)t.m0 * a.ldc + t.n0;
      const int rows_here = t.mrows - 32 * q;  // valid rows of this warp's quarter (may be <= 0)
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * GB_BN);
      float4* stg = reinterpret_cast<float4*>(epi + (size_t)q * 32 * 32);
#pragma unroll 1
      for (int c = 0; c < GB_BN / 32 && t.n0 + 32 * c < a.N; ++c) {
        uint32_t v[32];
        if (t.kb > 0) {
          tmem_ld32(tb + 32 * c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (a.rows_on_k) {  // the store that last read the staging block has finished reading it
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          stg[lane * 8 + (j ^ (lane & 7))] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                                         __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        if (a.rows_on_k) {
          // weight gradients: one asynchronous TMA store of the block (the layout above is the
          // tensor map's 128-byte swizzle); rows past M are clipped by the map
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && rows_here > 0) {
            tma_store_3d(&map_c, smem_u32(stg), t.n0 + 32 * c, t.m0 + 32 * q, t.g);
            bulk_commit();
          }
          __syncwarp();
          continue;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + (lane >> 3), ch = lane & 7;
          if (rr < rows_here) {
            float4 x = stg[rr * 8 + (ch ^ (rr & 7))];
            float4* dst = reinterpret_cast<float4*>(cbase + (size_t)(32 * q + rr) * a.ldc + 32 * c) + ch;
            if (a.beta) {
              const float4 o = *dst;
              x.x += o.x;
              x.y += o.y;
              x.z += o.z;
              x.w += o.w;
            }
            *dst = x;
          }
        }
        __syncwarp();
      }
      // the accumulator's reads have completed (tcgen05.wait::ld above): a plain remote arrive (no
      // cluster-wide release, which costs ~0.5 us) tells the leader it may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_rank(smem_u32(&ctl.tempty[acc]), 0));
    }
    if (lane == 0) bulk_wait_all();  // every tile store has completed before the CTA leaves
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // no signal of the peer can still be in flight towards this CTA, and neither CTA's TMEM is in
  // use, when the pair frees its TMEM together
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_cg2(tmem_base, GB_TMEM_COLS);
  }
}

// Pairs that fit the GPU at once (one CTA per SM): co-resident 2-CTA clusters of this kernel,
// asked once per device.
int max_pairs() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  if (ensure_smem_attr(reinterpret_cast<const void*>(k_gemm_bwd), GB_SMEM) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(GB_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GB_SMEM;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_bwd, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

cudaError_t launch_gb(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb2, const CUtensorMap& mc,
                      const GbArgs& a, long tiles_bound, cudaStream_t st) {
  if (tiles_bound <= 0) return cudaSuccess;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k_gemm_bwd), GB_SMEM);
  if (e != cudaSuccess) return e;
  const int npairs_max = max_pairs();
  if (npairs_max <= 0) return cudaErrorInvalidDevice;
  const long pairs = tiles_bound < npairs_max ? tiles_bound : npairs_max;
  k_gemm_bwd<<<(unsigned)(2 * pairs), GB_THREADS, GB_SMEM, st>>>(ma, mb, mb2, mc, a);  // cluster dims (2, 1, 1)
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

cudaError_t launch_gemm_bwd_rows_m_nmajor(const void* A, int rows_alloc, const void* B, const void* B2, int ksplit,
                                          int G_w, int N, int K, const int32_t* off, int G, int rows, float* C,
                                          int64_t ldc, int beta, uint32_t* status, cudaStream_t st, bool nmajor);

cudaError_t launch_gemm_bwd_rows_m(const void* A, int rows_alloc, const void* B, int G_w, int N, int K,
                                   const int32_t* off, int G, int rows, float* C, int64_t ldc, int beta,
                                   uint32_t* status, cudaStream_t st) {
  return launch_gemm_bwd_rows_m_nmajor(A, rows_alloc, B, nullptr, 0, G_w, N, K, off, G, rows, C, ldc, beta, status,
                                       st, false);
}

cudaError_t launch_gemm_bwd_rows_m_nmajor(const void* A, int rows_alloc, const void* B, const void* B2, int ksplit,
                                          int G_w, int N, int K, const int32_t* off, int G, int rows, float* C,
                                          int64_t ldc, int beta, uint32_t* status, cudaStream_t st, bool nmajor) {
  if (rows_alloc <= 0 || N <= 0) return cudaSuccess;
  if (K <= 0 || K % GB_BK || N % 32 || ldc % 4 || (off && (G < 1 || G > GB_MAXG)) || G_w < 1 || !aligned16(A) ||
      !aligned16(B) || !aligned16(C))
    return cudaErrorInvalidValue;
  if (nmajor && (N % 8 || ksplit <= 0 || ksplit % GB_BK || ksplit > K || (ksplit < K && !aligned16(B2))))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb, mb2;
  const cuuint64_t da[2] = {(cuuint64_t)K, (cuuint64_t)rows_alloc};
  const cuuint64_t sa[1] = {(cuuint64_t)K * 2};
  const cuuint32_t ba[2] = {GB_BK, GB_BM};
  if (!make_tmap_bf16(&ma, A, 2, da, sa, ba)) return cudaErrorInvalidValue;
  if (nmajor) {  // B_g(n, k) at [g][k][n]: boxes of 64 n by 64 k; the second tensor holds k >= ksplit
    const cuuint32_t bb[3] = {64, GB_BK, 1};
    const cuuint64_t db[3] = {(cuuint64_t)N, (cuuint64_t)ksplit, (cuuint64_t)G_w};
    const cuuint64_t sb[2] = {(cuuint64_t)N * 2, (cuuint64_t)N * ksplit * 2};
    if (!make_tmap_bf16(&mb, B, 3, db, sb, bb)) return cudaErrorInvalidValue;
    mb2 = mb;
    if (ksplit < K) {
      const cuuint64_t db2[3] = {(cuuint64_t)N, (cuuint64_t)(K - ksplit), (cuuint64_t)G_w};
      const cuuint64_t sb2[2] = {(cuuint64_t)N * 2, (cuuint64_t)N * (K - ksplit) * 2};
      if (!make_tmap_bf16(&mb2, B2, 3, db2, sb2, bb)) return cudaErrorInvalidValue;
    }
  } else {
    const cuuint64_t db[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)G_w};
    const cuuint64_t sb[2] = {(cuuint64_t)K * 2, (cuuint64_t)N * K * 2};
    const cuuint32_t bb[3] = {GB_BK, GB_BN / 2, 1};
    if (!make_tmap_bf16(&mb, B, 3, db, sb, bb)) return cudaErrorInvalidValue;
    mb2 = mb;
  }
  GbArgs a{};
  a.rows_on_k = 0;
  a.b_mn = nmajor ? 1 : 0;
  a.ksplit = nmajor ? ksplit : K;
  a.off = off;
  a.G = off ? G : 1;
  a.rows = rows;
  a.N = N;
  a.K = K;
  a.C = C;
  a.ldc = ldc;
  a.beta = beta;
  a.status = status;
  const long nt = (N + GB_BN - 1) / GB_BN;
  const long rt = off ? (long)(rows_alloc + 2 * GB_BM - 1) / (2 * GB_BM) + G : (long)(rows + 2 * GB_BM - 1) / (2 * GB_BM);
  return launch_gb(ma, mb, mb2, mb, a, rt * nt, st);  // (the C map is unused on rows on M)
}

cudaError_t launch_gemm_bwd_rows_k(const void* A, int M, const void* B, int N, int Kp, const int32_t* off, int G,
                                   int cols, float* C, int64_t ldc, int64_t c_stride, int beta, uint32_t* status,
                                   cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (Kp <= 0 || Kp % GB_BK || (!off && cols % GB_BK) || N % 32 || ldc % 4 || c_stride % 4 || beta ||
      (off && (G < 1 || G > GB_MAXG)) || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return cudaErrorInvalidValue;
  CUtensorMap ma, mb, mc;
  {  // C as [G][M][N] fp32 for the epilogue's 32 x 32 TMA stores
    const cuuint64_t dc[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)(off ? G : 1)};
    const cuuint64_t sc[2] = {(cuuint64_t)ldc * 4, (cuuint64_t)(c_stride > 0 ? c_stride : (int64_t)M * ldc) * 4};
    const cuuint32_t bc[3] = {32, 32, 1};
    if (!make_tmap_f32(&mc, C, 3, dc, sc, bc)) return cudaErrorInvalidValue;
  }
  const cuuint64_t da[2] = {(cuuint64_t)Kp, (cuuint64_t)M};
  const cuuint64_t db[2] = {(cuuint64_t)Kp, (cuuint64_t)N};
  const cuuint64_t s[1] = {(cuuint64_t)Kp * 2};
  const cuuint32_t ba[2] = {GB_BK, GB_BM}, bb[2] = {GB_BK, GB_BN / 2};
  if (!make_tmap_bf16(&ma, A, 2, da, s, ba) || !make_tmap_bf16(&mb, B, 2, db, s, bb)) return cudaErrorInvalidValue;
  GbArgs a{};
  a.rows_on_k = 1;
  a.off = off;
  a.G = off ? G : 1;
  a.rows = cols;
  a.M = M;
  a.N = N;
  a.C = C;
  a.ldc = ldc;
  a.c_stride = c_stride;
  a.beta = beta;
  a.status = status;
  a.ksplit = 0;
  const long tiles = (long)(off ? G : 1) * ((M + 2 * GB_BM - 1) / (2 * GB_BM)) * ((N + GB_BN - 1) / GB_BN);
  return launch_gb(ma, mb, mb, mc, a, tiles, st);
}

}  // namespace moe
