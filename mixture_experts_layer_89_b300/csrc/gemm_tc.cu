// Grouped expert projection on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Once tokens are grouped by expert, each expert's FFN is a dense matrix product over that
// expert's rows (the Naive-N0.5-Flash article, sec. 4.2, recommends exactly this grouping for
// inference), so the experts run here as one persistent grouped GEMM per projection:
//   up:   h = GELU(x_perm W_up^T + b_up)          or  h = SiLU(x_perm W_gate^T) * (x_perm W_up^T)
//   down: y_perm = h W_down^T (+ b_down)
// (expert forms: mini-moe tutorial, sec. 3.1; GPT-4 2% article, sec. 3.1).
//
// Tile: 128 rows x 256 accumulator columns, K step 64 (one 128-byte swizzle row of bf16).  For
// SwiGLU the 256 columns are 128 gate columns followed by the same 128 up columns, so one MMA
// (M=128, N=256, K=16) produces both halves and the epilogue multiplies them in registers.
// Warp roles (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: A tile (rows of one expert; only its 32-row groups when the tile
//               has few rows) + B tile (that expert's weights), 4 stages
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma per stage into a TMEM accumulator
//   warp 2      TMEM allocator (512 columns = two 256-column accumulators, double buffered)
//   warp 3      builds the tile table from the device-side expert offsets (no count returns to
//               the host)
//   warps 4..   EPIW epilogue warps: tcgen05.ld (thread = row), bias/activation, bf16 or fp32
//               32x32 tiles staged in swizzled shared memory and written by TMA tile stores.
//               Warp w reaches TMEM lanes 32 (w % 4)..; warps w, w + 4, ... split the columns.
// Paired mode (PAIR): 2-SM MMAs.  CTAs run in clusters of two that take the two 128-row halves of a
// 256-row tile of one expert; each holds its own 128 A rows and half of the 256 B rows in shared
// memory (32 KB per stage instead of 48, so 6 stages), and the even CTA issues
// tcgen05.mma.cta_group::2 (M=256) that reads both CTAs' operands and writes both CTAs' TMEM.
// Both CTAs' loads signal the leader's stage barriers; the leader's commits signal both CTAs'
// "stage free" and "accumulator full" barriers; both epilogues signal the leader's "accumulator
// free" barrier.  Per SM, operand traffic drops by a third for the same FLOPs.  Tiles are
// enumerated m-tile-major with n fastest (measured faster than n-major here).  Launched as a
// programmatic dependent launch: the set-up overlaps the previous kernel's tail.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BNB = 256;  // B rows per tile (accumulator columns)
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BNB * BK * 2;
constexpr int MAX_STAGES = 6;
// single CTA: A + the whole B tile per stage, 4 stages; pair: A + half of B per CTA, 6 stages
constexpr int stages_of(bool pair) { return pair ? 6 : 4; }
constexpr int stage_bytes_of(bool pair) { return A_BYTES + (pair ? B_BYTES / 2 : B_BYTES); }
constexpr int STAGE_REGION = 4 * (A_BYTES + B_BYTES);
static_assert(6 * (A_BYTES + B_BYTES / 2) == STAGE_REGION, "both stage layouts fill the same region");
constexpr int MAXG = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = umma_idesc_bf16(BM, BNB);
constexpr uint32_t IDESC_PAIR = umma_idesc_bf16(2 * BM, BNB);  // 2-SM MMA: M = 256 across the pair
constexpr uint16_t PAIR_MASK = 0x3;

struct TcArgs {
  const int32_t* offsets;
  int G;
  int rows_static;
  int N, K, N_w, K_w;
  const __nv_bfloat16* bias;
  void* out;  // bf16, or fp32 when the kernel's OUTF32 is set
  int64_t ldc;
  uint32_t* status;
};

struct SmemCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int u_pre[MAXG + 1];  // prefix over groups of row units (m-tiles, or m-tile pairs in PAIR mode)
};
// Epilogue staging for TMA tile stores: 32 x 32 tiles per warp (fp32 4 KB with the 128-byte
// swizzle, bf16 2 KB with the 64-byte swizzle), two per warp (the store of one chunk overlaps the
// staging of the next) except with 16 epilogue warps.  Shared memory: [alignment slack][stage
// region][staging][control].
constexpr int stg_bytes(bool outf32) { return outf32 ? 32 * 32 * 4 : 32 * 32 * 2; }
constexpr int stg_bufs(int epiw) { return epiw > 8 ? 1 : 2; }
constexpr size_t smem_total(bool outf32, int epiw) {
  return 1024 + (size_t)STAGE_REGION + (size_t)epiw * stg_bufs(epiw) * stg_bytes(outf32) + sizeof(SmemCtl);
}
static_assert(smem_total(true, 4) <= 232448 && smem_total(false, 16) <= 232448, "shared memory per CTA");

// Wait that ignores the abort flag (used to drain in-flight async operations before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Epilogue activations.  Their outputs are rounded to bf16 (relative spacing 2^-8), so they use
// the hardware exp2/reciprocal approximations (relative error ~1e-7) instead of IEEE expf/erff
// and division.
// GELU(u) = u Phi(u) with the complementary error function of Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (|error| <= 1.5e-7): for z >= 0,
// erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2), t = 1 / (1 + p z).  With
// z = |u| / sqrt 2 and g = |u| erfc(z) / 2:  u Phi(u) = u - g for u >= 0 and -g for u < 0, i.e.
// max(u, 0) - g in both cases.  Two columns at a time with the packed fp32x2 multiply-adds
// (the halved a_i fold the 1/2 into the polynomial); |u| is capped at 16 inside g, where
// erfc(16 / sqrt 2) underflows, so that u = +-inf gives inf / 0 rather than inf * 0.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float2 gelu_erf2(float2 u) {
  const float2 ax = make_float2(fabsf(u.x), fabsf(u.y));
  const float2 den = __ffma2_rn(ax, make_float2(0.3275911f * 0.70710678118654752f, 0.3275911f * 0.70710678118654752f),
                                make_float2(1.f, 1.f));
  const float2 t = make_float2(rcp_approx(den.x), rcp_approx(den.y));
  float2 poly = __ffma2_rn(t, make_float2(0.5f * 1.061405429f, 0.5f * 1.061405429f),
                           make_float2(0.5f * -1.453152027f, 0.5f * -1.453152027f));
  poly = __ffma2_rn(poly, t, make_float2(0.5f * 1.421413741f, 0.5f * 1.421413741f));
  poly = __ffma2_rn(poly, t, make_float2(0.5f * -0.284496736f, 0.5f * -0.284496736f));
  poly = __ffma2_rn(poly, t, make_float2(0.5f * 0.254829592f, 0.5f * 0.254829592f));
  poly = __fmul2_rn(poly, t);
  // exp(-z^2) = 2^(-u^2 log2(e) / 2)
  const float2 arg = __fmul2_rn(__fmul2_rn(u, u), make_float2(-0.72134752044448170f, -0.72134752044448170f));
  const float2 e = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
  const float2 g = __fmul2_rn(__fmul2_rn(make_float2(fminf(ax.x, 16.f), fminf(ax.y, 16.f)), poly), e);
  return __fadd2_rn(make_float2(fmaxf(u.x, 0.f), fmaxf(u.y, 0.f)), make_float2(-g.x, -g.y));
}
__device__ __forceinline__ float silu(float u) { return __fdividef(u, 1.f + __expf(-u)); }

// One warp's 32 rows x 32 bf16 columns (16 packed words per lane, lane = row): a TMA tile store
// through the warp's staging tile when all 32 rows are output rows (64-byte swizzle: 16-byte chunk
// j of row r sits at chunk j ^ ((r / 2) % 4), conflict-free), else direct row stores.
template <int NBUF>
__device__ __forceinline__ void store_bf16_chunk(const uint32_t (&pk)[16], bool full_rows, uint8_t* stg,
                                                 const CUtensorMap* tm, int col, int row0, __nv_bfloat16* dst_row,
                                                 int lane) {
  if (full_rows) {
    if (lane == 0) bulk_wait_read<NBUF - 1>();  // the store that last used stg has read it
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm, smem_u32(stg), col, row0);
      bulk_commit();
    }
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
}

template <int ACT, bool OUTF32, int EPIW, bool PAIR>
__global__ void __launch_bounds__(128 + 32 * EPIW, 1)
    k_proj_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA32,
              const __grid_constant__ CUtensorMap tmB0,
              const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmOut, const TcArgs args) {
  constexpr int NOUT = (ACT == ACT_SWIGLU) ? 128 : 256;
  constexpr int CW = NOUT / (EPIW / 4);  // output columns per epilogue warp
  constexpr int STAGES = stages_of(PAIR);
  constexpr int STAGE_BYTES = stage_bytes_of(PAIR);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = smem + (size_t)STAGE_REGION;  // 1024-byte aligned (the swizzle atoms)
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(stg_base + (size_t)EPIW * stg_bufs(EPIW) * stg_bytes(OUTF32));
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.offsets ? args.G : 1;
  const int n_tiles = (args.N + NOUT - 1) / NOUT;
  const int kblocks = args.K / BK;
  const int crank = PAIR ? (int)cluster_ctarank() : 0;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const bool leader = crank == 0;  // PAIR: the even CTA issues the 2-SM MMAs
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), PAIR ? 2 * EPIW : EPIW);  // one arrive per epilogue warp of the pair
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    if (!PAIR) tma_prefetch_desc(&tmA32);
    tma_prefetch_desc(&tmB0);
    if (ACT == ACT_SWIGLU) tma_prefetch_desc(&tmB1);
  }
  if (warp == 2) {
    if (PAIR) {  // both CTAs of the pair allocate together and receive the same address
      tmem_alloc_cg2(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish_cg2();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish();
    }
  }
  // the set-up above overlaps the previous kernel's tail; the offsets, the A rows and every output
  // buffer belong to earlier kernels from here on
  pdl_wait();
  if (warp == 3) {
    // unit prefix over groups: lane owns groups [8 lane, 8 lane + 8)
    int cnt[8];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int g = lane * 8 + i;
      cnt[i] = 0;
      if (g < G) {
        const int lo = args.offsets ? args.offsets[g] : 0;
        const int hi = args.offsets ? args.offsets[g + 1] : args.rows_static;
        const int mt = hi > lo ? (hi - lo + BM - 1) / BM : 0;
        cnt[i] = PAIR ? (mt + 1) >> 1 : mt;
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
      if (g < G) ctl->u_pre[g] = run;
      run += cnt[i];
    }
    if (lane == 31) ctl->u_pre[G] = incl;
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync_all();  // the peer's barriers are initialised before any remote signal
  tc_fence_after();

  const uint32_t tmem_base = ctl->tmem_base;
  const int total_units = ctl->u_pre[G] * n_tiles;

  // unit -> (group, first row, end of the group's rows, first output column); m-major, n fastest
  auto decode = [&](int u, int& g, int& m0, int& m_end, int& n0) {
    const int mu = u / n_tiles;
    const int nt = u - mu * n_tiles;
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl->u_pre[mid] <= mu) lo = mid; else hi = mid;
    }
    g = lo;
    const int mt_local = PAIR ? 2 * (mu - ctl->u_pre[g]) + crank : mu - ctl->u_pre[g];
    const int row_lo = args.offsets ? __ldg(args.offsets + g) : 0;
    m0 = row_lo + mt_local * BM;   // may lie past m_end in PAIR mode: nothing is stored
    m_end = args.offsets ? __ldg(args.offsets + g + 1) : args.rows_static;
    n0 = nt * NOUT;
  };

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      for (int u = unit0; u < total_units && !aborted; u += ustep) {
        int g, m0, m_end, n0;
        decode(u, g, m0, m_end, n0);
        const int nn = n0 % args.N_w;
        // single CTA: a tile with few rows (an expert with few tokens) loads only its 32-row groups
        // of A; the MMA rows past them read stale shared memory and give accumulator rows that are
        // never stored
        const int n32 = PAIR ? 4 : min(4, (max(m_end - m0, 1) + 31) >> 5);
        const uint32_t tx_bytes = (uint32_t)(STAGE_BYTES - (4 - n32) * (A_BYTES / 4));
        auto load_a = [&](uint8_t* sa, uint32_t fb, int k0) {
          if (n32 == 4) {
            tma_load_2d(smem_u32(sa), &tmA, fb, k0, m0);
          } else {
            for (int j = 0; j < n32; ++j) tma_load_2d(smem_u32(sa + j * (A_BYTES / 4)), &tmA32, fb, k0, m0 + 32 * j);
          }
        };
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          armed |= 1u << s;
          armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          const int k0 = kb * BK;
          const int gw = g + n0 / args.N_w + k0 / args.K_w;
          const int kk = k0 % args.K_w;
          uint8_t* sa = smem + (size_t)s * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          if (PAIR) {
            // this CTA's 128 A rows and its half of the B tile (SwiGLU: the gate or the up half;
            // else rows [128 crank, 128 crank + 128)), both signalling the leader's stage barrier
            const uint32_t lb = mapa_rank(fb, 0);
            if (leader) mbar_arrive_expect_tx(fb, 2 * STAGE_BYTES);
            tma_load_2d_cg2(smem_u32(sa), &tmA, lb, k0, m0);
            if (ACT == ACT_SWIGLU)
              tma_load_3d_cg2(smem_u32(sb), crank ? &tmB1 : &tmB0, lb, kk, nn, gw);
            else
              tma_load_3d_cg2(smem_u32(sb), &tmB0, lb, kk, nn + crank * (BNB / 2), gw);
          } else if (ACT == ACT_SWIGLU) {
            mbar_arrive_expect_tx(fb, tx_bytes);  // A (its existing rows) + the whole B tile
            load_a(sa, fb, k0);
            tma_load_3d(smem_u32(sb), &tmB0, fb, kk, nn, gw);
            tma_load_3d(smem_u32(sb + B_BYTES / 2), &tmB1, fb, kk, nn, gw);
          } else {
            mbar_arrive_expect_tx(fb, tx_bytes);
            load_a(sa, fb, k0);
            tma_load_3d(smem_u32(sb), &tmB0, fb, kk, nn, gw);
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted && leader) {  // let every armed copy (of both CTAs of a pair) land before leaving
        for (int i = 0; i < STAGES; ++i)
          if ((armed >> i) & 1u) drain_wait(smem_u32(&ctl->full[i]), (armed_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool aborted = false;
      for (int u = unit0; u < total_units && !aborted; u += ustep, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BNB);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (PAIR)
              umma_bf16_cg2(d_tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), IDESC_PAIR,
                            (kb | kk) != 0 ? 1u : 0u);
            else
              umma_bf16(d_tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), IDESC,
                        (kb | kk) != 0 ? 1u : 0u);
          }
          if (PAIR)
            umma_commit_cg2_mc(smem_u32(&ctl->empty[s]), PAIR_MASK);  // both CTAs' copies of the stage are free
          else
            umma_commit(smem_u32(&ctl->empty[s]));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        if (PAIR)
          umma_commit_cg2_mc(smem_u32(&ctl->tfull[acc]), PAIR_MASK);  // both CTAs' accumulators are full
        else
          umma_commit(smem_u32(&ctl->tfull[acc]));
      }
      if (PAIR)
        umma_commit_cg2_mc(smem_u32(&ctl->mma_done), PAIR_MASK);
      else
        umma_commit(smem_u32(&ctl->mma_done));
      drain_wait(smem_u32(&ctl->mma_done), 0);
    }
  } else if (warp >= 4) {
    const int q = warp & 3;                      // TMEM lanes 32q..32q+31 (a warp reaches only its quarter)
    const int c_lo = ((warp - 4) >> 2) * CW;     // this warp's share of the output columns
    constexpr int NBUF = stg_bufs(EPIW);
    uint8_t* stg_w = stg_base + (size_t)(warp - 4) * NBUF * stg_bytes(OUTF32);
    int chunk = 0;  // running chunk count of this warp: selects the staging buffer
    int it = 0;
    for (int u = unit0; u < total_units; u += ustep, ++it) {
      int g, m0, m_end, n0;
      decode(u, g, m0, m_end, n0);
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      // lane 0 waits, the warp follows its verdict (tcgen05.ld needs the whole warp converged)
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort_flag, args.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int row = m0 + q * 32 + lane;
      const bool valid = row < m_end;
      const bool full_rows = m0 + q * 32 + 32 <= m_end;  // all 32 rows of this warp are output rows
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BNB);
      const size_t orow = (size_t)(valid ? row : 0) * args.ldc;
      if (ACT == ACT_SWIGLU) {
#pragma unroll 1
        for (int c = c_lo; c < c_lo + CW; c += 32) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tb + c, gv);
          tmem_ld32(tb + 128 + c, uv);
          tmem_wait_ld();
          if (valid && n0 + c < args.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = silu(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]);
              const float h1 = silu(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]);
              pk[i] = pack_bf16x2(h0, h1);
            }
            store_bf16_chunk<NBUF>(pk, full_rows, stg_w + (chunk++ % NBUF) * stg_bytes(OUTF32), &tmOut, n0 + c,
                                   m0 + q * 32, static_cast<__nv_bfloat16*>(args.out) + orow + n0 + c, lane);
          }
        }
      } else {
#pragma unroll 1
        for (int c = c_lo; c < c_lo + CW; c += 32) {
          uint32_t v[32];
          tmem_ld32(tb + c, v);
          tmem_wait_ld();
          if (valid && n0 + c < args.N) {
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
            if (args.bias) {
              const int col = n0 + c;
              const int gw = g + col / args.N_w;
              const uint4* bp = reinterpret_cast<const uint4*>(args.bias + (size_t)gw * args.N_w + col % args.N_w);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint4 bq = bp[i];
                const uint32_t bw[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  f[8 * i + 2 * j] += __uint_as_float(bw[j] << 16);
                  f[8 * i + 2 * j + 1] += __uint_as_float(bw[j] & 0xffff0000u);
                }
              }
            }
            if (ACT == ACT_GELU) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float2 h2 = gelu_erf2(make_float2(f[i], f[i + 1]));
                f[i] = h2.x;
                f[i + 1] = h2.y;
              }
            }
            if (OUTF32 && full_rows) {
              // the warp's 32 rows x 32 columns go out as one TMA tile store through shared
              // memory (128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8))
              uint8_t* stg = stg_w + (chunk++ % NBUF) * stg_bytes(OUTF32);
              if (lane == 0) bulk_wait_read<NBUF - 1>();  // the store that last used stg has read it
              __syncwarp();
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                    make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmOut, smem_u32(stg), n0 + c, m0 + q * 32);
                bulk_commit();
              }
            } else if (OUTF32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.out) + orow + n0 + c);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            } else {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
              store_bf16_chunk<NBUF>(pk, full_rows, stg_w + (chunk++ % NBUF) * stg_bytes(OUTF32), &tmOut, n0 + c,
                                     m0 + q * 32, static_cast<__nv_bfloat16*>(args.out) + orow + n0 + c, lane);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(mapa_rank(smem_u32(&ctl->tempty[acc]), 0));  // the leader reuses the accumulator
        else
          mbar_arrive(smem_u32(&ctl->tempty[acc]));
      }
    }
    if (lane == 0) bulk_wait_all();  // tile stores complete before the CTA leaves
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // PAIR: no signal of the peer can still be in flight towards this CTA, and neither CTA's TMEM is
  // in use, when the pair frees its TMEM together
  if (PAIR) cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_cg2(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------- host side
}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Message of the last tensor-map failure on this host thread (tc_last_error).
static thread_local char g_err[256] = "";

// The driver's cuTensorMapEncodeTiled, looked up once (a function-local static: initialised once
// even when several host threads get here first together).
static EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

cudaError_t ensure_smem_attr(const void* kernel, size_t bytes) {
  // cudaFuncSetAttribute once per (kernel, device, size): it is a host call that need not repeat on
  // every launch (and is then also kept out of any stream capture after the first call).
  struct Entry { const void* k; int dev; size_t bytes; };
  static Entry seen[256];
  static int n_seen = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i].k == kernel && seen[i].dev == dev && seen[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && n_seen < 256) seen[n_seen++] = Entry{kernel, dev, bytes};
  return e;
}

static bool make_tmap(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides, const cuuint32_t* box,
                      CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    snprintf(g_err, sizeof(g_err), "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_err, sizeof(g_err), "cuTensorMapEncodeTiled failed (%d) rank %d dims %llu %llu %llu", (int)r, rank,
             (unsigned long long)dims[0], (unsigned long long)dims[1],
             rank > 2 ? (unsigned long long)dims[2] : 0ull);
    return false;
  }
  return true;
}

bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                    const cuuint32_t* box) {
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ptr, rank, dims, strides, box);
}

namespace {
// Largest number of co-resident 2-CTA clusters of a paired kernel (0 if none), per device.
template <typename K>
int max_pair_clusters(K kernel, int threads, size_t smem) {
  struct Entry { const void* k; int dev; int n; };
  static Entry seen[64];
  static int n_seen = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i].k == reinterpret_cast<const void*>(kernel) && seen[i].dev == dev) return seen[i].n;
  int n = 0;
  if (ensure_smem_attr(reinterpret_cast<const void*>(kernel), smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (n_seen < 64) seen[n_seen++] = Entry{reinterpret_cast<const void*>(kernel), dev, n};
  return n;
}

template <int ACT, bool OUTF32, int EPIW, bool PAIR>
cudaError_t launch_k(const CUtensorMap& mA, const CUtensorMap& mA32, const CUtensorMap& mB0, const CUtensorMap& mB1,
                     const CUtensorMap& mO,
                     const TcArgs& a, long grid, cudaStream_t st) {
  auto kern = k_proj_tc<ACT, OUTF32, EPIW, PAIR>;
  constexpr int threads = 128 + 32 * EPIW;
  constexpr size_t smem = smem_total(OUTF32, EPIW);
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  if (!PAIR) return launch_pdl(kern, dim3((unsigned)grid), dim3(threads), smem, st, mA, mA32, mB0, mB1, mO, a);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mA, mA32, mB0, mB1, mO, a);
}

template <int ACT, bool OUTF32>
cudaError_t launch_t(const Projection& p, uint32_t* status, int num_sms, cudaStream_t st) {
  constexpr int NOUT = (ACT == ACT_SWIGLU) ? 128 : 256;
  constexpr int EPIW = (ACT == ACT_GELU) ? 16 : 4;  // the erf epilogue is ALU-bound; the others are not
  const int rows_alloc = p.offsets ? p.rows_alloc : p.rows_static;
  if (rows_alloc <= 0 || p.N <= 0) return cudaSuccess;
  const int G = p.offsets ? p.G : 1;
  // Pairs pay off when groups average two or more row tiles (otherwise half the pair idles): a CTA
  // then holds 6 stages of half a B tile instead of 4 of a whole one, so more MMA work is in
  // flight per byte of shared memory while the tile loads are on their way.
  int n_clusters = 0;
  if ((long)rows_alloc >= 2L * BM * G)
    n_clusters = max_pair_clusters(k_proj_tc<ACT, OUTF32, EPIW, true>, 128 + 32 * EPIW, smem_total(OUTF32, EPIW));
  const bool pair = n_clusters > 0;
  CUtensorMap mA, mA32, mB0, mB1;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)rows_alloc};
    const cuuint64_t str[1] = {(cuuint64_t)p.lda * 2};
    const cuuint32_t box[2] = {BK, BM};
    if (!make_tmap_bf16(&mA, p.A, 2, dims, str, box)) return cudaErrorInvalidValue;
    const cuuint32_t box32[2] = {BK, 32};  // 32-row groups of A for tiles with few rows
    if (!make_tmap_bf16(&mA32, p.A, 2, dims, str, box32)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)p.K_w, (cuuint64_t)p.N_w, (cuuint64_t)p.G_w};
    const cuuint64_t str[2] = {(cuuint64_t)p.K_w * 2, (cuuint64_t)p.N_w * p.K_w * 2};
    const cuuint32_t box[3] = {BK, (cuuint32_t)((ACT == ACT_SWIGLU || pair) ? BNB / 2 : BNB), 1};
    if (!make_tmap_bf16(&mB0, p.B0, 3, dims, str, box)) return cudaErrorInvalidValue;
    if (ACT == ACT_SWIGLU) {
      if (!make_tmap_bf16(&mB1, p.B1, 3, dims, str, box)) return cudaErrorInvalidValue;
    } else {
      mB1 = mB0;
    }
  }
  CUtensorMap mO;
  {  // output tile map for the TMA stores of the epilogue: 32 x 32 boxes (fp32: 128-byte rows, bf16: 64-byte)
    const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)rows_alloc};
    const cuuint64_t str[1] = {(cuuint64_t)p.ldc * (OUTF32 ? 4 : 2)};
    const cuuint32_t box[2] = {32, 32};
    if (!make_tmap(&mO, OUTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.out, 2, dims,
                   str, box, OUTF32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  TcArgs a;
  a.offsets = p.offsets;
  a.G = p.G;
  a.rows_static = p.rows_static;
  a.N = p.N;
  a.K = p.K;
  a.N_w = p.N_w;
  a.K_w = p.K_w;
  a.bias = static_cast<const __nv_bfloat16*>(p.bias);
  a.out = p.out;
  a.ldc = p.ldc;
  a.status = status;
  const long n_tiles = (p.N + NOUT - 1) / NOUT;
  const long ub_mt = (rows_alloc + BM - 1) / BM + (p.offsets ? G : 0);  // each group adds <= 1 partial tile
  if (pair) {
    long units = (ub_mt + G + 1) / 2 * n_tiles;
    long clusters = units < n_clusters ? units : n_clusters;
    if (clusters < 1) clusters = 1;
    return launch_k<ACT, OUTF32, EPIW, true>(mA, mA32, mB0, mB1, mO, a, 2 * clusters, st);
  }
  long grid = ub_mt * n_tiles;
  if (grid > num_sms) grid = num_sms;
  if (grid < 1) grid = 1;
  return launch_k<ACT, OUTF32, EPIW, false>(mA, mA32, mB0, mB1, mO, a, grid, st);
}
}  // namespace

const char* tc_last_error() { return g_err; }

cudaError_t launch_projection_tc(const Projection& p, uint32_t* status, int num_sms, cudaStream_t st) {
  // hidden layers are bf16 (the next projection's MMA operand); projections to the model width
  // keep the fp32 accumulator so the layer output is rounded once
  switch (p.act) {
    case ACT_GELU: return launch_t<ACT_GELU, false>(p, status, num_sms, st);
    case ACT_SWIGLU: return launch_t<ACT_SWIGLU, false>(p, status, num_sms, st);
    default: return p.out_f32 ? launch_t<ACT_NONE, true>(p, status, num_sms, st)
                              : launch_t<ACT_NONE, false>(p, status, num_sms, st);
  }
}

}  // namespace moe
