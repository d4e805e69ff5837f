// Grouped expert projections on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Once tokens are grouped by expert, each expert's FFN is a dense matrix product over that
// expert's rows (the Naive-N0.5-Flash article, sec. 4.2, recommends exactly this grouping for
// inference), so the experts run as one persistent grouped GEMM per projection:
//   up:   h = GELU(x_perm W_up^T + b_up)          or  h = SiLU(x_perm W_gate^T) * (x_perm W_up^T)
//   down: y_perm = h W_down^T (+ b_down)
// (expert forms: mini-moe tutorial, sec. 3.1; GPT-4 2% article, sec. 3.1).  One launch may carry
// up to three such problems -- the routed experts, the always-on shared experts (FLAME-MoE
// summary, sec. 2) and a backup expert for assignments over capacity (mini-moe tutorial, sec. 6)
// -- whose tiles share the persistent CTAs.
//
// Orientation: the weights are the MMA's M side and the tokens its N side,
//   D[feature, token] = sum_k W[feature, k] X[token, k],
// so a tile always has 256 weight rows (the 2-SM MMA's M) and as many token rows as the expert
// has left, rounded up to 16 (the MMA's N step), at most 256.  An expert with 225 tokens costs a
// 240-column MMA instead of two 256-row tiles: each expert wastes at most 15 token rows.
//
// CTAs run in clusters of two (cta_group::2).  A tile is 256 weight rows x N token rows; CTA c of
// the pair holds weight rows [128c, 128c + 128) and token rows [c N/2, (c + 1) N/2) of each K step
// in its own shared memory, and the even CTA issues tcgen05.mma.cta_group::2 (M = 256) that reads
// both CTAs' operands; CTA c's TMEM receives the 128 x N accumulator of its own weight rows.
// SwiGLU: each CTA's 128 weight rows are the gate and the up rows of the same 64 features,
// interleaved in blocks of 16 (16 gate rows, their 16 up rows, ...), loaded as ONE box through a
// 5-D tensor map over (k, row in block, {gate, up}, block, expert) whose {gate, up} dimension
// strides from one weight tensor to the other; each 32-lane TMEM quarter then holds the gate and
// up accumulators of 16 features and one warp shuffle pairs them.  A pair tile covers 256 output
// features (GELU, down) or 128 (SwiGLU).  TMA boxes stay large throughout: a box's issue cost is
// nearly fixed, and splitting a stage into 8-row or 16-row boxes was measured 2-3x slower.
// Calls whose every group has at most 32 token rows (decode-sized batches) use a variant with
// 32-token tiles, whose small stages leave room for more weight bytes in flight.
//
// Warp roles (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: this CTA's weight rows and token rows of a K step, one box each
//               (6 stages of 32 KB, SwiGLU 7; decode-sized 10 of 18 KB), all signalling the even
//               CTA's stage barrier
//   warp 1      MMA issuer (one thread of the even CTA): tcgen05.mma per 16-wide K step into one
//               of two 256-column TMEM accumulators (double buffered: the epilogue of a tile
//               overlaps the next tile's MMAs)
//   warp 2      TMEM allocation (512 columns, both CTAs together)
//   warp 3      tile table from the device-side expert offsets (no count returns to the host)
//   warps 4..   EPIW epilogue warps: tcgen05.ld (thread = feature, registers = 32 tokens), bias,
//               activation, then the transposed 32-token x 32-feature block through shared memory
//               to a TMA tile store; blocks that reach past an expert's rows are stored directly
//               instead (SwiGLU always stores directly: each half-warp writes 32 contiguous bytes
//               of a token row).  Warp w reads TMEM lanes 32 (w % 4)..; warps w, w + 4, ... split
//               the token columns.
// 8-bit expert weights (INT8 or E4M3 codes with one fp32 scale per weight row; the mini-moe
// tutorial's deployment advice): warp 0 streams this CTA's raw weight boxes (one byte per weight)
// into a ring of its own, as deep as shared memory allows; warp 3 loads the token rows into the
// stage; converter warps (after the epilogue warps) widen each raw box exactly to bf16 -- into the
// swizzled shared-memory operand tile, or, for 32-token tiles, whose accumulators leave most of the
// tensor memory free, straight into tensor memory, from where the MMA reads its A operand -- and
// arrive on the pair leader's stage barrier; the epilogue multiplies each accumulator row by its
// weight row's scale.
// Tiles are ordered problem, expert, feature tile, token tile (token tiles fastest), so the pairs
// working at the same time share the weight tile in L2 and each weight tile is read from HBM once.
// Launched as a programmatic dependent launch: the set-up overlaps the previous kernel's tail.
// Every wait is bounded (one second); a CTA that gives up drains the copies and MMAs it started.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BK = 64;                          // K per stage: one 128-byte swizzle row of bf16
constexpr int AR = 128;                         // weight rows per CTA (the pair's M = 256)
constexpr int WBOX = AR * BK * 2;               // 16 KB: one weight tile of a CTA
constexpr int MAXP = 3;                         // problems per launch: routed, shared and backup experts
constexpr int MAXGT = 256 + 2;                  // groups over all problems
constexpr int TBL_PER_LANE = (MAXGT + 31) / 32;
constexpr int MAX_STAGES = 12;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint16_t PAIR_MASK = 0x3;

constexpr int SMEM_LIMIT = 232448;              // opt-in shared memory per CTA

// 8-bit expert weights (W8): the weight box of a K step arrives as one byte per weight in a ring
// of its own, and CONVW converter warps widen it to bf16 into the stage's swizzled operand tile
template <int ACT, int NTV> constexpr int conv_warps();
constexpr int RAW_BYTES = AR * BK;              // 8 KB: one CTA's 8-bit weight tile of a K step
constexpr int MAX_RAW = 24;

template <int ACT> constexpr int epi_warps() { return ACT == ACT_GELU ? 16 : 4; }  // the erf epilogue is ALU-bound
// converter warps: 8 (two per TMEM quarter when they widen into tensor memory), 4 beside the
// 16-warp GELU epilogue; measured, 16 warps were slower on both paths
template <int ACT, int NTV> constexpr int conv_warps() { return epi_warps<ACT>() > 8 ? 4 : 8; }
template <int ACT, int NTV, bool W8> constexpr int n_threads() {
  return 128 + 32 * (epi_warps<ACT>() + (W8 ? conv_warps<ACT, NTV>() : 0));
}
template <int ACT> constexpr bool out_f32() { return ACT == ACT_NONE; }           // projections to the model width
template <int ACT> constexpr int feat_per_tile() { return ACT == ACT_SWIGLU ? AR : 2 * AR; }  // output features per pair tile
// token rows per tile: NTV (256, or 32 for decode-sized calls)
template <int ACT, int NTV> constexpr int tile_tokens() { return NTV; }
template <int ACT, int NTV> constexpr int a_bytes() { return WBOX; }
template <int ACT, int NTV> constexpr int b_bytes() { return tile_tokens<ACT, NTV>() / 2 * BK * 2; }
template <int ACT, int NTV> constexpr int stage_bytes() { return a_bytes<ACT, NTV>() + b_bytes<ACT, NTV>(); }
// 8-bit weights: a ring of raw weight boxes (as deep as shared memory allows: the bytes in flight
// from HBM) feeds the stage ring, whose stages hold the widened bf16 weight tile and the token rows.
// Decode-sized calls (32-token tiles, whose accumulators need 32 TMEM columns each) widen the weights
// into tensor memory instead, which the MMA reads as its A operand: the stages then hold only the
// token rows, and widening adds no shared-memory traffic beside the tensor cores' operand reads.
template <int NTV, bool W8> constexpr bool a_in_tmem() { return W8 && NTV <= 32; }
template <int NTV, bool W8> constexpr int acc_cols() { return a_in_tmem<NTV, W8>() ? 32 : 256; }
template <int ACT, int NTV, bool W8> constexpr int stage_bytes_of() {
  return a_in_tmem<NTV, W8>() ? b_bytes<ACT, NTV>() : stage_bytes<ACT, NTV>();
}
// epilogue staging per warp: fp32 32 x 32 (128-byte rows) or bf16 32 x 32 (64-byte rows); two
// buffers per warp except with 16 warps; none for SwiGLU, which stores straight from registers
template <int ACT> constexpr int stg_bytes() { return ACT == ACT_NONE ? 4096 : 2048; }
template <int ACT> constexpr int stg_bufs() { return ACT == ACT_SWIGLU ? 0 : (epi_warps<ACT>() > 8 ? 1 : 2); }
constexpr int CTL_BYTES = 2048;  // >= sizeof(SmemCtl), checked below
template <int ACT> constexpr int stg_total() { return epi_warps<ACT>() * stg_bufs<ACT>() * stg_bytes<ACT>(); }
// bf16 operand stages: as many as fit (at most MAX_STAGES); with 8-bit weights a few, the bytes in
// flight from HBM being the raw ring's
template <int ACT, int NTV, bool W8 = false> constexpr int n_stages() {
  return W8 ? (NTV <= 32 ? 12 : 3)
             : ((SMEM_LIMIT - 1024 - CTL_BYTES - stg_total<ACT>()) / stage_bytes<ACT, NTV>() < MAX_STAGES
                    ? (SMEM_LIMIT - 1024 - CTL_BYTES - stg_total<ACT>()) / stage_bytes<ACT, NTV>()
                    : MAX_STAGES);
}
template <int ACT, int NTV, bool W8> constexpr int w8_fixed_bytes() {
  return n_stages<ACT, NTV, W8>() * stage_bytes_of<ACT, NTV, W8>();
}
template <int ACT, int NTV, bool W8> constexpr int raw_stages() {
  return !W8 ? 0
             : ((SMEM_LIMIT - 1024 - CTL_BYTES - stg_total<ACT>() - w8_fixed_bytes<ACT, NTV, W8>()) / RAW_BYTES < MAX_RAW
                    ? (SMEM_LIMIT - 1024 - CTL_BYTES - stg_total<ACT>() - w8_fixed_bytes<ACT, NTV, W8>()) / RAW_BYTES
                    : MAX_RAW);
}

struct ProbArgs {
  const int32_t* offsets;  // [G+1] device, or NULL: one group of rows [0, rows_static)
  int G, rows_static;
  int N, K, N_w, K_w;      // weight for feature n, reduction index kk of group g: matrix g + n / N_w + kk / K_w
  const __nv_bfloat16* bias;  // [G_w][N_w] or NULL
  void* out;
  int64_t ldc;
  int gate_first;          // SwiGLU: the gate rows come first in each 32-row group (else the up rows)
  const float* scale0;     // 8-bit weights: fp32 scale of each row of B0 (SwiGLU: the gate) and of
  const float* scale1;     // B1 (SwiGLU: the up rows), indexed like the bias
};
struct TcArgs {
  ProbArgs p[MAXP];
  int nprob;
  int wfmt;                // 8-bit weights: 1 int8, 2 E4M3 (0 otherwise)
  uint32_t* status;
};
// Tensor maps of each problem: weights (SwiGLU: gate and up together), token rows in boxes of
// NT/2 and 32 rows, and the output.
struct TcMaps {
  CUtensorMap w0[MAXP], x[MAXP], x32[MAXP], o[MAXP];
};

struct SmemCtl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t raw_full[MAX_RAW];   // 8-bit weights, slot ring: raw box loaded / widened
  uint64_t raw_empty[MAX_RAW];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int g0, g01;          // groups of problem 0, of problems 0 and 1
  int gt;               // groups over all problems
  int u_pre[MAXGT + 1]; // prefix over groups of their tiles
};
static_assert(sizeof(SmemCtl) <= CTL_BYTES, "control block");
template <int ACT, int NTV, bool W8 = false>
constexpr size_t smem_total() {
  return 1024 + (size_t)n_stages<ACT, NTV, W8>() * stage_bytes_of<ACT, NTV, W8>() +
         (size_t)raw_stages<ACT, NTV, W8>() * RAW_BYTES + (size_t)stg_total<ACT>() + CTL_BYTES;
}
// TMEM columns: two accumulators, then (A in TMEM) one 32-column bf16 weight tile per stage
template <int ACT, int NTV, bool W8> constexpr int tmem_cols_used() {
  return 2 * acc_cols<NTV, W8>() + (a_in_tmem<NTV, W8>() ? n_stages<ACT, NTV, W8>() * (BK / 2) : 0);
}
static_assert(smem_total<ACT_NONE, 256>() <= SMEM_LIMIT && smem_total<ACT_GELU, 256>() <= SMEM_LIMIT &&
                  smem_total<ACT_SWIGLU, 256>() <= SMEM_LIMIT && smem_total<ACT_SWIGLU, 32>() <= SMEM_LIMIT,
              "shared memory per CTA");
static_assert(smem_total<ACT_NONE, 256, true>() <= SMEM_LIMIT && smem_total<ACT_GELU, 256, true>() <= SMEM_LIMIT &&
                  smem_total<ACT_SWIGLU, 256, true>() <= SMEM_LIMIT && smem_total<ACT_SWIGLU, 32, true>() <= SMEM_LIMIT &&
                  smem_total<ACT_NONE, 32, true>() <= SMEM_LIMIT && smem_total<ACT_GELU, 32, true>() <= SMEM_LIMIT,
              "shared memory per CTA (8-bit weights)");
static_assert(tmem_cols_used<ACT_SWIGLU, 32, true>() <= (int)TMEM_COLS && tmem_cols_used<ACT_NONE, 32, true>() <= (int)TMEM_COLS &&
                  tmem_cols_used<ACT_SWIGLU, 256, false>() <= (int)TMEM_COLS,
              "tensor memory columns");
static_assert(raw_stages<ACT_SWIGLU, 32, true>() >= 16 && raw_stages<ACT_NONE, 32, true>() >= 12 &&
                  raw_stages<ACT_NONE, 256, true>() >= 8 && raw_stages<ACT_GELU, 256, true>() >= 8 &&
                  raw_stages<ACT_SWIGLU, 256, true>() >= 12,
              "8-bit weight bytes in flight");
static_assert(n_stages<ACT_NONE, 256>() == 6 && n_stages<ACT_SWIGLU, 256>() == 7 && n_stages<ACT_NONE, 32>() >= 10,
              "stage counts");

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
// max(u, 0) - g in both cases.  Two values at a time with the packed fp32x2 multiply-adds
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

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint16_t bf16_bits(float v) {
  const __nv_bfloat16 b = __float2bfloat16_rn(v);
  return *reinterpret_cast<const uint16_t*>(&b);
}

// ------------------------------------------------------------- 8-bit weights widened to bf16
// int8: q + 128 (the byte with its top bit flipped) placed in the low mantissa byte of 2^23 gives
// the float 2^23 + q + 128 exactly; subtracting 2^23 + 128 leaves q, which bf16 holds exactly.
__device__ __forceinline__ void int8x4_to_bf16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = x ^ 0x80808080u;
  const float2 a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                                          __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                              make_float2(-8388736.f, -8388736.f));
  const float2 b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                                          __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                              make_float2(-8388736.f, -8388736.f));
  lo = pack_bf16x2(a.x, a.y);
  hi = pack_bf16x2(b.x, b.y);
}
// E4M3: the hardware conversion to f16 is exact (every E4M3 value is a normal f16 or zero); moving
// the f16 exponent and mantissa fields down by 3 bits (the sign stays) gives the bf16 whose value
// is the f16's times 2^-112 (the two formats' exponent biases differ by 112), and one bf16x2
// multiply by 2^112 restores it -- exactly, zero included.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t pair) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)pair));
  const uint32_t t = ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x77807780u));  // 0x7780 = 2^112
  return r;
}
// One CTA's 8-bit weight tile (AR rows of BK bytes, row-major) -> the bf16 operand tile (AR rows
// of 128 bytes, 16-byte chunk j of row i at chunk j ^ (i % 8), the layout TMA's 128-byte swizzle
// writes).  Thread ct of the CONVW converter warps widens 16 weights per item; a warp's loads cover
// 512 contiguous bytes and its stores hit every bank once per quarter warp.  All loads of a thread
// are issued before its first conversion (plain shared-memory accesses, so the compiler may
// overlap them).
template <int CONVW>
__device__ __forceinline__ void widen_tile(const uint8_t* raw, uint8_t* dst, int ct, int fmt) {
  constexpr int ITEMS = AR * (BK / 16) / (CONVW * 32);
  uint4 v[ITEMS];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int item = it * CONVW * 32 + ct;
    v[it] = *reinterpret_cast<const uint4*>(raw + (item >> 2) * BK + (item & 3) * 16);
  }
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int item = it * CONVW * 32 + ct;
    const int row = item >> 2, piece = item & 3;
    uint32_t o[8];
    if (fmt == 1) {
      int8x4_to_bf16(v[it].x, o[0], o[1]);
      int8x4_to_bf16(v[it].y, o[2], o[3]);
      int8x4_to_bf16(v[it].z, o[4], o[5]);
      int8x4_to_bf16(v[it].w, o[6], o[7]);
    } else {
      o[0] = e4m3x2_to_bf16x2(v[it].x & 0xFFFFu);
      o[1] = e4m3x2_to_bf16x2(v[it].x >> 16);
      o[2] = e4m3x2_to_bf16x2(v[it].y & 0xFFFFu);
      o[3] = e4m3x2_to_bf16x2(v[it].y >> 16);
      o[4] = e4m3x2_to_bf16x2(v[it].z & 0xFFFFu);
      o[5] = e4m3x2_to_bf16x2(v[it].z >> 16);
      o[6] = e4m3x2_to_bf16x2(v[it].w & 0xFFFFu);
      o[7] = e4m3x2_to_bf16x2(v[it].w >> 16);
    }
    uint8_t* base = dst + row * 128;
    const int sw = row & 7;
    *reinterpret_cast<uint4*>(base + (((2 * piece) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(base + (((2 * piece + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// (A in TMEM) Thread `lane` of a converter warp in TMEM quarter q widens its row 32q + lane of the
// CTA's raw weight box -- the KPW weights [k0, k0 + KPW) -- into 32-bit TMEM columns (two weights
// each) starting at taddr.  The raw box is laid out by TMA's 64-byte swizzle (16-byte chunk c of
// row r at chunk c ^ ((r / 2) % 4)), so the quarter warp's loads of one chunk hit distinct banks.
template <int KPW>
__device__ __forceinline__ void widen_to_tmem(const uint8_t* raw, int row, int k0, uint32_t taddr, int fmt) {
  constexpr int CH = KPW / 16;  // 16-byte chunks of the thread's row
  uint4 v[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int chunk = (k0 / 16 + c) ^ ((row >> 1) & 3);
    v[c] = *reinterpret_cast<const uint4*>(raw + row * BK + chunk * 16);
  }
  uint32_t o[CH * 8];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    {
      const uint4 w = v[c];
      uint32_t* d = o + 8 * c;
      if (fmt == 1) {
        int8x4_to_bf16(w.x, d[0], d[1]);
        int8x4_to_bf16(w.y, d[2], d[3]);
        int8x4_to_bf16(w.z, d[4], d[5]);
        int8x4_to_bf16(w.w, d[6], d[7]);
      } else {
        d[0] = e4m3x2_to_bf16x2(w.x & 0xFFFFu);
        d[1] = e4m3x2_to_bf16x2(w.x >> 16);
        d[2] = e4m3x2_to_bf16x2(w.y & 0xFFFFu);
        d[3] = e4m3x2_to_bf16x2(w.y >> 16);
        d[4] = e4m3x2_to_bf16x2(w.z & 0xFFFFu);
        d[5] = e4m3x2_to_bf16x2(w.z >> 16);
        d[6] = e4m3x2_to_bf16x2(w.w & 0xFFFFu);
        d[7] = e4m3x2_to_bf16x2(w.w >> 16);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < CH; ++c) tmem_st8(taddr + 8 * c, o + 8 * c);
}

struct Tile {
  int p, g;        // problem, group (expert) within it
  int m0, m_end;   // first token row of the tile, end of the group's rows
  int n0;          // first output feature of the pair tile
  int ntok, nmma;  // token rows of the tile, and that rounded up to the MMA's N step of 16
  int kblocks;
};

template <int ACT, int NTV, bool W8>
__global__ void __launch_bounds__(n_threads<ACT, NTV, W8>(), 1)
    k_proj_tc(const __grid_constant__ TcMaps maps, const __grid_constant__ TcArgs args) {
  constexpr int EPIW = epi_warps<ACT>();
  constexpr int CONVW = conv_warps<ACT, NTV>();
  constexpr int NBUF = stg_bufs<ACT>() > 0 ? stg_bufs<ACT>() : 1;  // (SwiGLU stages nothing)
  constexpr int STG = stg_bytes<ACT>();
  constexpr int NT = tile_tokens<ACT, NTV>();
  constexpr int FT = feat_per_tile<ACT>();
  constexpr int A_BYTES = a_bytes<ACT, NTV>();
  constexpr bool TA = a_in_tmem<NTV, W8>();    // A operand widened into tensor memory
  constexpr int ACC_COLS = acc_cols<NTV, W8>();
  constexpr uint32_t A_COL0 = 2 * ACC_COLS;      // (TA) first column of the stages' weight tiles
  constexpr int STAGE_BYTES = stage_bytes_of<ACT, NTV, W8>();
  constexpr int B_OFF = TA ? 0 : A_BYTES;        // token rows within a stage
  constexpr int STAGES = n_stages<ACT, NTV, W8>();
  constexpr int RAWST = raw_stages<ACT, NTV, W8>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw_base = smem + (size_t)STAGES * STAGE_BYTES;  // W8: the raw weight ring
  uint8_t* stg_base = raw_base + (size_t)RAWST * RAW_BYTES; // 1024-byte aligned (the swizzle atoms)
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(stg_base + (size_t)EPIW * stg_bufs<ACT>() * STG);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const bool leader = crank == 0;  // the even CTA issues the 2-SM MMAs
  const int unit0 = (int)(blockIdx.x >> 1);
  const int ustep = (int)(gridDim.x >> 1);
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // W8: every converter warp of the pair arrives once the stage's weights are widened, and the
      // leader's token-row thread once it has armed both CTAs' token-row bytes
      mbar_init(smem_u32(&ctl->full[s]), W8 ? 2 * CONVW + 1 : 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int r = 0; r < RAWST; ++r) {
      mbar_init(smem_u32(&ctl->raw_full[r]), 1);
      mbar_init(smem_u32(&ctl->raw_empty[r]), CONVW);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), 2 * EPIW);  // one arrive per epilogue warp of the pair
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < args.nprob; ++p) {
      tma_prefetch_desc(&maps.w0[p]);
      tma_prefetch_desc(&maps.x[p]);
    }
  }
  if (warp == 2) {  // both CTAs of the pair allocate together and receive the same address
    tmem_alloc_cg2(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish_cg2();
  }
  // the set-up above overlaps the previous kernel's tail; the offsets, the token rows and every
  // output buffer belong to earlier kernels from here on
  pdl_wait();
  if (warp == 3) {
    // tiles of every group over both problems: lane owns groups [TBL_PER_LANE lane, + TBL_PER_LANE)
    const int g0 = args.p[0].offsets ? args.p[0].G : 1;
    const int g1 = args.nprob > 1 ? (args.p[1].offsets ? args.p[1].G : 1) : 0;
    const int g2 = args.nprob > 2 ? (args.p[2].offsets ? args.p[2].G : 1) : 0;
    const int gt = g0 + g1 + g2;
    int cnt[TBL_PER_LANE];
    int local = 0;
#pragma unroll
    for (int i = 0; i < TBL_PER_LANE; ++i) {
      const int g = lane * TBL_PER_LANE + i;
      cnt[i] = 0;
      if (g < gt) {
        const int p = g < g0 ? 0 : (g < g0 + g1 ? 1 : 2);
        const ProbArgs& P = args.p[p];
        const int gl = g - (p == 0 ? 0 : (p == 1 ? g0 : g0 + g1));
        const int lo = P.offsets ? P.offsets[gl] : 0;
        const int hi = P.offsets ? P.offsets[gl + 1] : P.rows_static;
        const int tt = hi > lo ? (hi - lo + NT - 1) / NT : 0;
        cnt[i] = tt * ((P.N + FT - 1) / FT);
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
    for (int i = 0; i < TBL_PER_LANE; ++i) {
      const int g = lane * TBL_PER_LANE + i;
      if (g < gt) ctl->u_pre[g] = run;
      run += cnt[i];
    }
    if (lane == 31) {
      ctl->u_pre[gt] = incl;
      ctl->g0 = g0;
      ctl->g01 = g0 + g1;
      ctl->gt = gt;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote signal
  tc_fence_after();

  const uint32_t tmem_base = ctl->tmem_base;
  const int n_groups = ctl->gt;
  const int total_units = ctl->u_pre[n_groups];

  auto decode = [&](int u) {
    int lo = 0, hi = n_groups;  // the largest group whose first tile is <= u
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl->u_pre[mid] <= u) lo = mid; else hi = mid;
    }
    Tile t;
    t.p = lo < ctl->g0 ? 0 : (lo < ctl->g01 ? 1 : 2);
    t.g = lo - (t.p == 0 ? 0 : (t.p == 1 ? ctl->g0 : ctl->g01));
    const ProbArgs& P = args.p[t.p];
    const int r0 = P.offsets ? __ldg(P.offsets + t.g) : 0;
    t.m_end = P.offsets ? __ldg(P.offsets + t.g + 1) : P.rows_static;
    const int tt = (t.m_end - r0 + NT - 1) / NT;
    const int local = u - ctl->u_pre[lo];
    const int fi = local / tt;
    const int ti = local - fi * tt;
    t.m0 = r0 + ti * NT;
    t.ntok = min(NT, t.m_end - t.m0);
    t.nmma = (t.ntok + 15) & ~15;
    t.n0 = fi * FT;
    t.kblocks = P.K / BK;
    return t;
  };

  if (W8 && warp == 0) {
    // 8-bit weights: this CTA's raw weight box of every K step (own barrier), as soon as the
    // converters have widened the slot's previous box
    if (lane == 0) {
      int r = 0;
      uint32_t rph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      for (int u = unit0; u < total_units && !aborted; u += ustep) {
        const Tile t = decode(u);
        const ProbArgs& P = args.p[t.p];
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->raw_empty[r]), rph ^ 1u, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->raw_full[r]);
          mbar_arrive_expect_tx(fb, RAW_BYTES);
          armed |= 1u << r;
          armed_ph = (armed_ph & ~(1u << r)) | (rph << r);
          const int k0 = kb * BK;
          const int kk = k0 % P.K_w;
          const int kq = k0 / P.K_w;
          const uint32_t dst = smem_u32(raw_base + (size_t)r * RAW_BYTES);
          if (ACT == ACT_SWIGLU) {
            const int f = t.n0 + (AR / 2) * crank;
            tma_load_5d(dst, &maps.w0[t.p], fb, kk, 0, 0, (f % P.N_w) / 16, t.g + f / P.N_w + kq);
          } else {
            const int f = t.n0 + AR * crank;
            tma_load_3d(dst, &maps.w0[t.p], fb, kk, f % P.N_w, t.g + f / P.N_w + kq);
          }
          if (++r == RAWST) {
            r = 0;
            rph ^= 1u;
          }
        }
      }
      if (aborted) {  // this CTA's own copies land before it leaves
        for (int i = 0; i < RAWST; ++i)
          if ((armed >> i) & 1u) drain_wait(smem_u32(&ctl->raw_full[i]), (armed_ph >> i) & 1u);
      }
    }
  } else if (W8 && warp == 3) {
    // 8-bit weights: this CTA's token rows of every K step into the stage, once the MMAs have
    // read it (the leader arms its stage barrier with both CTAs' bytes)
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      for (int u = unit0; u < total_units && !aborted; u += ustep) {
        const Tile t = decode(u);
        const int half = t.nmma >> 1;
        const int brow = t.m0 + crank * half;
        const bool small_box = NT / 2 > 32 && half <= 32;
        const uint32_t b_tx = 2u * (uint32_t)((small_box ? 32 : NT / 2) * BK * 2);  // both CTAs' token rows
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          if (leader) {
            mbar_arrive_expect_tx(fb, b_tx);
            armed |= 1u << s;
            armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          }
          const uint32_t dst = smem_u32(smem + (size_t)s * STAGE_BYTES + B_OFF);
          if (small_box)
            tma_load_2d_cg2(dst, &maps.x32[t.p], mapa_rank(fb, 0), kb * BK, brow);
          else
            tma_load_2d_cg2(dst, &maps.x[t.p], mapa_rank(fb, 0), kb * BK, brow);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted && leader) {  // both CTAs' armed token-row copies land (or the wait runs out)
        for (int i = 0; i < STAGES; ++i)
          if ((armed >> i) & 1u) drain_wait(smem_u32(&ctl->full[i]), (armed_ph >> i) & 1u);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      bool aborted = false;
      for (int u = unit0; u < total_units && !aborted; u += ustep) {
        const Tile t = decode(u);
        const ProbArgs& P = args.p[t.p];
        const int half = t.nmma >> 1;   // token rows of this CTA (a multiple of 8)
        const int brow = t.m0 + crank * half;
        // one token box per stage: 32 rows when this CTA's half fits, else the full NT/2 rows
        const bool small_box = NT / 2 > 32 && half <= 32;
        const uint32_t stage_tx = 2u * (uint32_t)(A_BYTES + (small_box ? 32 : NT / 2) * BK * 2);  // both CTAs' bytes
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          const uint32_t lb = mapa_rank(fb, 0);
          if (leader) {
            mbar_arrive_expect_tx(fb, stage_tx);
            armed |= 1u << s;
            armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          }
          const int k0 = kb * BK;
          const int kk = k0 % P.K_w;
          const int kq = k0 / P.K_w;
          uint8_t* sa = smem + (size_t)s * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          if (ACT == ACT_SWIGLU) {
            // this CTA's 64 features: gate and up rows interleaved in blocks of 16, one box
            const int f = t.n0 + (AR / 2) * crank;
            tma_load_5d_cg2(smem_u32(sa), &maps.w0[t.p], lb, kk, 0, 0, (f % P.N_w) / 16, t.g + f / P.N_w + kq);
          } else {
            const int f = t.n0 + AR * crank;
            tma_load_3d_cg2(smem_u32(sa), &maps.w0[t.p], lb, kk, f % P.N_w, t.g + f / P.N_w + kq);
          }
          if (small_box)
            tma_load_2d_cg2(smem_u32(sb), &maps.x32[t.p], lb, k0, brow);
          else
            tma_load_2d_cg2(smem_u32(sb), &maps.x[t.p], lb, k0, brow);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (aborted && leader) {  // let every armed copy (of both CTAs) land before leaving
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
        const Tile t = decode(u);
        const int acc = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
        const uint32_t idesc = umma_idesc_bf16(2 * AR, t.nmma);
        for (int kb = 0; kb < t.kblocks; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, args.status)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)s * STAGE_BYTES);
          const uint32_t sb = sa + B_OFF;
          if (TA) {
            const uint32_t a_tmem = tmem_base + A_COL0 + (uint32_t)(s * (BK / 2));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16_cg2_ta(d_tmem, a_tmem + kk * 8, sdesc_k_sw128(sb + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16_cg2(d_tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), idesc,
                            (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_cg2_mc(smem_u32(&ctl->empty[s]), PAIR_MASK);  // both CTAs' copies of the stage are free
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (aborted) break;
        umma_commit_cg2_mc(smem_u32(&ctl->tfull[acc]), PAIR_MASK);  // both CTAs' accumulators are full
      }
      umma_commit_cg2_mc(smem_u32(&ctl->mma_done), PAIR_MASK);
      drain_wait(smem_u32(&ctl->mma_done), 0);
    }
  } else if (W8 && warp >= 4 + EPIW) {
    // converter warps (8-bit weights): per K step, once the bf16 tile of the stage is free and the
    // slot's raw box has landed, widen the box into it and arrive on the leader's stage barrier
    const int cw = warp - 4 - EPIW;
    const int ct = cw * 32 + lane;
    int s = 0, r = 0;
    uint32_t ph = 0, rph = 0;
    bool aborted = false;
    for (int u = unit0; u < total_units && !aborted; u += ustep) {
      const Tile t = decode(u);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        int ok = 1;
        if (lane == 0)
          ok = (mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, args.status) &&
                mbar_wait_bounded(smem_u32(&ctl->raw_full[r]), rph, abort_flag, args.status))
                   ? 1
                   : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          aborted = true;
          break;
        }
        if (TA) {
          // this warp: TMEM quarter q (its rows 32q..32q+31) and the weights [k0, k0 + KPW) of them
          constexpr int KPW = BK / (CONVW / 4);
          const int q = warp & 3;
          const int k0 = (cw >> 2) * KPW;
          tc_fence_after();  // the MMAs that read this stage's tile before have completed
          widen_to_tmem<KPW>(raw_base + (size_t)r * RAW_BYTES, 32 * q + lane, k0,
                             tmem_base + ((uint32_t)(32 * q) << 16) + A_COL0 + (uint32_t)(s * (BK / 2) + k0 / 2),
                             args.wfmt);
          tmem_wait_st();
          tc_fence_before();
        } else {
          widen_tile<CONVW>(raw_base + (size_t)r * RAW_BYTES, smem + (size_t)s * STAGE_BYTES, ct, args.wfmt);
          fence_proxy_async_smem();  // the widened tile is read by the tensor cores (async proxy)
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&ctl->raw_empty[r]));
          mbar_arrive_remote(mapa_rank(smem_u32(&ctl->full[s]), 0));
        }
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
        if (++r == RAWST) {
          r = 0;
          rph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 4 + EPIW) {
    const int q = warp & 3;                  // TMEM lanes 32q..32q+31 (a warp reaches only its quarter)
    const int grp = (warp - 4) >> 2;         // this warp's share of the token columns
    constexpr int NGRP = EPIW / 4;
    uint8_t* stg_w = stg_base + (size_t)(warp - 4) * NBUF * STG;
    int chunk = 0;                           // running count of staged blocks: selects the buffer
    int it = 0;
    for (int u = unit0; u < total_units; u += ustep, ++it) {
      const Tile t = decode(u);
      const ProbArgs& P = args.p[t.p];
      const int acc = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      // lane 0 waits, the warp follows its verdict (tcgen05.ld needs the whole warp converged)
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(smem_u32(&ctl->tfull[acc]), aph, abort_flag, args.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
      if (ACT == ACT_SWIGLU) {
        // lanes 0-15 and 16-31 hold the two matrices (gate, up) of features fl..fl+15; lane i < 16
        // finishes tokens 0-15 of a 32-token block, lane i + 16 tokens 16-31
        const int fl = t.n0 + (AR / 2) * crank + 16 * q;
        const int f = fl + (lane & 15);
        const bool upper = lane >= 16;
        const bool gate_lo = P.gate_first != 0;  // lanes 0-15 hold the gate accumulators
        // `mine` below belongs to this lane's matrix, `got` to the other one
        const bool mine_is_gate = upper != gate_lo;
        float sc = 1.f;  // 8-bit weights: the scale of this lane's weight row
        if (W8 && f < P.N)
          sc = __ldg((mine_is_gate ? P.scale0 : P.scale1) + (size_t)(t.g + f / P.N_w) * P.N_w + f % P.N_w);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out);
#pragma unroll 1
        for (int cb = grp; cb * 32 < t.ntok; cb += NGRP) {
          uint32_t v[32];
          tmem_ld32(tb + cb * 32, v);
          tmem_wait_ld();
          const int tok0 = t.m0 + cb * 32;
          const int nval = min(32, t.ntok - cb * 32);
          const int tbase = upper ? 16 : 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float lo_v = W8 ? __uint_as_float(v[i]) * sc : __uint_as_float(v[i]);
            const float hi_v = W8 ? __uint_as_float(v[16 + i]) * sc : __uint_as_float(v[16 + i]);
            // lane < 16 keeps token i and receives the partner's value of it; lane >= 16 keeps 16 + i
            const float got = __shfl_xor_sync(0xffffffffu, upper ? lo_v : hi_v, 16);
            const float mine = upper ? hi_v : lo_v;
            const float gate = mine_is_gate ? mine : got;
            const float up = mine_is_gate ? got : mine;
            if (f < P.N && tbase + i < nval)
              out[(size_t)(tok0 + tbase + i) * P.ldc + f] = __float2bfloat16_rn(silu(gate) * up);
          }
        }
      } else {
        const int fl = t.n0 + AR * crank + 32 * q;  // first feature of this warp
        const int f = fl + lane;
        float b = 0.f, sc = 1.f;  // bias; 8-bit weights: the scale of this thread's weight row
        if (P.bias && f < P.N) {
          const int gw = t.g + f / P.N_w;
          b = __bfloat162float(P.bias[(size_t)gw * P.N_w + f % P.N_w]);
        }
        if (W8 && f < P.N) sc = __ldg(P.scale0 + (size_t)(t.g + f / P.N_w) * P.N_w + f % P.N_w);
#pragma unroll 1
        for (int cb = grp; cb * 32 < t.ntok; cb += NGRP) {
          float h[32];
          {
            uint32_t v[32];
            tmem_ld32(tb + cb * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = W8 ? fmaf(__uint_as_float(v[i]), sc, b) : __uint_as_float(v[i]) + b;
          }
          if (ACT == ACT_GELU) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 g2 = gelu_erf2(make_float2(h[i], h[i + 1]));
              h[i] = g2.x;
              h[i + 1] = g2.y;
            }
          }
          const int tok0 = t.m0 + cb * 32;
          const int nval = min(32, t.ntok - cb * 32);
          if (nval == 32 && fl + 32 <= P.N) {
            uint8_t* stg = stg_w + (chunk++ % NBUF) * STG;
            if (lane == 0) bulk_wait_read<NBUF - 1>();  // the store that last used stg has read it
            __syncwarp();
            const uint32_t sb = smem_u32(stg);
            if (out_f32<ACT>()) {
              // 128-byte rows, 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                st_shared_f32(sb + i * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(i & 7)) << 4) + (lane & 3) * 4, h[i]);
            } else {
              // 64-byte rows, 64-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ ((r / 2) % 4)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                st_shared_u16(sb + i * 64 + ((((uint32_t)lane >> 3) ^ (uint32_t)((i >> 1) & 3)) << 4) + (lane & 7) * 2,
                              bf16_bits(h[i]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&maps.o[t.p], sb, fl, tok0);
              bulk_commit();
            }
          } else if (f < P.N) {
            if (out_f32<ACT>()) {
              float* out = static_cast<float*>(P.out);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nval) out[(size_t)(tok0 + i) * P.ldc + f] = h[i];
            } else {
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nval) out[(size_t)(tok0 + i) * P.ldc + f] = __float2bfloat16_rn(h[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_rank(smem_u32(&ctl->tempty[acc]), 0));  // the leader reuses the accumulator
    }
    if (lane == 0) bulk_wait_all();  // tile stores complete before the CTA leaves
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // no signal of the peer can still be in flight towards this CTA, and neither CTA's TMEM is in
  // use, when the pair frees its TMEM together
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_cg2(tmem_base, TMEM_COLS);
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
  if (rank < 1 || rank > 5) {
    snprintf(g_err, sizeof(g_err), "tensor map rank %d out of range", rank);
    return false;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    snprintf(g_err, sizeof(g_err), "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
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

bool make_tmap_f32(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box) {
  return make_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ptr, rank, dims, strides, box);
}

namespace {
// Largest number of co-resident 2-CTA clusters of a kernel (0 if none), per device.
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

template <int ACT, int NTV, bool W8>
cudaError_t launch_t(const Projection* ps, int nprob, uint32_t* status, cudaStream_t st) {
  constexpr int NT = tile_tokens<ACT, NTV>();
  constexpr int FT = feat_per_tile<ACT>();
  constexpr int threads = n_threads<ACT, NTV, W8>();
  constexpr size_t smem = smem_total<ACT, NTV, W8>();
  // weights: bf16 through the 128-byte swizzle, or 8-bit codes as plain 64-byte rows
  constexpr int wel = W8 ? 1 : 2;
  const CUtensorMapDataType wdt = W8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle wsw = !W8 ? CU_TENSOR_MAP_SWIZZLE_128B
                                     : (a_in_tmem<NTV, W8>() ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE);
  auto kern = k_proj_tc<ACT, NTV, W8>;
  TcMaps maps;
  memset(&maps, 0, sizeof(maps));
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.status = status;
  a.wfmt = W8 ? ps[0].wfmt : 0;
  long units_bound = 0;
  int np = 0;
  for (int i = 0; i < nprob; ++i) {
    const Projection& p = ps[i];
    const int rows_alloc = p.offsets ? p.rows_alloc : p.rows_static;
    if (rows_alloc <= 0 || p.N <= 0) continue;
    if (p.offsets && p.G > MAXGT - 1) return cudaErrorInvalidValue;
    {
      const cuuint64_t dims[2] = {(cuuint64_t)p.K, (cuuint64_t)rows_alloc};
      const cuuint64_t str[1] = {(cuuint64_t)p.lda * 2};
      const cuuint32_t box[2] = {BK, NT / 2}, box32[2] = {BK, 32};
      if (!make_tmap_bf16(&maps.x[np], p.A, 2, dims, str, box) || !make_tmap_bf16(&maps.x32[np], p.A, 2, dims, str, box32))
        return cudaErrorInvalidValue;
    }
    int gate_first = 1;
    if (ACT == ACT_SWIGLU) {
      // gate (B0) and up (B1) as one 5-D tensor (k, row in block of 16, matrix, block, expert): the
      // matrix dimension steps from the lower-addressed weight tensor to the other, so one box of
      // {64, 16, 2, 4, 1} brings 16 rows of one matrix, the same 16 rows of the other, 4 times over
      const char* g = static_cast<const char*>(p.B0);
      const char* u = static_cast<const char*>(p.B1);
      if (g == u || p.N_w % 16) {
        snprintf(g_err, sizeof(g_err), "SwiGLU gate and up weights must be distinct tensors");
        return cudaErrorInvalidValue;
      }
      gate_first = g < u ? 1 : 0;
      const cuuint64_t dims[5] = {(cuuint64_t)p.K_w, 16, 2, (cuuint64_t)(p.N_w / 16), (cuuint64_t)p.G_w};
      const cuuint64_t str[4] = {(cuuint64_t)p.K_w * wel, (cuuint64_t)(gate_first ? u - g : g - u),
                                 (cuuint64_t)p.K_w * wel * 16, (cuuint64_t)p.N_w * p.K_w * wel};
      const cuuint32_t box[5] = {BK, 16, 2, 4, 1};
      if (!make_tmap(&maps.w0[np], wdt, gate_first ? g : u, 5, dims, str, box, wsw)) return cudaErrorInvalidValue;
    } else {
      const cuuint64_t dims[3] = {(cuuint64_t)p.K_w, (cuuint64_t)p.N_w, (cuuint64_t)p.G_w};
      const cuuint64_t str[2] = {(cuuint64_t)p.K_w * wel, (cuuint64_t)p.N_w * p.K_w * wel};
      const cuuint32_t box[3] = {BK, AR, 1};
      if (!make_tmap(&maps.w0[np], wdt, p.B0, 3, dims, str, box, wsw)) return cudaErrorInvalidValue;
    }
    if (W8 && (p.wfmt != a.wfmt || !p.scale0 || (ACT == ACT_SWIGLU && !p.scale1))) {
      snprintf(g_err, sizeof(g_err), "8-bit weights need one format and row scales for every matrix");
      return cudaErrorInvalidValue;
    }
    {  // output blocks of the epilogue's TMA stores: 32 tokens x 32 features
      const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)rows_alloc};
      const cuuint64_t str[1] = {(cuuint64_t)p.ldc * (out_f32<ACT>() ? 4 : 2)};
      const cuuint32_t box[2] = {32, 32};
      if (!make_tmap(&maps.o[np], out_f32<ACT>() ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     p.out, 2, dims, str, box, out_f32<ACT>() ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    }
    ProbArgs& q = a.p[np];
    q.offsets = p.offsets;
    q.G = p.G;
    q.rows_static = p.rows_static;
    q.N = p.N;
    q.K = p.K;
    q.N_w = p.N_w;
    q.K_w = p.K_w;
    q.bias = static_cast<const __nv_bfloat16*>(p.bias);
    q.out = p.out;
    q.ldc = p.ldc;
    q.gate_first = gate_first;
    q.scale0 = W8 ? p.scale0 : nullptr;
    q.scale1 = W8 ? p.scale1 : nullptr;
    const long groups = p.offsets ? p.G : 1;
    // each group adds at most one partial token tile
    units_bound += ((rows_alloc + NT - 1) / NT + (p.offsets ? groups : 0)) * (long)((p.N + FT - 1) / FT);
    ++np;
  }
  if (np == 0) return cudaSuccess;
  a.nprob = np;
  const int n_clusters = max_pair_clusters(kern, threads, smem);
  if (n_clusters <= 0) {
    snprintf(g_err, sizeof(g_err), "no co-resident pair of CTAs for the grouped GEMM");
    return cudaErrorInvalidConfiguration;
  }
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  long clusters = units_bound < n_clusters ? units_bound : n_clusters;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, a);
  if (e != cudaSuccess) snprintf(g_err, sizeof(g_err), "grouped GEMM launch: %s", cudaGetErrorString(e));
  return e;
}

template <int ACT>
cudaError_t launch_a(const Projection* ps, int nprob, uint32_t* status, cudaStream_t st) {
  // every group at most 32 token rows (decode-sized calls): 32-token tiles, more stages in flight
  bool small = true;
  for (int i = 0; i < nprob; ++i) small = small && ps[i].max_group_rows <= 32;
  if (ps[0].wfmt != 0)
    return small ? launch_t<ACT, 32, true>(ps, nprob, status, st) : launch_t<ACT, 256, true>(ps, nprob, status, st);
  return small ? launch_t<ACT, 32, false>(ps, nprob, status, st) : launch_t<ACT, 256, false>(ps, nprob, status, st);
}
}  // namespace

const char* tc_last_error() { return g_err; }

cudaError_t launch_projection_tc(const Projection* ps, int nprob, uint32_t* status, cudaStream_t st) {
  if (nprob < 1 || nprob > MAXP) return cudaErrorInvalidValue;
  const int act = ps[0].act;
  for (int i = 1; i < nprob; ++i)
    if (ps[i].act != act || ps[i].out_f32 != ps[0].out_f32 || ps[i].wfmt != ps[0].wfmt) return cudaErrorInvalidValue;
  if (ps[0].wfmt < 0 || ps[0].wfmt > 2) return cudaErrorInvalidValue;
  // hidden layers are bf16 (the next projection's MMA operand); projections to the model width
  // keep the fp32 accumulator so the layer output is rounded once
  switch (act) {
    case ACT_GELU: return launch_a<ACT_GELU>(ps, nprob, status, st);
    case ACT_SWIGLU: return launch_a<ACT_SWIGLU>(ps, nprob, status, st);
    default:
      if (!ps[0].out_f32) return cudaErrorInvalidValue;
      return launch_a<ACT_NONE>(ps, nprob, status, st);
  }
}

}  // namespace moe
