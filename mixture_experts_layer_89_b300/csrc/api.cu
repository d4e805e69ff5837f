// C ABI of the MoE layer (declared in include/moe.h): argument validation, exact capacity,
// workspace layout and the stream-ordered launch sequence of each step.
#include <limits.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

struct WsLayout {
  size_t status, r_hist, r_psum, r_lse2, r_z, p_hist, p_base, drops, b_count, b_offs;
  size_t topk_idx, topk_w, counts, offsets, kept, row_of, tok_of;
  size_t x_perm, h, y_perm, h_sh, y_sh;
  size_t total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
inline size_t elt(const moe_config* c) { return c->dtype == MOE_BF16 ? 2 : 4; }
inline bool is_bf16(const moe_config* c) { return c->dtype == MOE_BF16; }
// 1 / router temperature (0 in the config means no temperature)
inline float inv_tau_of(const moe_config* c) { return c->router_temperature > 0.f ? 1.f / c->router_temperature : 1.f; }

// cap = ceil(cf T k / E) computed exactly from the binary value of the float32 cf; -1 = dropless.
int64_t capacity_exact(float cf, int64_t T, int64_t k, int64_t E) {
  if (!(cf > 0.f)) return -1;
  if (isinf(cf)) return T * k;
  int ex = 0;
  const float m = frexpf(cf, &ex);                         // cf = m 2^ex, m in [0.5, 1)
  const int64_t mi = (int64_t)ldexpf(m, 24);               // cf = mi 2^(ex - 24), exactly
  const int sh = ex - 24;
  __int128 num = (__int128)mi * T * k;
  __int128 den = E;
  if (sh >= 0) {
    if (sh > 40) return T * k;                             // cap >= T k: nothing can drop
    num <<= sh;
  } else {
    if (-sh > 90) return num > 0 ? 1 : 0;                  // 0 < cf T k / E < 1
    den <<= -sh;
  }
  __int128 c = (num + den - 1) / den;
  if (c > (__int128)T * k) c = (__int128)T * k;            // identical behaviour, keeps it in range
  return (int64_t)c;
}

int64_t a_max_of(const moe_config* c) {
  const int64_t tk = (int64_t)c->T * c->k;
  if (c->backup_expert) return tk;  // every assignment gets a row: kept ones, then the backup expert's
  const int64_t cap = capacity_exact(c->capacity_factor, c->T, c->k, c->E);
  if (cap < 0) return tk;
  const int64_t ec = cap * c->E;
  return ec < tk ? ec : tk;
}

moe_status validate(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d < 1 || c->E < 1 || c->k < 1 || c->dff < 1 || c->n_shared < 0) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_GELU_ERF && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (isnan(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
  if (!(c->router_temperature >= 0.f) || isinf(c->router_temperature)) return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->k > 8 || c->k > c->E || c->n_shared > 64) return MOE_ERR_UNSUPPORTED;
  if (c->has_bias && c->act != MOE_ACT_GELU_ERF) return MOE_ERR_UNSUPPORTED;
  if (c->backup_expert != 0 && c->backup_expert != 1) return MOE_ERR_INVALID_ARG;
  if (c->expert_weights < MOE_EXPERT_WEIGHTS_DTYPE || c->expert_weights > MOE_EXPERT_WEIGHTS_E4M3)
    return MOE_ERR_INVALID_ARG;
  if (c->expert_weights != MOE_EXPERT_WEIGHTS_DTYPE && !is_bf16(c)) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->k > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->n_shared * c->dff > INT_MAX / 2) return MOE_ERR_UNSUPPORTED;
  if (is_bf16(c)) {
    if (c->d % 64 || c->dff % 64) return MOE_ERR_UNSUPPORTED;
    if (c->n_shared > 1 && (c->dff % (c->act == MOE_ACT_SWIGLU ? 128 : 256))) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

WsLayout layout(const moe_config* c) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  const size_t T = (size_t)c->T, E = (size_t)c->E, k = (size_t)c->k, d = (size_t)c->d, f = (size_t)c->dff;
  const size_t S = (size_t)c->n_shared;
  const size_t nrb = (size_t)route_blocks(c->T), npb = (size_t)perm_blocks(c->T);
  const size_t A = (size_t)a_max_of(c);
  L.status = take(256);
  L.r_hist = take(nrb * E * 4);
  L.r_psum = take(nrb * E * 4);
  L.r_lse2 = take(nrb * 4);
  // per-token probabilities and lse^2 of the small-batch router (part of the router's scratch,
  // before the dispatch's buffers)
  L.r_z = take(is_bf16(c) && T <= (size_t)kSmallRouteTokens ? T * (E + 1) * 4 : 0);
  L.p_hist = take(npb * E * 4);
  L.p_base = take(npb * E * 4);
  L.drops = take(4);
  L.b_count = take(c->backup_expert ? npb * 4 : 0);
  L.b_offs = take(c->backup_expert ? 8 : 0);
  L.topk_idx = take(T * k * 4);
  L.topk_w = take(T * k * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.kept = take(E * 4);
  L.row_of = take(T * k * 4);
  L.tok_of = take(A * 4);
  L.x_perm = take(A * d * elt(c));
  L.h = take(A * f * elt(c));
  L.y_perm = take(A * d * 4);
  L.h_sh = take(T * S * f * elt(c));
  L.y_sh = take(S ? T * d * 4 : 0);
  L.total = off;
  return L;
}

// Scratch of the expert FFN backward: a status word; three [R, dff] fp32 buffers (pre-activations,
// then their gradients and h) for R = max(A_max, T when there are shared experts) rows, and the
// permuted rows' input gradients [A_max, d] fp32.  bf16 layers add the tensor-core operands: the
// padded column offsets, D [R, Kd] and h [R, dff] in bf16, and the transposed copies over Kp
// columns (every expert's rows padded to 64, or T padded to 64).
struct ExpertBwdScratch {
  size_t status, s0, s1, s2, dx_perm, koff, D, h, DT, hT, xT, dyT, total;
  int64_t Kp;
};

int64_t round64(int64_t v) { return (v + 63) & ~(int64_t)63; }

ExpertBwdScratch expert_bwd_scratch(const moe_config* c) {
  ExpertBwdScratch L;
  const size_t A = (size_t)a_max_of(c);
  const size_t R = std::max(A, c->n_shared > 0 ? (size_t)c->T : (size_t)0);
  const size_t f = (size_t)c->dff, d = (size_t)c->d, E = (size_t)c->E;
  const bool glu = c->act == MOE_ACT_SWIGLU, tc = is_bf16(c);
  const size_t Kd = glu ? 2 * f : f;
  L.Kp = std::max(A > 0 ? round64((int64_t)A + 63 * (int64_t)E) : (int64_t)0,
                  c->n_shared > 0 ? round64(c->T) : (int64_t)0);
  const size_t Kp = tc ? (size_t)L.Kp : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t a = off;
    off += align256(bytes);
    return a;
  };
  L.status = take(256);
  L.s0 = take(R * f * 4);
  L.s1 = take(glu ? R * f * 4 : 0);
  L.s2 = take(R * f * 4);
  L.dx_perm = take(A * d * 4);
  L.koff = take(tc ? (E + 1) * 4 : 0);
  L.D = take(tc ? R * Kd * 2 : 0);
  L.h = take(tc ? R * f * 2 : 0);
  L.DT = take(Kd * Kp * 2);
  L.hT = take(f * Kp * 2);
  L.xT = take(d * Kp * 2);
  L.dyT = take(d * Kp * 2);
  L.total = off;
  return L;
}

// Scratch of the router backward's tensor-core path: bf16 layers with E a multiple of 64 and T > 0;
// 0 bytes otherwise (the CUDA-core path needs none).
struct RouterBwdLayout {
  size_t status, dzs, dzsT, xT, part, koff, total;
};

RouterBwdLayout route_bwd_layout(const moe_config* c) {
  RouterBwdLayout L{};
  if (!is_bf16(c) || c->E % 64 || c->T <= 0) return L;
  const size_t Tp = (size_t)round64(c->T), E = (size_t)c->E, d = (size_t)c->d;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t a = off;
    off += align256(bytes);
    return a;
  };
  L.status = take(256);
  L.dzs = take((size_t)c->T * 2 * E * 2);
  L.dzsT = take(2 * E * Tp * 2);
  L.xT = take(d * Tp * 2);
  L.part = take((size_t)kRouterBwdSlices * 2 * E * d * 4);
  L.koff = take((kRouterBwdSlices + 1) * 4);
  L.total = off;
  return L;
}

template <typename P>
inline P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

inline bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// NVTX range around one C-ABI call (host side: it brackets the argument checks and the launches,
// which is what a profiler's timeline lines up with the kernels).  Costs nothing measurable when no
// tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

#define MOE_TRY(expr)                      \
  do {                                     \
    const moe_status _s = (expr);          \
    if (_s != MOE_OK) return _s;           \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// ------------------------------------------------------------------------------ steps
// scan != NULL: the tensor-core router may also do the dispatch scan (route_tc_fuses_scan).
moe_status route_impl(const moe_config* c, const void* x, const void* wr, const float* lbias, int32_t* topk_idx,
                      float* topk_w, int32_t* counts, float* losses, void* ws, cudaStream_t st,
                      const RouteScan* scan = nullptr, bool finalize = true) {
  const WsLayout L = layout(c);
  uint32_t* status = at<uint32_t>(ws, L.status);
  if (is_bf16(c) && c->T > 0 && c->T <= kSmallRouteTokens && !scan) {  // decode-sized batches
    float* ptok = at<float>(ws, L.r_z);
    return cuda_status(launch_route_small(x, wr, lbias, c->T, c->d, c->E, c->k, inv_tau_of(c), ptok,
                                          ptok + (size_t)c->T * c->E, status + 1, topk_idx, topk_w,
                                          at<int32_t>(ws, L.r_hist), at<float>(ws, L.r_psum), at<float>(ws, L.r_lse2),
                                          finalize, counts, losses, c->lb_coef, c->z_coef, status, st));
  }
  if (is_bf16(c)) {  // tensor-core router; the last CTA reduces the partials (counter: status block word 1)
    return cuda_status(launch_route_tc(x, wr, lbias, c->T, c->d, c->E, c->k, topk_idx, topk_w,
                                       at<int32_t>(ws, L.r_hist), at<float>(ws, L.r_psum), at<float>(ws, L.r_lse2),
                                       status + 1, counts, losses, c->lb_coef, c->z_coef, status, st, scan,
                                       finalize, inv_tau_of(c)));
  }
  MOE_CUDA(launch_route(false, x, wr, lbias, c->T, c->d, c->E, c->k, topk_idx, topk_w, at<int32_t>(ws, L.r_hist),
                        at<float>(ws, L.r_psum), at<float>(ws, L.r_lse2), status, st, inv_tau_of(c)));
  MOE_CUDA(launch_route_finalize(at<int32_t>(ws, L.r_hist), at<float>(ws, L.r_psum), at<float>(ws, L.r_lse2),
                                 route_blocks(c->T), c->T, c->E, c->k, c->lb_coef, c->z_coef, counts, losses, st));
  return MOE_OK;
}

// Backup expert: the assignments the capacity dropped take the rows after the kept ones, in token
// order (row range kept in the workspace for the projections).
moe_status backup_impl(const moe_config* c, const void* x, const int32_t* offsets, int32_t* row_of, int32_t* tok_of,
                       void* x_perm, void* ws, cudaStream_t st) {
  if (!c->backup_expert || c->T <= 0) return MOE_OK;
  const WsLayout L = layout(c);
  return cuda_status(launch_backup_dispatch(is_bf16(c), offsets + c->E, c->T, c->k, c->d, x, row_of, tok_of, x_perm,
                                            at<int32_t>(ws, L.b_count), at<int32_t>(ws, L.b_offs), st));
}

// scanned: the router already wrote the rank bases (p_base), kept, offsets and drops.
moe_status permute_impl(const moe_config* c, const void* x, const int32_t* topk_idx, const int32_t* counts,
                        int32_t* offsets, int32_t* kept, int32_t* row_of, int32_t* tok_of, void* x_perm,
                        int32_t* drops, void* ws, cudaStream_t st, bool scanned = false) {
  const WsLayout L = layout(c);
  uint32_t* status = at<uint32_t>(ws, L.status);
  const int64_t cap64 = capacity_exact(c->capacity_factor, c->T, c->k, c->E);
  const int cap = cap64 < 0 ? INT_MAX : (int)cap64;
  const int npb = perm_blocks(c->T);
  if (!scanned) {
    MOE_CUDA(launch_perm_hist(topk_idx, c->T, c->E, c->k, at<int32_t>(ws, L.p_hist), status, st));
    MOE_CUDA(launch_perm_scan(at<int32_t>(ws, L.p_hist), npb, counts, c->E, c->T * c->k, cap,
                              at<int32_t>(ws, L.p_base), offsets, kept, drops, status, st));
  }
  MOE_CUDA(launch_dispatch(is_bf16(c), topk_idx, at<int32_t>(ws, L.p_base), offsets, c->T, c->E, c->k, cap, x, c->d,
                           row_of, tok_of, x_perm, (int)a_max_of(c), status, st));
  return backup_impl(c, x, offsets, row_of, tok_of, x_perm, ws, st);
}

moe_status run_projection_simt(const Projection& p, cudaStream_t st) {
  return cuda_status(launch_projection_simt(false, p, st));
}

// The projections of the expert FFNs: routed experts over x_perm (groups from the device-side
// offsets) and the shared experts over x, concatenated into one expert whose hidden layer is S dff
// wide.  bf16 layers run both in one launch per projection (up, then down); fp32 layers run four
// CUDA-core launches.  ev_up / ev_down (timed variant only) are recorded after the up and the down
// projections of the routed experts.
moe_status ffn_impl(const moe_config* c, const void* x_perm, const int32_t* offsets, const moe_weights* w,
                    void* y_perm, const void* x, void* y_shared, void* ws, cudaStream_t st, cudaEvent_t ev_up,
                    cudaEvent_t ev_down) {
  const WsLayout L = layout(c);
  uint32_t* status = at<uint32_t>(ws, L.status);
  const int A = (int)a_max_of(c);
  const bool swiglu = c->act == MOE_ACT_SWIGLU;
  const int S = c->n_shared;
  const bool shared = S > 0 && c->T > 0;
  void* h = at<char>(ws, L.h);
  void* hs = at<char>(ws, L.h_sh);
  Projection up[3] = {}, dn[3] = {};
  int nup = 0;
  // a token picks an expert at most once, so no expert receives more than T rows (or C with a capacity)
  const int64_t cap64 = capacity_exact(c->capacity_factor, c->T, c->k, c->E);
  const int routed_rows = (int)(cap64 >= 0 && cap64 < c->T ? cap64 : c->T);
  if (A > 0) {
    Projection& p = up[nup++];
    p.A = x_perm; p.lda = c->d; p.rows_alloc = A;
    p.offsets = offsets; p.G = c->E; p.rows_static = 0;
    p.B0 = swiglu ? w->w_gate : w->w_up; p.B1 = w->w_up;
    p.bias = c->has_bias ? w->b_up : nullptr;
    p.N = c->dff; p.K = c->d; p.N_w = c->dff; p.K_w = c->d; p.G_w = c->E;
    p.act = swiglu ? ACT_SWIGLU : ACT_GELU;
    p.out = h; p.ldc = c->dff; p.max_group_rows = routed_rows;
    p.scale0 = swiglu ? w->s_gate : w->s_up; p.scale1 = w->s_up;
    Projection& q = dn[nup - 1];
    q.A = h; q.lda = c->dff; q.rows_alloc = A;
    q.offsets = offsets; q.G = c->E; q.rows_static = 0;
    q.B0 = w->w_down; q.B1 = nullptr; q.scale0 = w->s_down;
    q.bias = c->has_bias ? w->b_down : nullptr;
    q.N = c->d; q.K = c->dff; q.N_w = c->d; q.K_w = c->dff; q.G_w = c->E;
    q.act = ACT_NONE;
    q.out = y_perm; q.ldc = c->d; q.out_f32 = true; q.max_group_rows = routed_rows;
  }
  if (shared) {
    Projection& p = up[nup++];
    p.A = x; p.lda = c->d; p.rows_alloc = c->T;
    p.offsets = nullptr; p.G = 1; p.rows_static = c->T;
    p.B0 = swiglu ? w->ws_gate : w->ws_up; p.B1 = w->ws_up;
    p.bias = nullptr;
    p.N = S * c->dff; p.K = c->d; p.N_w = c->dff; p.K_w = c->d; p.G_w = S;
    p.act = swiglu ? ACT_SWIGLU : ACT_GELU;
    p.out = hs; p.ldc = (int64_t)S * c->dff; p.max_group_rows = c->T;
    p.scale0 = swiglu ? w->ss_gate : w->ss_up; p.scale1 = w->ss_up;
    Projection& q = dn[nup - 1];
    q.A = hs; q.lda = (int64_t)S * c->dff; q.rows_alloc = c->T;
    q.offsets = nullptr; q.G = 1; q.rows_static = c->T;
    q.B0 = w->ws_down; q.B1 = nullptr; q.bias = nullptr;
    q.scale0 = w->ss_down;  // one scale per row of the S down matrices side by side
    q.N = c->d; q.K = S * c->dff; q.N_w = c->d; q.K_w = c->dff; q.G_w = S;
    q.act = ACT_NONE;
    q.out = y_shared; q.ldc = c->d; q.out_f32 = true; q.max_group_rows = c->T;
  }
  int nbk = -1;  // index of the backup expert's problem
  if (c->backup_expert && A > 0) {
    nbk = nup;
    const int32_t* boffs = at<int32_t>(ws, L.b_offs);  // {first backup row, end}, written by the dispatch
    Projection& p = up[nup++];
    p.A = x_perm; p.lda = c->d; p.rows_alloc = A;
    p.offsets = boffs; p.G = 1; p.rows_static = 0;
    p.B0 = swiglu ? w->wb_gate : w->wb_up; p.B1 = w->wb_up;
    p.bias = c->has_bias ? w->bb_up : nullptr;
    p.N = c->dff; p.K = c->d; p.N_w = c->dff; p.K_w = c->d; p.G_w = 1;
    p.act = swiglu ? ACT_SWIGLU : ACT_GELU;
    p.out = h; p.ldc = c->dff; p.max_group_rows = A;
    p.scale0 = swiglu ? w->sb_gate : w->sb_up; p.scale1 = w->sb_up;
    Projection& q = dn[nup - 1];
    q.A = h; q.lda = c->dff; q.rows_alloc = A;
    q.offsets = boffs; q.G = 1; q.rows_static = 0;
    q.B0 = w->wb_down; q.B1 = nullptr; q.scale0 = w->sb_down;
    q.bias = c->has_bias ? w->bb_down : nullptr;
    q.N = c->d; q.K = c->dff; q.N_w = c->d; q.K_w = c->dff; q.G_w = 1;
    q.act = ACT_NONE;
    q.out = y_perm; q.ldc = c->d; q.out_f32 = true; q.max_group_rows = A;
  }
  for (int i = 0; i < nup; ++i) up[i].wfmt = dn[i].wfmt = c->expert_weights;
  if (is_bf16(c)) {
    if (nup) MOE_CUDA(launch_projection_tc(up, nup, status, st));
    if (ev_up) MOE_CUDA(cudaEventRecord(ev_up, st));
    if (nup) MOE_CUDA(launch_projection_tc(dn, nup, status, st));
    if (ev_down) MOE_CUDA(cudaEventRecord(ev_down, st));
    return MOE_OK;
  }
  const int nrouted = A > 0 ? 1 : 0;
  if (nrouted) MOE_TRY(run_projection_simt(up[0], st));
  if (ev_up) MOE_CUDA(cudaEventRecord(ev_up, st));
  if (nrouted) MOE_TRY(run_projection_simt(dn[0], st));
  if (ev_down) MOE_CUDA(cudaEventRecord(ev_down, st));
  if (shared) {
    MOE_TRY(run_projection_simt(up[nrouted], st));
    MOE_TRY(run_projection_simt(dn[nrouted], st));
  }
  if (nbk >= 0) {
    MOE_TRY(run_projection_simt(up[nbk], st));
    MOE_TRY(run_projection_simt(dn[nbk], st));
  }
  return MOE_OK;
}

moe_status check_weights(const moe_config* c, const moe_weights* w) {
  if (!w || !w->w_router || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  if (c->act == MOE_ACT_SWIGLU && !w->w_gate) return MOE_ERR_INVALID_ARG;
  if (c->has_bias && (!w->b_up || !w->b_down)) return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && (!w->ws_up || !w->ws_down || (c->act == MOE_ACT_SWIGLU && !w->ws_gate)))
    return MOE_ERR_INVALID_ARG;
  if (c->backup_expert && (!w->wb_up || !w->wb_down || (c->act == MOE_ACT_SWIGLU && !w->wb_gate) ||
                           (c->has_bias && (!w->bb_up || !w->bb_down))))
    return MOE_ERR_INVALID_ARG;
  if (is_bf16(c) && c->act == MOE_ACT_SWIGLU && c->backup_expert && w->wb_gate == w->wb_up) return MOE_ERR_UNSUPPORTED;
  // bf16 SwiGLU experts read their gate and up rows through one tensor map spanning both tensors
  if (is_bf16(c) && c->act == MOE_ACT_SWIGLU && (w->w_gate == w->w_up || (c->n_shared > 0 && w->ws_gate == w->ws_up)))
    return MOE_ERR_UNSUPPORTED;
  if (c->expert_weights != MOE_EXPERT_WEIGHTS_DTYPE) {  // row scales of every 8-bit matrix
    const bool sw = c->act == MOE_ACT_SWIGLU;
    if (!w->s_up || !w->s_down || (sw && !w->s_gate)) return MOE_ERR_INVALID_ARG;
    if (c->n_shared > 0 && (!w->ss_up || !w->ss_down || (sw && !w->ss_gate))) return MOE_ERR_INVALID_ARG;
    if (c->backup_expert && (!w->sb_up || !w->sb_down || (sw && !w->sb_gate))) return MOE_ERR_INVALID_ARG;
  }
  const void* ps[] = {w->w_router, w->w_up, w->w_gate, w->w_down, w->b_up, w->b_down, w->ws_up, w->ws_gate, w->ws_down,
                      w->wb_up, w->wb_gate, w->wb_down, w->bb_up, w->bb_down};
  for (const void* p : ps)
    if (p && misaligned(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status layer_impl(const moe_config* c, const moe_weights* w, const void* x, void* y, float* losses,
                      int32_t* counts_out, int32_t* drops_out, void* ws, cudaStream_t st, cudaEvent_t const* ev) {
  MOE_TRY(validate(c));
  MOE_TRY(check_weights(c, w));
  if (!ws || !losses || (c->T > 0 && (!x || !y))) return MOE_ERR_INVALID_ARG;
  if (misaligned(ws) || misaligned(x) || misaligned(y)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(c);
  int32_t* topk_idx = at<int32_t>(ws, L.topk_idx);
  float* topk_w = at<float>(ws, L.topk_w);
  int32_t* counts = counts_out ? counts_out : at<int32_t>(ws, L.counts);
  int32_t* drops = drops_out ? drops_out : at<int32_t>(ws, L.drops);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* row_of = at<int32_t>(ws, L.row_of);
  void* x_perm = at<char>(ws, L.x_perm);
  void* y_perm = at<char>(ws, L.y_perm);
  void* y_sh = c->n_shared > 0 ? at<char>(ws, L.y_sh) : nullptr;
  auto rec = [&](int i) -> moe_status { return ev ? cuda_status(cudaEventRecord(ev[i], st)) : MOE_OK; };

  // bf16 layers: the router's last CTA also does the dispatch scan over its per-block histograms
  const int64_t cap64 = capacity_exact(c->capacity_factor, c->T, c->k, c->E);
  RouteScan scan;
  scan.cap = cap64 < 0 ? INT_MAX : (int)cap64;
  scan.pbase = at<int32_t>(ws, L.p_base);
  scan.kept = at<int32_t>(ws, L.kept);
  scan.offsets = offsets;
  scan.drops = drops;
  // bf16 layers: the dispatch kernel finalises the router (counts, losses, scan) when the per-block
  // histograms fit its shared memory; else the router's last CTA does, scan included when it fits
  const bool dfused = is_bf16(c) && dispatch_fuses_scan(c->T, c->E);
  const bool scanned = !dfused && is_bf16(c) && route_tc_fuses_scan(c->T, c->E);
  MOE_TRY(rec(0));
  MOE_TRY(route_impl(c, x, w->w_router, w->router_logit_bias, topk_idx, topk_w, counts, losses, ws, st,
                     dfused ? nullptr : &scan, !dfused));
  MOE_TRY(rec(1));
  if (dfused) {
    MOE_CUDA(launch_dispatch_fused(true, topk_idx, at<int32_t>(ws, L.r_hist), at<float>(ws, L.r_psum),
                                   at<float>(ws, L.r_lse2), c->T, c->E, c->k, scan.cap, c->lb_coef, c->z_coef, x, c->d,
                                   counts, losses, offsets, at<int32_t>(ws, L.kept), drops, row_of,
                                   at<int32_t>(ws, L.tok_of), x_perm, (int)a_max_of(c), at<uint32_t>(ws, L.status),
                                   st));
    MOE_TRY(backup_impl(c, x, offsets, row_of, at<int32_t>(ws, L.tok_of), x_perm, ws, st));
  } else {
    MOE_TRY(permute_impl(c, x, topk_idx, counts, offsets, at<int32_t>(ws, L.kept), row_of, at<int32_t>(ws, L.tok_of),
                         x_perm, drops, ws, st, scanned));
  }
  MOE_TRY(rec(2));
  // routed and shared experts (bf16: one launch per projection carries both)
  MOE_TRY(ffn_impl(c, x_perm, offsets, w, y_perm, x, y_sh, ws, st, ev ? ev[3] : nullptr, ev ? ev[4] : nullptr));
  MOE_TRY(rec(5));
  MOE_CUDA(launch_combine(is_bf16(c), static_cast<const float*>(y_perm), row_of, topk_w,
                          static_cast<const float*>(y_sh), y, c->T, c->d, c->k, st));
  MOE_TRY(rec(6));
  return MOE_OK;
}

}  // namespace


// ------------------------------------------------------------------ router without a workspace
// Scratch of moe_route_noalloc: a file-scope device array.  Host code must not hand the array's
// name to a kernel (in host code it names a host-side shadow, not device memory); its device
// address is looked up once per device with cudaGetSymbolAddress and cached.
static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_route_scratch_mu;
void* g_route_scratch_ptr[kMaxDevices] = {nullptr};
CUcontext g_route_scratch_ctx[kMaxDevices] = {nullptr};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's cuCtxGetCurrent, looked up once.
CtxGetCurrentFn ctx_get_current_fn() {
  static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<CtxGetCurrentFn>(p);
    return nullptr;
  }();
  return fn;
}

// Device address of g_route_scratch on the current device.  Looked up with cudaGetSymbolAddress
// the first time a device is used, and again whenever that device's current context is no longer
// the one the address was taken in (after a cudaDeviceReset the module is loaded afresh and the
// array may move).
moe_status route_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  CUcontext ctx = nullptr;
  const CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_route_scratch_mu);
  if (!g_route_scratch_ptr[dev] || g_route_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_route_scratch_ptr[dev] = p;
    g_route_scratch_ctx[dev] = ctx;
  }
  *out = g_route_scratch_ptr[dev];
  return MOE_OK;
}
}  // namespace

// ================================================================================ C ABI
extern "C" {

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = layout(cfg).total;
  return MOE_OK;
}

moe_status moe_capacity(const moe_config* cfg, int32_t* cap, int32_t* a_max) {
  MOE_TRY(validate(cfg));
  if (cap) {
    const int64_t c = capacity_exact(cfg->capacity_factor, cfg->T, cfg->k, cfg->E);
    *cap = c < 0 ? -1 : (int32_t)c;
  }
  if (a_max) *a_max = (int32_t)a_max_of(cfg);
  return MOE_OK;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router, const float* logit_bias,
                     int32_t* topk_idx, float* topk_w, int32_t* counts, float* losses, void* ws, void* stream) {
  NvtxRange nvtx_range("moe_route");
  MOE_TRY(validate(cfg));
  if (!w_router || !counts || !losses || !ws) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!x || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (misaligned(ws) || misaligned(x) || misaligned(w_router)) return MOE_ERR_INVALID_ARG;
  return route_impl(cfg, x, w_router, logit_bias, topk_idx, topk_w, counts, losses, ws,
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_route_noalloc(const moe_config* cfg, const void* x, const void* w_router, const float* logit_bias,
                             int32_t* topk_idx, float* topk_w, int32_t* counts, float* losses, void* stream) {
  NvtxRange nvtx_range("moe_route_noalloc");
  MOE_TRY(validate(cfg));
  if (!w_router || !counts || !losses) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!x || !topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (misaligned(x) || misaligned(w_router)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > MOE_ROUTE_NOALLOC_MAX_T || (int64_t)cfg->T * cfg->E > MOE_ROUTE_NOALLOC_MAX_TE)
    return MOE_ERR_UNSUPPORTED;
  // the router's scratch is the front of the workspace layout, up to the dispatch's first buffer
  if (layout(cfg).p_hist > (size_t)MOE_ROUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  MOE_TRY(route_scratch_address(&scratch));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // status word, CTA counter and wait-limit override (default) start at zero
  MOE_CUDA(cudaMemsetAsync(scratch, 0, 4 * sizeof(uint32_t), st));
  return route_impl(cfg, x, w_router, logit_bias, topk_idx, topk_w, counts, losses, scratch, st);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* kept, int32_t* row_of, int32_t* tok_of, void* x_perm, void* ws,
                       void* stream) {
  NvtxRange nvtx_range("moe_permute");
  MOE_TRY(validate(cfg));
  if (!offsets || !kept || !ws) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!x || !topk_idx || !row_of || !tok_of || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (misaligned(ws) || misaligned(x) || misaligned(x_perm)) return MOE_ERR_INVALID_ARG;
  return permute_impl(cfg, x, topk_idx, counts, offsets, kept, row_of, tok_of, x_perm, nullptr, ws,
                      static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets, const moe_weights* w,
                          void* y_perm, const void* x, void* y_shared, void* ws, void* stream) {
  NvtxRange nvtx_range("moe_expert_ffn");
  MOE_TRY(validate(cfg));
  MOE_TRY(check_weights(cfg, w));
  if (!offsets || !ws) return MOE_ERR_INVALID_ARG;
  if (a_max_of(cfg) > 0 && (!x_perm || !y_perm)) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared > 0 && cfg->T > 0 && (!x || !y_shared)) return MOE_ERR_INVALID_ARG;
  if (misaligned(ws) || misaligned(x_perm) || misaligned(y_perm) || misaligned(x) || misaligned(y_shared))
    return MOE_ERR_INVALID_ARG;
  return ffn_impl(cfg, x_perm, offsets, w, y_perm, x, y_shared, ws, static_cast<cudaStream_t>(stream), nullptr,
                  nullptr);
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_of, const float* topk_w,
                       const void* y_shared, void* y, void* stream) {
  NvtxRange nvtx_range("moe_combine");
  MOE_TRY(validate(cfg));
  if (cfg->T > 0 && (!row_of || !topk_w || !y || (!y_perm && a_max_of(cfg) > 0))) return MOE_ERR_INVALID_ARG;
  if (misaligned(y_perm) || misaligned(y_shared) || misaligned(y)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(is_bf16(cfg), static_cast<const float*>(y_perm), row_of, topk_w,
                                    static_cast<const float*>(y_shared), y, cfg->T, cfg->d, cfg->k,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_stats(const moe_config* cfg, const int32_t* topk_idx, const int32_t* offsets, int32_t* coact,
                           float* stats, void* ws, void* stream) {
  NvtxRange nvtx_range("moe_route_stats");
  MOE_TRY(validate(cfg));
  if (!coact || !stats || !ws || (cfg->T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
  if (cfg->k > 8) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = layout(cfg);
  return cuda_status(launch_route_stats(topk_idx, offsets, cfg->T, cfg->E, cfg->k, coact, stats,
                                        at<uint32_t>(ws, L.status), static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_diagnostics(const moe_config* cfg, const void* x, const void* w_router, const float* logit_bias,
                                 float* diag, float* entropy_tok, void* ws, void* stream) {
  NvtxRange nvtx_range("moe_route_diagnostics");
  MOE_TRY(validate(cfg));
  if (!w_router || !diag || !ws || (cfg->T > 0 && !x)) return MOE_ERR_INVALID_ARG;
  if (misaligned(ws) || misaligned(x) || misaligned(w_router)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg);
  static_assert(kRouteTokens == 32, "the diagnostics reuse the router's 32-token block scratch");
  if (route_diag_blocks(cfg->T) > route_blocks(cfg->T)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_route_diag(is_bf16(cfg), x, w_router, logit_bias, cfg->T, cfg->d, cfg->E, cfg->k,
                                       inv_tau_of(cfg), cfg->lb_coef, diag, entropy_tok, at<float>(ws, L.r_psum),
                                       at<int32_t>(ws, L.r_hist), at<float>(ws, L.r_lse2), at<uint32_t>(ws, L.status),
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x, void* y, float* losses,
                             int32_t* counts_out, int32_t* drops_out, void* ws, void* stream) {
  NvtxRange nvtx_range("moe_layer_forward");
  return layer_impl(cfg, w, x, y, losses, counts_out, drops_out, ws, static_cast<cudaStream_t>(stream), nullptr);
}

moe_status moe_layer_forward_timed(const moe_config* cfg, const moe_weights* w, const void* x, void* y,
                                   float* losses, int32_t* counts_out, int32_t* drops_out, void* ws, void* stream,
                                   void* const* events, int32_t n_events) {
  NvtxRange nvtx_range("moe_layer_forward_timed");
  if (!events || n_events != 7) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[7];
  for (int i = 0; i < 7; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
    ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  return layer_impl(cfg, w, x, y, losses, counts_out, drops_out, ws, static_cast<cudaStream_t>(stream), ev);
}

moe_status moe_read_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v == 0) return MOE_OK;
  if (cudaMemset(ws, 0, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v & DEV_TIMEOUT) return MOE_ERR_TIMEOUT;
  return MOE_ERR_DEVICE_STATUS;
}

moe_status moe_set_wait_limit(void* ws, uint64_t limit_ns, void* stream) {
  if (!ws || misaligned(ws)) return MOE_ERR_INVALID_ARG;
  const uint32_t w[2] = {(uint32_t)limit_ns, (uint32_t)(limit_ns >> 32)};
  // from pageable host memory: the source is staged before the call returns
  return cuda_status(cudaMemcpyAsync(static_cast<uint32_t*>(ws) + 2, w, sizeof(w), cudaMemcpyHostToDevice,
                                     static_cast<cudaStream_t>(stream)));
}

int32_t moe_layer_forward_launches(const moe_config* cfg) {
  if (validate(cfg) != MOE_OK) return -1;
  int n = 0;
  const bool tokens = cfg->T > 0;
  if (is_bf16(cfg)) n += tokens ? 1 : 0;      // tensor-core or small-batch router (finalize fused; T = 0: memsets)
  else n += tokens ? 2 : 1;                   // router + finalize
  const bool dfused = is_bf16(cfg) && dispatch_fuses_scan(cfg->T, cfg->E);
  const bool scanned = dfused || (is_bf16(cfg) && route_tc_fuses_scan(cfg->T, cfg->E));
  if (!tokens) n += 1;                        // scan (writes zero offsets)
  else n += (scanned ? 0 : 2) + dispatch_launches(true, cfg->d, is_bf16(cfg) ? 2 : 4);  // [hist, scan,] dispatch
  if (tokens && cfg->backup_expert) n += 2;   // backup rows: count, place
  const bool routed = a_max_of(cfg) > 0, shared = cfg->n_shared > 0 && tokens;
  if (is_bf16(cfg)) n += (routed || shared) ? 2 : 0;           // up + down, routed and shared together
  else n += (routed ? 2 : 0) + (shared ? 2 : 0) + (routed && cfg->backup_expert ? 2 : 0);  // routed, shared, backup
  if (tokens) n += 1;                         // combine
  return n;
}

moe_status moe_quantize_experts(const void* w, int32_t dtype, int32_t format, int32_t blocks, int32_t rows,
                                int32_t cols, void* codes, float* scale, int32_t* nonfinite, void* stream) {
  NvtxRange nvtx_range("moe_quantize_experts");
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (format != MOE_EXPERT_WEIGHTS_INT8 && format != MOE_EXPERT_WEIGHTS_E4M3) return MOE_ERR_UNSUPPORTED;
  if (blocks < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)blocks * rows * cols >= (int64_t)1 << 40 || cols > (1 << 20)) return MOE_ERR_INVALID_ARG;
  if ((int64_t)blocks * rows * cols == 0) return MOE_OK;
  if (!w || !codes || !scale) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scale) & 3u) || (reinterpret_cast<uintptr_t>(nonfinite) & 3u) ||
      (reinterpret_cast<uintptr_t>(w) & (dtype == MOE_BF16 ? 1u : 3u)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize(dtype == MOE_BF16, format, w, blocks, rows, cols, static_cast<uint8_t*>(codes),
                                     scale, nonfinite, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_backward(const moe_config* cfg, const void* dy, const float* y_perm, const int32_t* row_of,
                                const float* topk_w, float* dw, void* dy_perm, void* stream) {
  NvtxRange nvtx_range("moe_combine_backward");
  MOE_TRY(validate(cfg));
  if (cfg->T > 0 && (!dy || !row_of || !topk_w || !dw || (a_max_of(cfg) > 0 && (!y_perm || !dy_perm))))
    return MOE_ERR_INVALID_ARG;
  if (misaligned(dy) || misaligned(y_perm) || misaligned(row_of) || misaligned(topk_w) || misaligned(dw) ||
      misaligned(dy_perm))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_backward(is_bf16(cfg), dy, y_perm, row_of, topk_w, cfg->T, cfg->d, cfg->k, dw,
                                             dy_perm, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_backward_scratch_size(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = route_bwd_layout(cfg).total;
  return MOE_OK;
}

moe_status moe_route_backward(const moe_config* cfg, const void* x, const void* w_router, const float* logit_bias,
                              const int32_t* topk_idx, const float* topk_w, const int32_t* counts, const float* dw,
                              float dlb, float dzl, float* dz, float* dw_router, float* dx, void* scratch,
                              void* stream) {
  NvtxRange nvtx_range("moe_route_backward");
  MOE_TRY(validate(cfg));
  if (!w_router || !counts || !dw_router) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!x || !topk_idx || !topk_w || !dw || !dz || !dx)) return MOE_ERR_INVALID_ARG;
  if (!isfinite(dlb) || !isfinite(dzl)) return MOE_ERR_INVALID_ARG;
  const void* ps[] = {x, w_router, logit_bias, topk_idx, topk_w, counts, dw, dz, dw_router, dx, scratch};
  for (const void* p : ps)
    if (misaligned(p)) return MOE_ERR_INVALID_ARG;
  const RouterBwdLayout L = route_bwd_layout(cfg);
  RouterBwdScratch sc{};
  const bool tc = scratch && L.total > 0;
  if (tc) {
    sc.status = at<uint32_t>(scratch, L.status);
    sc.dzs = at<__nv_bfloat16>(scratch, L.dzs);
    sc.dzsT = at<__nv_bfloat16>(scratch, L.dzsT);
    sc.xT = at<__nv_bfloat16>(scratch, L.xT);
    sc.part = at<float>(scratch, L.part);
    sc.koff = at<int32_t>(scratch, L.koff);
  }
  return cuda_status(launch_router_backward(is_bf16(cfg), x, w_router, logit_bias, topk_idx, topk_w, counts, dw,
                                            cfg->T, cfg->d, cfg->E, cfg->k, inv_tau_of(cfg), cfg->lb_coef,
                                            cfg->z_coef, dlb, dzl, dz, dw_router, dx, tc ? &sc : nullptr,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_backward_scratch_size(const moe_config* cfg, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (cfg->backup_expert || cfg->expert_weights != MOE_EXPERT_WEIGHTS_DTYPE) return MOE_ERR_UNSUPPORTED;
  *bytes = expert_bwd_scratch(cfg).total;
  return MOE_OK;
}

moe_status moe_expert_ffn_backward(const moe_config* cfg, const moe_weights* w, const void* x, const void* x_perm,
                                   const int32_t* offsets, const int32_t* row_of, const void* dy,
                                   const void* dy_perm, const moe_expert_grads* g, float* dx, void* scratch,
                                   void* stream) {
  NvtxRange nvtx_range("moe_expert_ffn_backward");
  MOE_TRY(validate(cfg));
  if (cfg->backup_expert || cfg->expert_weights != MOE_EXPERT_WEIGHTS_DTYPE) return MOE_ERR_UNSUPPORTED;
  if (!w || !g) return MOE_ERR_INVALID_ARG;
  const bool glu = cfg->act == MOE_ACT_SWIGLU, routed = a_max_of(cfg) > 0, S = cfg->n_shared > 0;
  if (!w->w_up || !w->w_down || !g->dw_up || !g->dw_down || (glu && (!w->w_gate || !g->dw_gate)))
    return MOE_ERR_INVALID_ARG;
  if (cfg->has_bias && (!w->b_up || !g->db_up || !g->db_down)) return MOE_ERR_INVALID_ARG;
  if (S && (!w->ws_up || !w->ws_down || !g->dws_up || !g->dws_down || (glu && (!w->ws_gate || !g->dws_gate))))
    return MOE_ERR_INVALID_ARG;
  if (routed && (!x_perm || !offsets || !row_of || !dy_perm || !dx || !scratch)) return MOE_ERR_INVALID_ARG;
  if (S && cfg->T > 0 && (!x || !dy || !dx || !scratch)) return MOE_ERR_INVALID_ARG;
  if (!scratch) return MOE_ERR_INVALID_ARG;  // the status word lives there
  const void* ps[] = {x, x_perm, offsets, row_of, dy, dy_perm, dx, scratch, w->w_up, w->w_gate, w->w_down,
                      w->b_up, w->ws_up, w->ws_gate, w->ws_down, g->dw_up, g->dw_gate, g->dw_down, g->db_up,
                      g->db_down, g->dws_up, g->dws_gate, g->dws_down};
  for (const void* p : ps)
    if (misaligned(p)) return MOE_ERR_INVALID_ARG;
  const ExpertBwdScratch L = expert_bwd_scratch(cfg);
  const int64_t cap = capacity_exact(cfg->capacity_factor, cfg->T, cfg->k, cfg->E);
  ExpertBackward b{};
  b.T = cfg->T, b.d = cfg->d, b.E = cfg->E, b.k = cfg->k, b.dff = cfg->dff, b.n_shared = cfg->n_shared;
  b.act = glu ? ACT_SWIGLU : ACT_GELU;
  b.rows_bound = routed ? (int)(cap >= 0 && cap < cfg->T ? cap : cfg->T) : 0;
  b.rows_alloc = (int)a_max_of(cfg);
  b.Kp = L.Kp;
  b.x = x, b.x_perm = x_perm, b.dy = dy, b.dy_perm = dy_perm, b.offsets = offsets, b.row_of = row_of;
  b.w_up = w->w_up, b.w_gate = glu ? w->w_gate : nullptr, b.w_down = w->w_down;
  b.b_up = cfg->has_bias ? w->b_up : nullptr;
  b.ws_up = w->ws_up, b.ws_gate = glu ? w->ws_gate : nullptr, b.ws_down = w->ws_down;
  b.dw_up = g->dw_up, b.dw_gate = glu ? g->dw_gate : nullptr, b.dw_down = g->dw_down;
  b.db_up = cfg->has_bias ? g->db_up : nullptr, b.db_down = cfg->has_bias ? g->db_down : nullptr;
  b.dws_up = g->dws_up, b.dws_gate = glu ? g->dws_gate : nullptr, b.dws_down = g->dws_down;
  b.dx = dx;
  b.dx_perm = at<float>(scratch, L.dx_perm);
  b.s0 = at<float>(scratch, L.s0), b.s1 = at<float>(scratch, L.s1), b.s2 = at<float>(scratch, L.s2);
  b.status = at<uint32_t>(scratch, L.status);
  b.koff = at<int32_t>(scratch, L.koff);
  using bf = __nv_bfloat16;
  b.D = at<bf>(scratch, L.D);
  b.h = at<bf>(scratch, L.h), b.DT = at<bf>(scratch, L.DT), b.hT = at<bf>(scratch, L.hT);
  b.xT = at<bf>(scratch, L.xT), b.dyT = at<bf>(scratch, L.dyT);
  return cuda_status(launch_expert_backward(is_bf16(cfg), b, static_cast<cudaStream_t>(stream)));
}

moe_status moe_workspace_views(const moe_config* cfg, void* ws, moe_forward_views* v) {
  MOE_TRY(validate(cfg));
  if (!ws || !v || misaligned(ws)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout(cfg);
  v->topk_idx = at<int32_t>(ws, L.topk_idx);
  v->topk_w = at<float>(ws, L.topk_w);
  v->counts = at<int32_t>(ws, L.counts);
  v->offsets = at<int32_t>(ws, L.offsets);
  v->row_of = at<int32_t>(ws, L.row_of);
  v->tok_of = at<int32_t>(ws, L.tok_of);
  v->x_perm = at<char>(ws, L.x_perm);
  v->y_perm = at<float>(ws, L.y_perm);
  return MOE_OK;
}

const char* moe_last_error(void) { return tc_last_error(); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_STATUS: return "device reported bad data";
  }
  return "unknown status";
}

}  // extern "C"
