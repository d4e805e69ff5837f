// Host-side launchers of the MoE kernels (internal to the library; the public ABI is moe.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- router (route.cu)
constexpr int kRouteTokens = 32;  // tokens per router CTA
int route_blocks(int T);
// x [T,d] and w_router [E,d] of type `bf16` (else fp32).  Writes top-k, per-CTA histograms,
// per-CTA softmax column sums and per-CTA sums of lse^2.
// inv_tau: 1 / router temperature (the softmax, the weights and lse use z / tau; the top-k uses z)
cudaError_t launch_route(bool bf16, const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                         int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2,
                         uint32_t* status, cudaStream_t st, float inv_tau = 1.f);
// Tensor-core router of bf16 layers (one launch, 128 tokens per CTA): writes top-k, and through
// the last CTA to finish, counts [E] and losses [2].  hist/psum/lse2 hold route_tc_blocks(T) rows
// of partials; *done must be zero before the launch and is zero again after it.
// With `scan`, and when route_tc_fuses_scan(T, E), the last CTA also does the dispatch scan over
// the router's per-block histograms (blocks of kPermTokens tokens).
struct RouteScan {
  int cap;          // expert capacity (INT_MAX when dropless)
  int32_t* pbase;   // [nb][E] exclusive prefix of each expert's histogram over blocks
  int32_t* kept;    // [E]
  int32_t* offsets; // [E+1]
  int32_t* drops;   // [1]
};
int route_tc_blocks(int T);
bool route_tc_fuses_scan(int T, int E);
cudaError_t launch_route_tc(const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                            int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum, float* lse2, uint32_t* done,
                            int32_t* counts, float* losses, float lb_coef, float z_coef, uint32_t* status,
                            cudaStream_t st, const RouteScan* scan, bool finalize = true, float inv_tau = 1.f);
// Router of bf16 layers for T <= kSmallRouteTokens (route_small.cu): one CTA per token
// (compensated fp32 logits, top-k, weights, softmax), per-token probabilities ptok [T][E] and
// lse^2 l2tok [T] in the workspace; the last CTA (counter *done, zero between calls) writes the
// router's partials of one block (hist, psum [E], lse2 [1]) and, with finalize, counts and losses.
constexpr int kSmallRouteTokens = 64;
cudaError_t launch_route_small(const void* x, const void* wr, const float* lbias, int T, int d, int E, int k,
                               float inv_tau, float* ptok, float* l2tok, uint32_t* done, int32_t* topk_idx,
                               float* topk_w, int32_t* hist, float* psum, float* lse2, bool finalize, int32_t* counts,
                               float* losses, float lb_coef, float z_coef, uint32_t* status, cudaStream_t st);
// Reduces the per-CTA partials: counts [E] and losses [2].
cudaError_t launch_route_finalize(const int32_t* hist, const float* psum, const float* lse2, int nb, int T, int E,
                                  int k, float lb_coef, float z_coef, int32_t* counts, float* losses,
                                  cudaStream_t st);

// ---------------------------------------------------------------- dispatch (permute.cu)
constexpr int kPermTokens = 128;  // tokens per dispatch block (= the tensor-core router's block)
int perm_blocks(int T);
cudaError_t launch_perm_hist(const int32_t* topk_idx, int T, int E, int k, int32_t* phist, uint32_t* status,
                             cudaStream_t st);
cudaError_t launch_perm_scan(const int32_t* phist, int npb, const int32_t* counts, int E, int Tk, int cap,
                             int32_t* pbase, int32_t* offsets, int32_t* kept, int32_t* drops, uint32_t* status,
                             cudaStream_t st);
// Ranks and row_of / tok_of (one CTA per block), then (x_perm != NULL) the row copy x -> x_perm.
cudaError_t launch_dispatch(bool bf16, const int32_t* topk_idx, const int32_t* pbase, const int32_t* offsets, int T,
                            int E, int k, int cap, const void* x, int d, int32_t* row_of, int32_t* tok_of,
                            void* x_perm, int max_rows, uint32_t* status, cudaStream_t st);
// Dispatch that also finalises the router (bf16 layers): the router ran with finalize = false and
// left its per-block partials (hist, psum [nb][E], lse2 [nb]); every dispatch CTA stages the
// histograms, derives its rank bases, the kept counts and the offsets, and CTA 0 also writes
// offsets, kept, drops, counts and both losses.  Usable when dispatch_fuses_scan(T, E).
bool dispatch_fuses_scan(int T, int E);
cudaError_t launch_dispatch_fused(bool bf16, const int32_t* topk_idx, const int32_t* hist, const float* psum,
                                  const float* lse2, int T, int E, int k, int cap, float lb_coef, float z_coef,
                                  const void* x, int d, int32_t* counts, float* losses, int32_t* offsets,
                                  int32_t* kept, int32_t* drops, int32_t* row_of, int32_t* tok_of, void* x_perm,
                                  int max_rows, uint32_t* status, cudaStream_t st);

// Routing statistics: co-activation counts coact [E][E] (zeroed here), stats [2] (load imbalance,
// dropped fraction; offsets may be NULL).
cudaError_t launch_route_stats(const int32_t* topk_idx, const int32_t* offsets, int T, int E, int k, int32_t* coact,
                               float* stats, uint32_t* status, cudaStream_t st);

// Routing diagnostics (route_diag.cu): diag [4] = {mean router entropy, lb_coef E sum Pbar^2,
// lb_coef (KL(uniform || Pbar + 1e-8) + sum (f - 1/E)^2), lb_coef E sum f Pbar}; ent_tok [T] or NULL.
// psum/cnt [route_diag_blocks(T)][E] and hsum [route_diag_blocks(T)] are scratch.
int route_diag_blocks(int T);
cudaError_t launch_route_diag(bool bf16, const void* x, const void* wr, const float* lbias, int T, int d, int E,
                              int k, float inv_tau, float lb_coef, float* diag, float* ent_tok, float* psum,
                              int32_t* cnt, float* hsum, uint32_t* status, cudaStream_t st);

// Backup expert: after a dispatch with capacity drops, the dropped assignments take rows
// kept_rows[0] .. (in token order) of row_of / tok_of / x_perm; backup_offs [2] = that row range.
// bcount [perm_blocks(T)] is scratch.  Two launches.
cudaError_t launch_backup_dispatch(bool bf16, const int32_t* kept_rows, int T, int k, int d, const void* x,
                                   int32_t* row_of, int32_t* tok_of, void* x_perm, int32_t* bcount,
                                   int32_t* backup_offs, cudaStream_t st);

// Kernels launch_dispatch launches (2 with the row copy, else 1).
int dispatch_launches(bool with_rows, int d, int elt_bytes);

// ---------------------------------------------------------------- combine (combine.cu)
// y_perm [rows, d] and y_shared [T, d] are fp32; y is bf16 or fp32.
cudaError_t launch_combine(bool bf16, const float* y_perm, const int32_t* row_of, const float* topk_w,
                           const float* y_shared, void* y, int T, int d, int k, cudaStream_t st);

// ---------------------------------------------------------------- grouped FFN GEMMs
// One grouped projection  out[r, n] = act(sum_k A[r, k] B_{g(r)}[n, k] (+ bias)).
// Rows of A are split into G groups by offsets (device, [G+1]); offsets == NULL means one group of
// rows [0, rows_static).  Weights are viewed as [G_w][N_w][K_w]; the weight matrix used for output
// column n and reduction index kk of group g is g + n / N_w + kk / K_w, at (n % N_w, kk % K_w), so
// routed experts (N_w = N, K_w = K) and concatenated shared experts (spanning N or K) share code.
enum Act { ACT_NONE = 0, ACT_GELU = 1, ACT_SWIGLU = 2 };
struct Projection {
  const void* A; int64_t lda; int rows_alloc;      // A [rows_alloc, K] (lda elements)
  const int32_t* offsets; int G; int rows_static;
  const void* B0; const void* B1;                  // B1: the W_up half of SwiGLU
  const void* bias;                                // [G_w][N_w] or NULL
  int N, K, N_w, K_w, G_w;
  int act;
  void* out; int64_t ldc;
  bool out_f32;                                    // out is fp32 (else the layer dtype)
  int max_group_rows;                              // bound on the rows of any one group (host-known)
  int wfmt;                                        // weights: 0 layer dtype, 1 int8, 2 E4M3 codes
  const float* scale0; const float* scale1;        // 8-bit weights: fp32 row scales of B0, B1
};
// Backward of the routing half: dw [T,k] and dy_perm (rows of kept slots) from dy and y_perm; the
// router's dz [T,E], dW_r [E,d] and dx [T,d] from dw (see backward.cu).
cudaError_t launch_combine_backward(bool bf16, const void* dy, const float* y_perm, const int32_t* row_of,
                                    const float* topk_w, int T, int d, int k, float* dw, void* dy_perm,
                                    cudaStream_t st);
// Scratch of the router backward's tensor-core path (bf16 layers, E a multiple of 64): status
// word, dzs [T][2E] and dzsT [2E][Tp] bf16, xT [d][Tp] bf16, part [kRouterBwdSlices][2E][d] fp32
// and koff [kRouterBwdSlices + 1] (Tp = T padded to 64).
constexpr int kRouterBwdSlices = 8;
struct RouterBwdScratch {
  uint32_t* status;
  __nv_bfloat16 *dzs, *dzsT, *xT;
  float* part;
  int32_t* koff;
};
// sc == NULL (or an fp32 layer): the CUDA-core path.
cudaError_t launch_router_backward(bool bf16, const void* x, const void* wr, const float* lbias, const int32_t* idx,
                                   const float* tw, const int32_t* counts, const float* dw, int T, int d, int E, int k,
                                   float inv_tau, float lb_coef, float z_coef, float dlb, float dzl, float* dz,
                                   float* dwr, float* dx, const RouterBwdScratch* sc, cudaStream_t st);
// Backward of the expert FFNs (routed over the permuted rows, then the shared experts over all
// tokens).  Weights and activations in the layer dtype, gradients fp32; act is ACT_GELU or
// ACT_SWIGLU; rows_bound bounds any expert's rows (0: no routed rows), rows_alloc = A_max; s0..s2
// hold max(A_max, T) x dff floats each (s1 SwiGLU only), dx_perm A_max x d.  bf16 layers (tensor
// cores) also use: status (one word, zeroed by the call), koff [E+1], D [max(A_max, T)][Kd]
// (Kd = 2 dff for SwiGLU, else dff) and h [..][dff] bf16, and the transposed copies DT [Kd][Kp],
// hT [dff][Kp], xT and dyT [d][Kp] (Kp a multiple of 64 at least the rows padded per expert and T
// padded).
struct ExpertBackward {
  int T, d, E, k, dff, n_shared, act, rows_bound, rows_alloc;
  int64_t Kp;
  const void *x, *x_perm, *dy, *dy_perm;
  const int32_t *offsets, *row_of;
  const void *w_up, *w_gate, *w_down, *b_up, *ws_up, *ws_gate, *ws_down;
  float *dw_up, *dw_gate, *dw_down, *db_up, *db_down, *dws_up, *dws_gate, *dws_down;
  float *dx, *dx_perm, *s0, *s1, *s2;
  uint32_t* status;
  int32_t* koff;
  __nv_bfloat16 *D, *h, *DT, *hT, *xT, *dyT;
};
// Grouped bf16 tensor-core GEMM of the backward, C (+)= A B^T with fp32 output (gemm_bwd.cu):
// rows on M (A [rows_alloc][K], B [G_w][N][K], group rows from off or [0, rows)) and rows on K
// (A [M][Kp], B [N][Kp], group columns from off -- multiples of 64 -- or [0, cols)).
cudaError_t launch_gemm_bwd_rows_m(const void* A, int rows_alloc, const void* B, int G_w, int N, int K,
                                   const int32_t* off, int G, int rows, float* C, int64_t ldc, int beta,
                                   uint32_t* status, cudaStream_t st);
// Rows on M with B read N-major from the weights as stored: B_g(n, k) = B[g][k][n] for k < ksplit,
// B2[g][k - ksplit][n] beyond (B2 unused when ksplit == K).
cudaError_t launch_gemm_bwd_rows_m_nmajor(const void* A, int rows_alloc, const void* B, const void* B2, int ksplit,
                                          int G_w, int N, int K, const int32_t* off, int G, int rows, float* C,
                                          int64_t ldc, int beta, uint32_t* status, cudaStream_t st, bool nmajor);
cudaError_t launch_gemm_bwd_rows_k(const void* A, int M, const void* B, int N, int Kp, const int32_t* off, int G,
                                   int cols, float* C, int64_t ldc, int64_t c_stride, int beta, uint32_t* status,
                                   cudaStream_t st);
cudaError_t launch_expert_backward(bool bf16, const ExpertBackward& b, cudaStream_t st);
// Per-row scaled 8-bit codes of w [blocks][rows][cols] (fmt 1 int8, 2 E4M3), one CTA per row.
cudaError_t launch_quantize(bool bf16, int fmt, const void* w, int blocks, int rows, int cols, uint8_t* codes,
                            float* scale, int32_t* nonfinite, cudaStream_t st);
cudaError_t launch_projection_simt(bool bf16, const Projection& p, cudaStream_t st);
// bf16 layers: nprob (1 or 2) projections with the same activation in one launch of the paired
// tensor-core kernel (the routed and the shared experts share its persistent CTAs).
cudaError_t launch_projection_tc(const Projection* ps, int nprob, uint32_t* status, cudaStream_t st);
const char* tc_last_error();

// Raise a kernel's dynamic shared-memory limit to `bytes` (once per kernel and device).
cudaError_t ensure_smem_attr(const void* kernel, size_t bytes);

// bf16 tensor map with the 128-byte swizzle (tiles of 64 bf16 along the innermost dimension);
// out-of-range elements of a box read as zero.  False (message in tc_last_error) on failure.
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                    const cuuint32_t* box);
// The same for fp32 tensors (32 floats per 128-byte swizzle row).
bool make_tmap_f32(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box);

}  // namespace moe
