/*
 * moe.h -- C ABI of the B300 (sm_103a) sparse Mixture-of-Experts FFN layer: the forward pass and
 * the backward pass (routing half and expert FFNs).
 *
 * The layer (mini-moe tutorial, sec. 3.1 MoELayer; OpenMythos article, sec. 3.1; FLAME-MoE
 * summary, sec. 2) maps T tokens x[T,d] to y[T,d]:
 *   z = x W_r^T (+ fixed logit bias)        P = softmax(z / tau) S_t = top-k of z_t
 *   w_tj = P_t[e_j] / sum_{e in S_t} P_t[e]
 *   per-expert capacity C = ceil(cf T k / E) (cf <= 0: dropless), assignments ranked in token
 *   order, rank >= C dropped (weight 0)
 *   y_t = sum_{kept j} w_tj FFN_{e_j}(x_t) + sum_s FFN^shared_s(x_t)
 *   lb = lb_coef E sum_e f_e Pbar_e  (f_e = counts_e/(T k), Pbar_e = mean_t P_te)
 *   zl = z_coef mean_t logsumexp(z_t / tau)^2        (tau: router temperature, 1 by default)
 * The residual add x + y is not part of the layer.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers allocated and owned by the caller; the library
 *    allocates no memory and keeps no per-call state.  Tensors are dense row-major.
 *  - Weights use the nn.Linear layout [out, in], stacked on a leading expert axis.
 *  - Activations and weights share the dtype of moe_config.dtype (fp32 or bf16); router logits,
 *    softmax and routing weights are fp32; indices and counts are int32.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream); calls return
 *    without synchronising.  The return value reports argument validation and launch errors.
 *    Errors detected on the device (non-finite logits, inconsistent counts, a bounded wait
 *    that gave up) are recorded in a status word inside the workspace; read it with
 *    moe_read_device_status.
 *  - `ws` is a device workspace of at least moe_workspace_size bytes, 256-byte aligned, owned
 *    by the caller and zero-filled before its first use (its first word is the device status
 *    word); the same workspace must not be used by two calls that may run concurrently.
 *  - Every tensor pointer must be 16-byte aligned (MOE_ERR_INVALID_ARG otherwise).
 *  - A_max = T*k (dropless) or min(T*k, E*C): the row capacity of the expert-sorted buffers.
 *  - Shape limits: 1 <= k <= min(E, 8), 1 <= E <= 256, T >= 0, d >= 1, dff >= 1.  bf16 layers
 *    also need d % 64 == 0 and dff % 64 == 0 (tensor-core tiles), and with n_shared > 1 also
 *    dff % 128 == 0 (SwiGLU) or dff % 256 == 0 (GELU); bf16 SwiGLU layers need distinct gate and
 *    up weight tensors (w_gate != w_up, ws_gate != ws_up).  Violations return MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* NULL pointer, negative size, misaligned pointer          */
  MOE_ERR_UNSUPPORTED = -2,   /* shape outside the limits above                           */
  MOE_ERR_CUDA = -3,          /* a CUDA runtime/driver call failed                        */
  MOE_ERR_TIMEOUT = -4,       /* device: a bounded wait inside a kernel gave up           */
  MOE_ERR_DEVICE_STATUS = -5  /* device: non-finite logits or inconsistent inputs         */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_ACT_GELU_ERF = 0,  /* W_down gelu(W_up x + b_up) + b_down   (mini-moe tutorial, sec. 3.1) */
  MOE_ACT_SWIGLU = 1     /* W_down (silu(W_gate x) * W_up x)      (GPT-4 2% article, sec. 3.1)  */
} moe_act;

/* Storage of the expert FFN weights (routed, shared and backup experts; the router keeps the
 * layer dtype).  The mini-moe tutorial (deployment optimisation) suggests quantising every expert
 * to INT8 to cut what is stored and loaded; the 8-bit formats hold one code per weight and one
 * fp32 scale per output row (see moe_quantize_experts), need a bf16 layer, and multiply the codes
 * by the bf16 activations on the tensor cores (codes widened exactly to bf16 on the SM, into shared
 * or tensor memory) with the scale applied to the fp32 accumulator. */
typedef enum {
  MOE_EXPERT_WEIGHTS_DTYPE = 0,  /* the layer dtype                                              */
  MOE_EXPERT_WEIGHTS_INT8 = 1,   /* int8 codes q, weight = q * scale_row, |q| <= 127              */
  MOE_EXPERT_WEIGHTS_E4M3 = 2    /* OCP FP8 E4M3 codes, weight = value(code) * scale_row          */
} moe_expert_weights;

typedef struct {
  int32_t T;               /* tokens                                                        */
  int32_t d;               /* model width                                                   */
  int32_t E;               /* routed experts                                                */
  int32_t k;               /* experts per token                                             */
  int32_t dff;             /* expert hidden width                                           */
  int32_t n_shared;        /* always-on shared experts (same act, no biases)                */
  int32_t act;             /* moe_act                                                       */
  int32_t dtype;           /* moe_dtype of activations and weights                          */
  int32_t has_bias;        /* routed GELU experts carry b_up [E,dff] and b_down [E,d]       */
  float capacity_factor;   /* <= 0: dropless                                                */
  float lb_coef;           /* load-balance loss coefficient (alpha)                         */
  float z_coef;            /* router z-loss coefficient (beta)                              */
  float router_temperature;/* tau > 0 divides the logits before the softmax, the renormalised
                              weights and both losses (the top-k choice is that of the raw
                              logits); 0 means none (tau = 1).  Negative: MOE_ERR_INVALID_ARG */
  int32_t backup_expert;   /* 1: assignments over the capacity go, with their routing weight, to
                              one extra expert (weights wb_* / bb_*) instead of being dropped
                              (mini-moe tutorial, sec. 6); A_max becomes T*k.  0: dropped      */
  int32_t expert_weights;  /* moe_expert_weights; 8-bit formats need dtype == MOE_BF16, else
                              MOE_ERR_UNSUPPORTED                                              */
} moe_config;

typedef struct {
  const void* w_router;           /* [E,d]                                                  */
  const float* router_logit_bias; /* [E] fp32 added to the logits, or NULL                   */
  const void* w_up;               /* [E,dff,d]                                              */
  const void* w_gate;             /* [E,dff,d] (SwiGLU) or NULL                              */
  const void* w_down;             /* [E,d,dff]                                              */
  const void* b_up;               /* [E,dff] or NULL (has_bias)                              */
  const void* b_down;             /* [E,d]   or NULL (has_bias)                              */
  const void* ws_up;              /* shared [S,dff,d] or NULL when n_shared == 0             */
  const void* ws_gate;            /* shared [S,dff,d] (SwiGLU) or NULL                       */
  const void* ws_down;            /* shared [S,d,dff] or NULL                                */
  const void* wb_up;              /* backup expert [dff,d] (backup_expert) or NULL           */
  const void* wb_gate;            /* backup expert [dff,d] (SwiGLU) or NULL                  */
  const void* wb_down;            /* backup expert [d,dff] or NULL                           */
  const void* bb_up;              /* backup expert bias [dff] (has_bias) or NULL             */
  const void* bb_down;            /* backup expert bias [d] (has_bias) or NULL               */
  /* 8-bit expert weights only (else ignored): the tensors above hold codes (same shapes, one
   * byte each; biases stay bf16) and these hold the fp32 scale of every output row.          */
  const float* s_up;              /* [E,dff]                                                */
  const float* s_gate;            /* [E,dff] (SwiGLU)                                       */
  const float* s_down;            /* [E,d]                                                  */
  const float* ss_up;             /* [S,dff]                                                */
  const float* ss_gate;           /* [S,dff] (SwiGLU)                                       */
  const float* ss_down;           /* [d]: one scale per row of the [d, S*dff] matrix that the
                                     shared experts' down projections form side by side    */
  const float* sb_up;             /* [dff] backup expert                                    */
  const float* sb_gate;           /* [dff] backup expert (SwiGLU)                           */
  const float* sb_down;           /* [d]   backup expert                                    */
} moe_weights;

/* Workspace bytes needed by every call below for this config (host only, no GPU work).
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for a bad config. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Expert capacity C (-1 when dropless) and A_max for this config, exactly as the kernels use
 * them: C = ceil(cf * T * k / E) evaluated exactly on the float32 value of cf. Host only. */
moe_status moe_capacity(const moe_config* cfg, int32_t* cap, int32_t* a_max);

/* Router (mini-moe tutorial, sec. 3.1; OpenMythos article, sec. 3.1; losses: OpenMythos
 * article sec. 3.1 and FLAME-MoE summary sec. 2).
 *   x [T,d], w_router [E,d], logit_bias [E] fp32 or NULL
 *   -> topk_idx [T,k] int32 (descending logit, ties to the lower expert index),
 *      topk_w [T,k] fp32 (renormalised over the k), counts [E] int32 (pre-drop assignments),
 *      losses [2] fp32 = {load-balance loss, router z-loss}.
 * Logits are accumulated in fp32: bf16 layers on the tensor cores (one launch; the reduction of
 * the per-CTA partials into counts and losses is done by the last CTA to finish), fp32 layers on
 * CUDA cores.  A bf16 token whose leading k+1 logits lie closer together than a bound on the
 * tensor cores' accumulation error (about 2^-22 (d/16) max(1, |z|)) is re-decided from logits
 * recomputed with compensated fp32 sums, so the selection and its order do not depend on the
 * tensor cores' accumulation order. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* w_router,
                     const float* logit_bias, int32_t* topk_idx, float* topk_w,
                     int32_t* counts, float* losses, void* ws, void* stream);

/* Dispatch (Naive-N0.5-Flash article sec. 4.2: group tokens by target expert; OpenMythos
 * article sec. 3.1: flatten + index reorder, capacity and overflow).
 *   x [T,d], topk_idx [T,k], counts [E] (as produced by moe_route)
 *   -> offsets [E+1] (expert e owns rows offsets[e]..offsets[e+1]-1 of the sorted layout),
 *      kept [E] = min(counts, C), row_of [T,k] (sorted row of slot j of token t, -1 if dropped),
 *      tok_of [A_max] (token of each sorted row), x_perm [A_max,d] = x[tok_of[r]].
 * Rows of an expert are in increasing token order; rows >= offsets[E] are left untouched -- except
 * with a backup expert, where the assignments over capacity take rows offsets[E] .. offsets[E] +
 * drops - 1 in (token, slot) order (their row_of entries are then >= 0, and the row range is kept
 * in ws for moe_expert_ffn).
 * A counts vector that disagrees with topk_idx sets MOE_ERR_DEVICE_STATUS in the status word. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                       const int32_t* counts, int32_t* offsets, int32_t* kept,
                       int32_t* row_of, int32_t* tok_of, void* x_perm, void* ws, void* stream);

/* Expert FFNs (mini-moe tutorial sec. 3.1; GPT-4 2% article sec. 3.1; shared experts:
 * FLAME-MoE summary sec. 2).
 *   x_perm [A_max,d] with offsets [E+1] from moe_permute -> y_perm [A_max,d] fp32 (rows < offsets[E]);
 *   when n_shared > 0 also x [T,d] -> y_shared [T,d] fp32 = sum_s FFN^shared_s(x) (else both NULL).
 * y_perm and y_shared keep the fp32 accumulators so that the layer output is rounded only once.
 * Hidden activations are kept in the workspace; bf16 layers round them to bf16 (they are the
 * operand of the down-projection's bf16 tensor-core MMA). */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const moe_weights* w, void* y_perm, const void* x, void* y_shared,
                          void* ws, void* stream);

/* Combine (FLAME-MoE summary sec. 2: output = routing-weighted sum of the selected experts).
 *   y[t] = sum_{j: row_of[t,j] >= 0} topk_w[t,j] * y_perm[row_of[t,j]]  (+ y_shared[t])
 * y_perm [A_max,d] and y_shared [T,d] are fp32 (as moe_expert_ffn writes them); y [T,d] has the
 * layer dtype.  Accumulated in fp32 in slot order, shared output last, rounded once.
 * y_shared may be NULL. */
moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_of,
                       const float* topk_w, const void* y_shared, void* y, void* stream);

/* The whole layer: route -> permute -> expert FFNs -> combine, no host sync.
 *   x [T,d] -> y [T,d]; losses [2]; counts_out [E] (nullable); drops_out [1] (nullable,
 *   number of dropped assignments).  Intermediates live in ws.
 * Ordering: everything is ordered after the work already queued on `stream`, and the work queued
 * on `stream` afterwards is ordered after the whole layer.  Every kernel runs on `stream` (the
 * shared and backup experts ride in the routed experts' GEMM launches); the kernels use
 * programmatic dependent launch, so a kernel's set-up may overlap the previous kernel on `stream`
 * (each waits for it before touching memory), which CUDA graph capture of `stream` keeps.
 * Calls that share a workspace must not overlap on the GPU. */
moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                             void* y, float* losses, int32_t* counts_out, int32_t* drops_out,
                             void* ws, void* stream);

/* Same as moe_layer_forward, and records caller-created CUDA events (cudaEvent_t, cast to
 * void*) on `stream` at the stage boundaries, for timing:
 *   events[0] before routing, [1] after routing, [2] after dispatch, [3] after the routed
 *   up-projection, [4] after the routed down-projection, [5] after the shared experts,
 *   [6] after the combine.  n_events must be 7. */
moe_status moe_layer_forward_timed(const moe_config* cfg, const moe_weights* w, const void* x,
                                   void* y, float* losses, int32_t* counts_out,
                                   int32_t* drops_out, void* ws, void* stream,
                                   void* const* events, int32_t n_events);

/* Synchronises `stream`, returns the device status word of `ws` as a moe_status (MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_STATUS) and clears it. */
moe_status moe_read_device_status(void* ws, void* stream);

/* Failure-detection test hook: sets, for every later call that uses the workspace `ws`, how long
 * a bounded wait inside the tensor-core router (moe_route and the routing step of
 * moe_layer_forward) may last before it gives up, in nanoseconds (counted on the SM's cycle
 * counter at a nominal 2 cycles per nanosecond); 0 restores the default of one second.  A wait that gives up stops the CTA's pipeline, lets its copies and tensor-core work in
 * flight finish, records MOE_ERR_TIMEOUT in the status word and returns (the results of that call
 * are then meaningless).  The grouped expert GEMMs always keep the one-second limit.  Ordered on
 * `stream` like the other calls.  MOE_ERR_INVALID_ARG for a NULL or misaligned ws. */
moe_status moe_set_wait_limit(void* ws, uint64_t limit_ns, void* stream);

/* Number of kernels moe_layer_forward launches for this config (for launch accounting). */
int32_t moe_layer_forward_launches(const moe_config* cfg);

/* Router without a caller-supplied workspace (no counterpart in the pages: an addition of this
 * library for callers that cannot allocate device memory, such as an engine that reserves all of
 * HBM for weights and caches at start-up and forbids later cudaMalloc calls (they synchronise the
 * device and fragment its memory), or a plug-in running inside another framework's operator with
 * no handle on that framework's allocator).
 *   Same arguments, results and error codes as moe_route, without `ws`.  Its scratch (the status
 *   word and the per-CTA partial sums of the router) lives in a fixed device array of
 *   MOE_ROUTE_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 *   holds until the process exits.  This call allocates nothing.
 *   Limits: T <= MOE_ROUTE_NOALLOC_MAX_T and T * E <= MOE_ROUTE_NOALLOC_MAX_TE, else
 *   MOE_ERR_UNSUPPORTED (before any GPU work).
 *   The first call on a device looks up that array's device address (once per device and CUDA
 *   context, with that device current; again after a cudaDeviceReset replaced the context); make
 *   that first call outside any CUDA stream capture.
 *   All calls share the one array and it keeps the previous call's contents: each call clears the
 *   status word itself, but two calls whose GPU work may overlap (different streams, or different
 *   host threads, without ordering between them) race on the array and must not be issued.
 *   Device-side error flags (non-finite logits) are cleared at the start of every call and are
 *   not reported back; use moe_route with a workspace when they are needed. */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (2u << 20)
#define MOE_ROUTE_NOALLOC_MAX_T (1 << 20)
#define MOE_ROUTE_NOALLOC_MAX_TE (1 << 22)
moe_status moe_route_noalloc(const moe_config* cfg, const void* x, const void* w_router,
                             const float* logit_bias, int32_t* topk_idx, float* topk_w,
                             int32_t* counts, float* losses, void* stream);

/* Routing statistics (beyond the layer itself): how the router spread the tokens over the
 * experts.  Expert co-activation is discussed in the FLAME-MoE summary; load imbalance and
 * capacity overflow in the Naive-N0.5-Flash article, sec. 4.
 *   topk_idx [T,k] int32 from moe_route; offsets [E+1] from moe_permute, or NULL.
 *   coact [E,E] int32, overwritten: coact[i][j] (i != j) = number of tokens whose k experts
 *     include both i and j; coact[i][i] = number of tokens that chose i (moe_route's counts).
 *     P(E_j | E_i) = coact[i][j] / coact[i][i].
 *   stats [2] float, overwritten: [0] max_e coact[e][e] / (T k / E), the load of the busiest
 *     expert relative to a uniform spread (1 = uniform); [1] dropped assignments / (T k) from
 *     offsets[E] (0 when offsets is NULL).
 *   ws: a workspace of this config (only its status word is used: an index outside [0, E) sets
 *     MOE_ERR_DEVICE_STATUS and that token is skipped).  Deterministic (integer counts). */
moe_status moe_route_stats(const moe_config* cfg, const int32_t* topk_idx, const int32_t* offsets,
                           int32_t* coact, float* stats, void* ws, void* stream);

/* Routing diagnostics (beyond the layer itself): the router entropy that the Naive-N0.5-Flash
 * article (sec. 4, monitoring) and the GPT-4 2% article (routing-collapse tips) watch, and the two
 * other balance-loss forms the pages give, beside the layer's own (OpenMythos article, sec. 3.1).
 *   x [T,d], w_router [E,d], logit_bias [E] or NULL, with cfg's router temperature tau
 *   -> diag [4] fp32, overwritten:
 *      [0] mean over tokens of -sum_e P_te ln P_te (nats; P = softmax(z / tau))
 *      [1] lb_coef E sum_e Pbar_e^2                             (mini-moe tutorial, sec. 3.1)
 *      [2] lb_coef (sum_e (1/E)(ln(1/E) - ln(Pbar_e + 1e-8)) + sum_e (f_e - 1/E)^2)
 *                                                               (GPT-4 2% article, sec. 4.2)
 *      [3] lb_coef E sum_e f_e Pbar_e, the layer's load-balance loss
 *      with Pbar_e = mean_t P_te and f_e = counts_e / (T k) from the top-k of the raw logits;
 *   entropy_tok [T] fp32 or NULL: each token's entropy.
 * The logits are recomputed in fp32 on CUDA cores in a fixed order; the per-block partials are
 * reduced in block order (deterministic).  ws: a workspace of this config; the call overwrites
 * the router's scratch in it (not the status word, where non-finite logits are reported). */
moe_status moe_route_diagnostics(const moe_config* cfg, const void* x, const void* w_router,
                                 const float* logit_bias, float* diag, float* entropy_tok, void* ws,
                                 void* stream);

/* 8-bit expert weights (mini-moe tutorial, deployment optimisation: quantise each expert).
 *   w [blocks, rows, cols] of dtype (moe_dtype) -> codes [blocks, rows, cols] (one byte each),
 *   scale [rows] fp32, where logical row r is row r of every block placed side by side:
 *     scale_r = max |w[:, r, :]| / qmax  (an IEEE fp32 division; 1 for an all-zero row),
 *     codes   = the code nearest to w / scale_r (an IEEE fp32 division), ties to even;
 *   format MOE_EXPERT_WEIGHTS_INT8: qmax 127, int8 codes in [-127, 127];
 *   format MOE_EXPERT_WEIGHTS_E4M3: qmax 448, E4M3 codes (saturating at +-448).
 *   For per-row scales of an expert stack [E, rows, cols] pass blocks = 1, rows = E * rows; for
 *   the shared experts' down projections [S, d, dff] (one wide matrix) pass blocks = S, rows = d.
 *   nonfinite: NULL, or a device int32 the call adds the number of non-finite weights to (their
 *   codes are meaningless).  Deterministic; blocks * rows * cols < 2^40, cols <= 2^20.
 *   MOE_ERR_INVALID_ARG for bad sizes or pointers, MOE_ERR_UNSUPPORTED for another format. */
moe_status moe_quantize_experts(const void* w, int32_t dtype, int32_t format, int32_t blocks,
                                int32_t rows, int32_t cols, void* codes, float* scale,
                                int32_t* nonfinite, void* stream);

/* Backward pass of the layer, in three calls: moe_combine_backward, moe_route_backward and
 * moe_expert_ffn_backward (below).  The objective is L = sum_t <dy_t, y_t> + dlb lb + dzl zl (the
 * pages train with the load-balance loss and the router z-loss added: mini-moe tutorial, training
 * loop; FLAME-MoE summary, sec. 2).  Top-k selection, capacity drops and the expert counts pass no
 * gradient.  All sums in a fixed order (bit-identical repeats).
 *
 * moe_combine_backward (FLAME-MoE summary sec. 2: y = routing-weighted sum of the experts):
 *   dy [T,d] (layer dtype), y_perm [A_max,d] fp32, row_of [T,k], topk_w [T,k] as the forward
 *   steps left them -> dw [T,k] fp32 = <dy_t, y_perm[row_of[t,j]]> (0 for a dropped slot) and
 *   dy_perm [A_max,d] (layer dtype): row row_of[t,j] = topk_w[t,j] dy_t, the upstream gradient of
 *   the expert FFN of that row (rows of no kept slot are left untouched).
 *
 * moe_route_backward (the router of moe_route, with cfg's temperature, lb_coef and z_coef):
 *   x [T,d], w_router [E,d], logit_bias [E] or NULL, topk_idx / topk_w [T,k] and counts [E] as
 *   moe_route returned them, dw [T,k] from moe_combine_backward, dlb / dzl the weights of the two
 *   losses in the objective
 *   -> dz [T,E] fp32, the gradient of the logits (z recomputed with fp32 accumulation);
 *      dw_router [E,d] fp32 = dz^T x; dx [T,d] fp32 = dz W_r, the router's part of the input
 *      gradient (overwritten).
 *   scratch: NULL, or moe_route_backward_scratch_size bytes of device memory (256-byte aligned).
 *   With it, a bf16 layer whose E is a multiple of 64 runs the three contractions on the tensor
 *   cores (dz entering them as two bf16 parts, hi + lo, so within ~2^-17 of fp32); its first word
 *   is then a device status word (moe_read_device_status).  Without it, or for other layers
 *   (size 0), they run in fp32 on the CUDA cores.
 * MOE_ERR_INVALID_ARG for NULL or misaligned pointers, MOE_ERR_UNSUPPORTED outside the shape
 * limits of the forward. */
moe_status moe_combine_backward(const moe_config* cfg, const void* dy, const float* y_perm,
                                const int32_t* row_of, const float* topk_w, float* dw, void* dy_perm,
                                void* stream);
moe_status moe_route_backward_scratch_size(const moe_config* cfg, size_t* bytes);
moe_status moe_route_backward(const moe_config* cfg, const void* x, const void* w_router,
                              const float* logit_bias, const int32_t* topk_idx, const float* topk_w,
                              const int32_t* counts, const float* dw, float dlb, float dzl, float* dz,
                              float* dw_router, float* dx, void* scratch, void* stream);

/* Gradients of the expert FFN weights, fp32, in the layouts of the weights in moe_weights. */
typedef struct {
  float* dw_up;    /* [E,dff,d]                                      */
  float* dw_gate;  /* [E,dff,d] (SwiGLU) or NULL                     */
  float* dw_down;  /* [E,d,dff]                                      */
  float* db_up;    /* [E,dff] (has_bias) or NULL                     */
  float* db_down;  /* [E,d]   (has_bias) or NULL                     */
  float* dws_up;   /* shared [S,dff,d] or NULL when n_shared == 0    */
  float* dws_gate; /* shared [S,dff,d] (SwiGLU) or NULL              */
  float* dws_down; /* shared [S,d,dff] or NULL                       */
} moe_expert_grads;

/* moe_expert_ffn_backward: the backward of the expert FFNs of moe_expert_ffn and of the shared
 * experts (the GELU FFN of the GPT-4 2% article, sec. 3.1, and the SwiGLU FFN of the same section;
 * shared experts see every token with weight 1, DeepSeekMoE in the OpenMythos article, sec. 3.2):
 *   x [T,d], x_perm [A_max,d], offsets [E+1] and row_of [T,k] as moe_permute left them, dy [T,d]
 *   the layer output's upstream gradient, dy_perm [A_max,d] from moe_combine_backward
 *   -> every gradient of g (overwritten; an expert with no rows gets zeros) and dx [T,d] fp32, to
 *      which the experts' part of the input gradient is ADDED (first the routed experts, each
 *      token's kept slots in slot order, then the shared experts in order), so that dx after
 *      moe_route_backward and this call is the layer's input gradient.
 * The pre-activations are recomputed from x_perm / x with fp32 accumulation; every sum runs in a
 * fixed order (bit-identical repeats).  bf16 layers contract on the tensor cores, with the
 * operands the backward creates (du, dg or da, h) rounded to bf16 and fp32 accumulation; fp32
 * layers run in fp32 on the CUDA cores.
 * scratch: moe_expert_backward_scratch_size bytes of device memory, 256-byte aligned; its first
 * word is a device status word that the call zeroes and moe_read_device_status(scratch) reads
 * (MOE_ERR_TIMEOUT when a bounded wait of the tensor-core kernel ran out).
 * MOE_ERR_UNSUPPORTED with a backup expert or 8-bit expert weights; MOE_ERR_INVALID_ARG for a
 * NULL or misaligned (16-byte) pointer that the config needs. */
moe_status moe_expert_backward_scratch_size(const moe_config* cfg, size_t* bytes);
moe_status moe_expert_ffn_backward(const moe_config* cfg, const moe_weights* w, const void* x,
                                   const void* x_perm, const int32_t* offsets, const int32_t* row_of,
                                   const void* dy, const void* dy_perm, const moe_expert_grads* g,
                                   float* dx, void* scratch, void* stream);

/* Device pointers to the forward's intermediates inside a workspace (host-only pointer arithmetic,
 * no GPU work).  After moe_layer_forward(cfg, ..., ws) they hold that call's topk_idx and topk_w
 * [T,k], counts [E] (only when the call's counts_out was NULL: otherwise that array holds them),
 * offsets [E+1], row_of [T,k], tok_of [A_max], x_perm [A_max,d] (layer dtype) and y_perm
 * [A_max,d] fp32 -- what moe_combine_backward, moe_route_backward and moe_expert_ffn_backward
 * take -- until the next call that uses the workspace.  MOE_ERR_INVALID_ARG for a NULL or
 * misaligned workspace or a NULL v. */
typedef struct {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* row_of;
  int32_t* tok_of;
  void* x_perm;
  float* y_perm;
} moe_forward_views;
moe_status moe_workspace_views(const moe_config* cfg, void* ws, moe_forward_views* v);

/* Static string for a status code. */
const char* moe_status_string(moe_status s);

/* Text of the last host-side failure behind a MOE_ERR_CUDA on this host thread (a tensor-map
 * encoding or a launch-configuration problem of the tensor-core kernels); "" if none.  Valid until
 * the next call on this thread. */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
