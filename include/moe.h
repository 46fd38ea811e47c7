/*
 * moe.h -- C ABI of the B300 (sm_103a) top-k Mixture-of-Experts FFN forward.
 *
 * The layer computes, for T tokens x[t] of width d, E experts of hidden width
 * h and k experts per token:
 *
 *   logits = x . W_g (+ logit_bias)                      router contraction
 *   G(x)   = softmax(TopK(logits))                       gate, two equal forms
 *   y[t]   = sum_{kept slots j} G_j(x_t) * E_{e_j}(x_t)   combine, slot order
 *   E_e(x) = W2[e] . SiLU(W1[e] . x + b1[e]) + b2[e]      expert FFN
 *   loss   = E * sum_e f_e * P_e                         load-balancing statistic
 *
 * as written on the page "MoE mixture-of-experts routing mechanism: principles
 * and sparse activation" (yunthe.com): the gating formula and output sum of
 * section "MoE architecture and gated routing principle", the TopKRouter /
 * Expert / MoELayer listing and load_balancing_loss of section "Top-K gated
 * routing PyTorch implementation", and the capacity rule of section "Expert
 * Choice routing and capacity-factor tuning".  The router / executor split
 * (indices and weights handed from the gate to an expert executor that groups
 * tokens by expert) follows "Breaking the MoE trilemma" (0539edu.com), 3.2-3.3.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller (CUDA allocations on the
 *    current device; the batches of moe_forward_host are host pointers),
 *    contiguous and row-major.  Activations, weights, expert
 *    biases, row buffers and the workspace are 16-byte aligned; int32 and fp32
 *    arrays 4-byte aligned; misalignment is MOE_ERR_INVALID_ARGUMENT.  With an
 *    empty batch (T = 0) the token-indexed buffers may be NULL.  The library
 *    allocates no memory (moe_forward_host creates two copy streams and some
 *    events per call and releases them), keeps no per-call state and may be
 *    called from several host threads on different streams with different
 *    workspaces.
 *  - Calls enqueue work on `stream` and return after host-side validation; no
 *    call waits for the GPU except moe_device_error.  The number of kept rows M
 *    never travels to the host: row buffers are sized for the worst case T*k.
 *  - Host-detectable problems return an error before anything is enqueued.
 *    Problems only the GPU can see (an expert index out of range, a row index
 *    out of range, a non-finite logit, a pipeline wait that gave up) set bits
 *    in a flag word at the start of the workspace; moe_device_error reads it.
 *    Kernels never trap.  Each entry point first clears the flag word and the
 *    bookkeeping that follows it (the first 5376 bytes of the workspace; the
 *    expert GEMMs' split-tile counters, which every completed layer leaves
 *    zeroed again).
 *  - Supported range: 1 <= k <= 8, k <= E <= 256, d and h multiples of 8 (and
 *    at least 8), 0 <= T and T*k < 2^31.  Outside it: MOE_ERR_UNSUPPORTED.
 *  - Weights use the nn.Linear orientation [out_features, in_features] stacked
 *    with the expert index first: W_g [E,d], W1 [E,h,d], b1 [E,h], W2 [E,d,h],
 *    b2 [E,d].  x, weights, expert biases and all row buffers share `dtype`;
 *    logits, gate weights, the logit bias and the loss are fp32.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1, /* NULL required pointer, misaligned pointer, bad enum */
  MOE_ERR_UNSUPPORTED = 2,      /* sizes outside the supported range */
  MOE_ERR_WORKSPACE = 3,        /* ws NULL or ws_bytes below the required size */
  MOE_ERR_CUDA = 4,             /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_DEVICE = 5            /* moe_device_error: the GPU raised a flag */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  /* G(x) = softmax(TopK(x . W_g)): non-kept logits at -inf, softmax over the kept
     (gating formula, "MoE architecture and gated routing principle"). */
  MOE_GATE_TOPK_SOFTMAX = 0,
  /* p = softmax(x . W_g); keep the top-k of p; divide them by their sum
     (TopKRouter.forward in the listing).  Same function as mode 0 up to rounding. */
  MOE_GATE_SOFTMAX_TOPK_RENORM = 1
} moe_gate;

/* Routing noise.  The random draws are an input, noise[T,E] fp32, supplied by the
   caller (so a run is reproducible and testable); the library applies the variant's
   arithmetic to the router logits l and selects the top-k of the resulting scores:
   - MOE_NOISE_GUMBEL: noise holds uniform draws u in (0,1); score = l + g with
     g = -log(-log(u + 1e-9) + 1e-9) (Gumbel top-k of the sparse-inference article
     (lpnh.cn), sections 2.3 and 3.2).  Gate weights and f use the scores as logits.
   - MOE_NOISE_PROB_GAUSS: noise holds scaled Gaussian draws n; score = softmax(l) + n
     (noise on the probabilities, MoE overview (cnnetsun.cn) section 2.1).  Gate
     weights and f use the clean logits l of the selected experts.
   - MOE_NOISE_LOGIT_SOFTMAX: noise holds scaled draws n; score = l + n * softmax(l)
     (noise injection of the routing-mechanism page, router-collapse section).  Gate
     weights and f use the scores as logits.
   With noise, the `logits` output holds the scores the selection used. */
typedef enum {
  MOE_NOISE_NONE = 0,
  MOE_NOISE_GUMBEL = 1,
  MOE_NOISE_PROB_GAUSS = 2,
  MOE_NOISE_LOGIT_SOFTMAX = 3
} moe_noise;

/* Routing statistics of the pre-drop per-expert counts, in this order (load_e =
   count_e / sum(count); sample standard deviations, divisor E-1, 0 when E = 1):
   cv = std(load)/mean(load); dead_ratio = share of experts with load < 1e-4;
   max_over_avg = max(load)/mean(load); entropy = -sum load ln(load + 1e-10);
   effective_experts = exp(entropy); count_cv_loss = std(count)/(mean(count) + 1e-6).
   From the monitoring script of "LLM MoE guide" (walkerchi.com) section 4.1 and the
   router load loss of the sparse-inference article (lpnh.cn) sections 2.3 and 3.2.
   All zero when there are no assignments. */
#define MOE_ROUTING_STATS 6
enum {
  MOE_STAT_CV = 0,
  MOE_STAT_DEAD_RATIO = 1,
  MOE_STAT_MAX_OVER_AVG = 2,
  MOE_STAT_ENTROPY = 3,
  MOE_STAT_EFFECTIVE_EXPERTS = 4,
  MOE_STAT_COUNT_CV_LOSS = 5
};

/* Bits of the device flag word (moe_device_error). */
enum {
  MOE_DEVERR_BAD_INDEX = 1, /* an expert index outside [0,E) reached dispatch; that slot was dropped */
  MOE_DEVERR_BAD_ROW = 2,   /* a slot_row outside [-1, T*k) reached combine; that slot was skipped */
  MOE_DEVERR_NONFINITE = 4, /* a router logit was NaN or infinite */
  MOE_DEVERR_TIMEOUT = 8    /* a bounded pipeline wait inside a GEMM gave up; outputs are invalid */
};

typedef struct moe_config {
  int64_t T;              /* tokens */
  int32_t d;              /* model width */
  int32_t h;              /* expert hidden width */
  int32_t E;              /* experts */
  int32_t k;              /* experts per token */
  int32_t dtype;          /* moe_dtype */
  int32_t gate;           /* moe_gate */
  double capacity_factor; /* > 0: capacity C = ceil(T * capacity_factor / E) kept assignments
                             per expert, later ones dropped; <= 0: no limit */
  int32_t noise;          /* moe_noise: routing noise applied before selection */
  /* 0 (default): moe_forward copies each kept token row into expert order (x_perm) before
     the expert GEMMs.  1: moe_forward's first expert GEMM reads the token rows straight
     from x (tile::gather4 loads by the dispatch's row -> token map) and the workspace holds
     no expert-ordered copy, T*k*d*2 bytes smaller (940 MB for T = 8192, k = 8,
     d = 7168) -- for callers short of device memory.  Results are bitwise identical; it
     is slower (the gathers issue more copies per k-block than the tiled loads).  bf16
     top-k layers only (MOE_ERR_UNSUPPORTED otherwise); a forward that is given an x_perm
     buffer fills it and uses it as with 0.  Stage calls are unaffected. */
  int32_t fused_gather;
} moe_config;

/* Inputs and outputs of moe_forward.  Outputs marked "or NULL" are optional;
   when NULL the library keeps them inside the workspace. */
typedef struct moe_forward_args {
  const void* x;            /* [T,d] dtype */
  const void* w_gate;       /* [E,d] dtype */
  const float* logit_bias;  /* [E] fp32 added to every token's logits, or NULL */
  const float* noise;       /* [T,E] fp32 random draws when cfg->noise != NONE, else NULL */
  const void* w1;           /* [E,h,d] dtype */
  const void* b1;           /* [E,h] dtype, or NULL for zero */
  const void* w2;           /* [E,d,h] dtype */
  const void* b2;           /* [E,d] dtype, or NULL for zero */
  void* y;                  /* [T,d] dtype, required */
  float* logits;            /* [T,E] fp32, or NULL */
  int32_t* topk_idx;        /* [T,k], or NULL */
  float* topk_w;            /* [T,k] fp32, or NULL */
  int32_t* counts;          /* [E] pre-drop assignments per expert, or NULL */
  float* aux_loss;          /* [1] fp32, or NULL */
  int32_t* offsets;         /* [E+1], or NULL */
  int32_t* kept_counts;     /* [E], or NULL */
  int32_t* slot_row;        /* [T,k], or NULL */
  int32_t* row_token;       /* [T*k], or NULL */
  int32_t* dropped;         /* [1], or NULL */
  float* routing_stats;     /* [MOE_ROUTING_STATS] fp32, or NULL (see moe_route) */
  /* Activations saved for moe_backward (each [T*k, .] dtype, or NULL to keep the
     forward's copy inside the workspace; h_pre is only written when given): */
  void* x_perm;             /* [T*k,d] the gathered token rows Xp */
  void* h_act;              /* [T*k,h] H = SiLU(A), GEMM1's output */
  void* y_perm;             /* [T*k,d] Yp, GEMM2's output.  A bf16 top-1 layer (k = 1)
                               whose groups are at most 128 rows (T, or C under a
                               capacity) folds the combine into the expert GEMMs when
                               this is NULL -- GEMM2 writes each kept token's row of y,
                               GEMM1 zeroes the dropped tokens' rows -- and then writes
                               no Yp anywhere; y is bitwise the same either way. */
  void* h_pre;              /* [T*k,h] A = W1 x + b1, the pre-activation */
} moe_forward_args;

/* Human-readable name of a status code.  Never NULL. */
const char* moe_status_str(moe_status s);

/* Capacity of the configuration: ceil(T * capacity_factor / E) computed in double
   ("capacity = tokens_per_batch / num_experts * capacity_factor", rounded up to a
   whole token), or -1 when capacity_factor <= 0.  Host only. */
moe_status moe_capacity(const moe_config* cfg, int64_t* capacity);

/* Workspace bytes moe_forward needs (includes the permuted row buffers
   [T*k,d] + [T*k,h] + [T*k,d]).  Host only. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Workspace bytes the stage calls (moe_route, moe_dispatch, moe_expert_ffn,
   moe_combine) need: the flag word, per-chunk histograms and partial sums,
   the [T,E] logits when moe_route is not given a logits buffer, and, when no
   expert can get more than 128 rows (bf16), the fp32 pieces of expert-GEMM tiles
   split between SMs (at most 20 MiB).  Host only. */
moe_status moe_stage_workspace_size(const moe_config* cfg, size_t* bytes);

/* Router (gating formula and TopKRouter.forward):
   logits[t,e] = sum_i x[t,i] W_g[e,i] + logit_bias[e]   (fp32 accumulation)
   topk_idx[t,j]: the j-th largest logit of token t (ties -> lower expert index)
   topk_w[t,j]  : gate weight of that expert by cfg->gate
   counts[e]    : number of (t,j) with topk_idx[t,j] == e (before any capacity drop)
   aux_loss[0]  : E * sum_e f_e P_e, f_e = mean_t softmax(logits)[t,e], P_e = counts[e]/T
   routing_stats: the MOE_ROUTING_STATS statistics of counts (above)
   noise        : [T,E] draws for cfg->noise (required then, else ignored)
   logits, counts, aux_loss and routing_stats may be NULL.  Selection and weights
   are computed from exactly the fp32 logits written.  Results are deterministic. */
moe_status moe_route(const moe_config* cfg, const void* x, const void* w_gate,
                     const float* logit_bias, const float* noise, float* logits,
                     int32_t* topk_idx, float* topk_w,
                     int32_t* counts, float* aux_loss, float* routing_stats, void* ws,
                     size_t ws_bytes, moe_stream_t stream);

/* Dispatch (capacity section; grouping by expert id of "Breaking the MoE
   trilemma" 3.3).  Visiting assignments token by token, slot by slot, expert e
   hands out positions 0,1,2,...; an assignment is kept iff capacity is off or
   its position < C.  offsets = exclusive prefix sum of kept_counts (offsets[E]
   = M kept rows).  Kept (t,j) of expert e goes to row offsets[e] + position:
   slot_row[t,j] = that row (-1 when dropped), row_token[row] = t (rows >= M are
   -1), x_perm[row,:] = x[t,:].  dropped[0] = T*k - M (may be NULL).  An index
   outside [0,E) is treated as dropped and raises MOE_DEVERR_BAD_INDEX. */
moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        int32_t* offsets, int32_t* kept_counts, int32_t* slot_row,
                        int32_t* row_token, int32_t* dropped, void* x_perm, void* ws,
                        size_t ws_bytes, moe_stream_t stream);

/* Expert FFN (Expert.forward) on the expert-contiguous rows:
   for every expert e and row r in [offsets[e], offsets[e+1]):
     h_buf[r,:]  = SiLU(x_perm[r,:] . W1[e]^T + b1[e])      (rounded to dtype)
     y_perm[r,:] = h_buf[r,:] . W2[e]^T + b2[e]             (rounded to dtype)
   with fp32 accumulation.  x_perm, h_buf and y_perm have T*k rows; rows >=
   offsets[E] are neither read for results nor written.  offsets must be
   non-decreasing with offsets[0] = 0 and offsets[E] <= T*k. */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const void* w1, const void* b1, const void* w2, const void* b2,
                          void* h_buf, void* y_perm, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* Combine (output sum; the listing adds each slot's expert output in slot order):
   y[t,:] = sum over j = 0..k-1 with slot_row[t,j] >= 0 of topk_w[t,j] * y_perm[slot_row[t,j],:]
   accumulated in fp32 in slot order and rounded once; a token with every slot
   dropped gets exactly 0.  No atomics: results are deterministic. */
moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot_row,
                       const float* topk_w, void* y, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* The whole layer: route, dispatch, expert FFN and combine on one stream, with
   every intermediate kept in `ws` (size from moe_workspace_size).  Equivalent to
   the four stage calls in order. */
moe_status moe_forward(const moe_config* cfg, const moe_forward_args* args, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* ---- Backward ------------------------------------------------------------------
   Gradients of the layer for training (the pages train the MoELayer but print no
   backward; this is the chain rule through the forward above).  With dy = dL/dy and
   d_aux = dL/d(aux_loss), for every kept slot (t,j) of expert e in row r:
     dYp[r] = w_tj dy_t;  dw_tj = <dy_t, Yp[r]>;  dA[r] = (dYp[r] W2[e]) * SiLU'(A[r]);
     dXp[r] = dA[r] W1[e];
     dW2[e] = sum_r dYp[r]^T H[r];  db2[e] = sum_r dYp[r];
     dW1[e] = sum_r dA[r]^T Xp[r];  db1[e] = sum_r dA[r];
     dl_t   = w_j (dw_j - sum_i w_i dw_i) on the TopK set (both gate forms) plus the
              balance-loss term d_aux (E/T) p_c (P_c - sum_e P_e p_e), P_e = counts_e / T;
     dW_g   = dl^T x;  dlogit_bias = sum_t dl_t;  dx_t = dl_t W_g + sum_j dXp[slot j].
   bf16 layers only (MOE_ERR_UNSUPPORTED for fp32), no routing noise.  GEMMs run on the
   tensor cores with bf16 operands (dYp, dA, dXp and dl rounded to bf16) and fp32
   accumulation; dW1, dW2 and the router's part of dx are rounded to bf16 once, dx once
   more after the slot sum; the other gradients are fp32.  Results are deterministic.  The routing and saved-activation inputs are the
   outputs of the moe_forward call being differentiated (same cfg). */
typedef struct moe_backward_args {
  const void* dy;           /* [T,d] dtype */
  const void* x;            /* [T,d] dtype */
  const void* w_gate;       /* [E,d] dtype */
  const void* w1;           /* [E,h,d] dtype */
  const void* w2;           /* [E,d,h] dtype */
  const float* logits;      /* [T,E] fp32 forward logits */
  const int32_t* topk_idx;  /* [T,k] */
  const float* topk_w;      /* [T,k] fp32 */
  const int32_t* counts;    /* [E] pre-drop assignments per expert */
  const int32_t* offsets;   /* [E+1] */
  const int32_t* slot_row;  /* [T,k] */
  const void* x_perm;       /* [T*k,d] dtype, forward's Xp */
  const void* h_pre;        /* [T*k,h] dtype, forward's A */
  const void* h_act;        /* [T*k,h] dtype, forward's H */
  const void* y_perm;       /* [T*k,d] dtype, forward's Yp */
  float d_aux;              /* dL / d aux_loss */
  void* dx;                 /* [T,d] dtype, required */
  float* dw_gate;           /* [E,d] fp32, or NULL */
  float* dlogit_bias;       /* [E] fp32, or NULL */
  void* dw1;                /* [E,h,d] dtype, or NULL */
  float* db1;               /* [E,h] fp32, or NULL */
  void* dw2;                /* [E,d,h] dtype, or NULL */
  float* db2;               /* [E,d] fp32, or NULL */
} moe_backward_args;

/* Workspace bytes moe_backward needs (dYp, dA, dXp row buffers, the router's part of
   dx and per-token gradients of the gate).  Host only. */
moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);

/* The layer's backward on one stream.  Device flags: MOE_DEVERR_TIMEOUT. */
moe_status moe_backward(const moe_config* cfg, const moe_backward_args* args, void* ws,
                        size_t ws_bytes, moe_stream_t stream);

/* ---- Expert-choice routing -------------------------------------------------
   The selection direction reversed (routing-mechanism page, section "Expert Choice
   routing and capacity-factor tuning"): instead of each token taking k experts,
   each expert takes a fixed number C of tokens, which balances the load by
   construction.  With p = softmax(logits) over the experts of each token:
     C             = min(T, ceil(T * capacity_factor / E))      (capacity rule)
     expert e takes the C tokens with the largest p[t,e] (equal p: lower t first)
     y[t,:]        = sum over experts e that took t, in ascending e, of
                     p[t,e] * E_e(x_t), accumulated in fp32 and rounded once;
                     a token no expert took gets exactly 0 (it leaves the layer
                     through the residual path).
   cfg->k and cfg->gate are not read; cfg->noise must be MOE_NOISE_NONE and
   cfg->capacity_factor > 0.  Selection is decided on exactly the fp32 p written to
   `probs`.  Supported range: 1 <= E <= 256, d and h as above, E*C < 2^31.
   Results are deterministic. */
typedef struct moe_expert_choice_args {
  const void* x;            /* [T,d] dtype */
  const void* w_gate;       /* [E,d] dtype */
  const float* logit_bias;  /* [E] fp32, or NULL */
  const void* w1;           /* [E,h,d] dtype */
  const void* b1;           /* [E,h] dtype, or NULL for zero */
  const void* w2;           /* [E,d,h] dtype */
  const void* b2;           /* [E,d] dtype, or NULL for zero */
  void* y;                  /* [T,d] dtype, required */
  float* logits;            /* [T,E] fp32, or NULL */
  float* probs;             /* [T,E] fp32 softmax of the logits, or NULL */
  int32_t* sel_token;       /* [E,C]: expert e's chosen tokens, ascending, or NULL */
  float* sel_w;             /* [E,C] fp32: p[sel_token, e], or NULL */
  int32_t* token_experts;   /* [T]: how many experts took each token, or NULL */
  int32_t* unrouted;        /* [1]: tokens no expert took, or NULL */
} moe_expert_choice_args;

/* C of the expert-choice layer (above).  Host only. */
moe_status moe_expert_choice_capacity(const moe_config* cfg, int64_t* capacity);

/* Workspace bytes moe_expert_choice_forward needs: router output, the [E,T]
   transposed probabilities and row map, and the row buffers [E*C,d] + [E*C,h] +
   [E*C,d].  Host only. */
moe_status moe_expert_choice_workspace_size(const moe_config* cfg, size_t* bytes);

/* The expert-choice layer on one stream: router contraction, softmax, per-expert
   top-C selection, row gather into expert-contiguous order (expert e owns rows
   [e*C, (e+1)*C)), the expert FFN on those rows (same kernels as moe_expert_ffn)
   and the per-token combine.  Device flags: MOE_DEVERR_NONFINITE (a non-finite
   logit), MOE_DEVERR_TIMEOUT (a GEMM wait gave up). */
moe_status moe_expert_choice_forward(const moe_config* cfg, const moe_expert_choice_args* args,
                                     void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---- Batches in host memory --------------------------------------------------
   A pipelined forward over a sequence of independent batches whose token rows x
   and outputs y live in HOST memory, for a caller that streams batches through one
   resident copy of the weights.  The pages have no counterpart; the layer itself is
   the one above.  Batch i's x is copied to the device, the layer runs on it (exactly
   the kernels of moe_forward, or of moe_expert_choice_forward, so its y is bitwise
   the y of that call on the same x), and its y is copied back.  The copies run on
   two streams the call creates (and releases before returning; CUDA frees them when
   their work completes), each batch's x and y double-buffered in the workspace, so
   batch i+1's host-to-device copy and batch i-1's device-to-host copy overlap batch
   i's layer.  A single batch, or batches of less than 256 KiB of x, run copy in,
   layer, copy out in order on `stream` alone (no streams created): there the copies
   are latency-bound and the hand-offs between streams cost more than they hide.
   Ordering: all of it starts after the work already enqueued on
   `stream`, and work enqueued on `stream` afterwards starts after all of it,
   including the last copy back; synchronise `stream` before reading y.
   Host buffers are the caller's and must stay valid (x unmodified) until then; they
   should be page-locked (cudaHostAlloc / cudaHostRegister): pageable memory gives the
   same results but the copies then do not overlap the layer.  Device flags
   accumulate over the batches (cleared once at the start; moe_device_error(ws)). */
typedef enum { MOE_ROUTING_TOPK = 0, MOE_ROUTING_EXPERT_CHOICE = 1 } moe_routing;

/* Device-resident weights shared by every batch (same shapes, dtype and rules as
   the fields of moe_forward_args of the same names). */
typedef struct moe_weights {
  const void* w_gate;       /* [E,d] dtype */
  const float* logit_bias;  /* [E] fp32, or NULL */
  const void* w1;           /* [E,h,d] dtype */
  const void* b1;           /* [E,h] dtype, or NULL for zero */
  const void* w2;           /* [E,d,h] dtype */
  const void* b2;           /* [E,d] dtype, or NULL for zero */
} moe_weights;

typedef struct moe_host_batches {
  int64_t n;                /* number of batches, >= 1 */
  const void* const* x;     /* [n] HOST pointers, each to a [T,d] dtype batch (NULL only if T = 0) */
  void* const* y;           /* [n] HOST pointers, each to [T,d] dtype outputs (NULL only if T = 0) */
  float* aux_loss;          /* [n] HOST fp32: batch i's balance statistic (top-k routing
                               only; must be NULL for expert choice), or NULL */
} moe_host_batches;

/* Workspace bytes moe_forward_host needs: the routing's forward workspace followed
   by two device copies of a batch's x and two of its y.  routing: moe_routing.
   Host only. */
moe_status moe_forward_host_workspace_size(const moe_config* cfg, int32_t routing,
                                           size_t* bytes);

/* The pipelined forward over host batches (above).  cfg->noise must be
   MOE_NOISE_NONE (the draws are per-batch device inputs): otherwise
   MOE_ERR_UNSUPPORTED.  Every argument, and the layer's own validation, is checked
   before anything is enqueued.  With T = 0 nothing is copied and aux_loss, when
   given, is set to 0 on the host before the call returns. */
moe_status moe_forward_host(const moe_config* cfg, int32_t routing, const moe_weights* weights,
                            const moe_host_batches* batches, void* ws, size_t ws_bytes,
                            moe_stream_t stream);

/* Waits for `stream`, then reads the device flag word at the start of `ws` into
   *flags (may be NULL).  Returns MOE_ERR_DEVICE when any bit is set, MOE_OK
   otherwise, MOE_ERR_CUDA if the wait or the read failed. */
moe_status moe_device_error(const void* ws, moe_stream_t stream, int32_t* flags);

/* Diagnostic of the bounded waits.  Every mbarrier wait in the GEMM pipelines gives
   up after a time limit instead of spinning forever: it sets MOE_DEVERR_TIMEOUT, lets
   the CTA's own copies and MMAs land, frees tensor memory and returns.  This call runs
   that same wait routine on a barrier phase nothing completes, for limit_ns
   nanoseconds (1 .. 2e9), in one small kernel on `stream`; afterwards *device_flags (a
   [1] int32 device buffer, cleared first) holds MOE_DEVERR_TIMEOUT and the GPU context
   is unaffected.  The pages have no counterpart. */
moe_status moe_selftest_wait_timeout(int32_t* device_flags, uint64_t limit_ns,
                                     moe_stream_t stream);

/* Table cells (ceil(T/64) * E) that moe_dispatch_static's library-held scratch holds:
   2 MiB of device memory in every GPU that loads the library. */
#define MOE_DISPATCH_STATIC_MAX_CELLS 262144

/* moe_dispatch without a workspace.  The pages have no counterpart to this entry
   point: it exists for callers that cannot allocate device memory at the call site
   -- code running under a host framework that owns all device memory and forbids
   allocation once it is serving, or a plugin that is handed only its inputs and
   outputs -- and so cannot pass the workspace moe_dispatch needs.  It computes
   exactly what moe_dispatch computes (same arguments and outputs, same kernels)
   and calls no allocator.  Its scratch (per-chunk tables and the flag word) is one
   array owned by the library:
    - sizes with ceil(T/64) * E > MOE_DISPATCH_STATIC_MAX_CELLS return
      MOE_ERR_UNSUPPORTED (T <= 65536 tokens at E = 256);
    - every call shares the array and it keeps the last call's contents; each call
      rewrites what it reads and clears the flag word, but calls whose GPU work
      overlaps (other streams, other host threads) race on it: serialise them;
    - the array's device address is looked up by the first call made in a CUDA
      context (the device's primary context, for runtime-API callers) and reused
      while that context is current; a call in a new context (after
      cudaDeviceReset, say) looks it up again.  Make the first call in a context
      before any stream capture begins.
   Arguments are validated exactly as moe_dispatch validates them.
   device_flags: optional [1] int32 device buffer that receives the device flag word
   (MOE_DEVERR_BAD_INDEX); NULL keeps it inside the library's array. */
moe_status moe_dispatch_static(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               int32_t* offsets, int32_t* kept_counts, int32_t* slot_row,
                               int32_t* row_token, int32_t* dropped, void* x_perm,
                               int32_t* device_flags, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
