// Host-side launchers of the MoE kernels (one per kernel family).  Each returns
// the launch status; none allocates or synchronises.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// R2 + R3: softmax, top-k, gate weights, per-chunk expert histogram and per-chunk
// softmax column sums.  The logits of token t are
//   l[t,e] = sum_{s < nsplit} src[s * split_stride + t*E + e]  (+ bias[e] if bias)
// added in that order; when logits_out is given they are written there.
// With noise_mode != 0 the selection scores follow moe.h's moe_noise (draws in
// noise[T,E]) and logits_out receives those scores.
cudaError_t launch_route_topk(const float* src, int nsplit, int64_t split_stride,
                              const float* bias, const float* noise, int noise_mode,
                              float* logits_out, int64_t T, int E, int k, int gate,
                              int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum,
                              int* flags, cudaStream_t stream);

// R4 + D1: reduces the per-chunk histograms (and, when psum != nullptr, the softmax
// sums into the balance loss), then applies the capacity and scans the offsets;
// with stats != nullptr also writes the six routing statistics of the counts.
// Any of counts/aux/chunk_base/kept/offsets/dropped/stats may be nullptr.
cudaError_t launch_route_finalize(const int32_t* hist, const float* psum, int nchunks, int E,
                                  int64_t T, int64_t C, int32_t* counts, float* aux,
                                  int32_t* chunk_base, int32_t* kept, int32_t* offsets,
                                  int32_t* dropped, float* stats, cudaStream_t stream);

// Per-chunk expert histogram of caller-provided indices (moe_dispatch on its own).
cudaError_t launch_dispatch_hist(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* hist,
                                 int* flags, cudaStream_t stream);

// D2 + D3: stable positions, capacity drop, slot_row / row_token and the expert-ordered
// rows (copied token by token to each kept row; not copied when x_perm is nullptr).
cudaError_t launch_dispatch_place(int dtype, const int32_t* topk_idx, int64_t T, int E, int k,
                                  int64_t C, const int32_t* chunk_base, const int32_t* offsets,
                                  int32_t* slot_row, int32_t* row_token, const void* x,
                                  void* x_perm, int d, int* flags, cudaStream_t stream);

// D3 alone: x_perm[r] = x[row_token[r]] for r < offsets[E]; `rows` bounds offsets[E].
cudaError_t launch_gather_rows(int dtype, const int32_t* row_token, const int32_t* offsets, int E,
                               const void* x, void* x_perm, int d, int64_t rows,
                               cudaStream_t stream);

// EC1: logits l (split partials added in order, then the bias), p = softmax(l) per
// token; writes logits_out / probs_out [T,E] when given and probs_et [E,T] always.
cudaError_t launch_ec_softmax(const float* src, int nsplit, int64_t split_stride,
                              const float* bias, float* logits_out, float* probs_out,
                              float* probs_et, int64_t T, int E, int* flags, cudaStream_t stream);

// EC2: per expert e, its C largest p[., e] (lower token first on equal values) in
// ascending token order: sel_token / sel_w [E,C]; rowmap_et[e,t] = position c or -1;
// offsets[e] = e*C.  Requires C <= T.
cudaError_t launch_ec_select(const float* probs_et, int64_t T, int E, int64_t C,
                             int32_t* sel_token, float* sel_w, int32_t* rowmap_et,
                             int32_t* offsets, cudaStream_t stream);

// EC3: y[t] = sum over experts e with rowmap_et[e,t] = c >= 0, ascending e, of
// probs_et[e,t] * y_perm[e*C + c]; token_experts[t] and unrouted (both optional).
cudaError_t launch_ec_combine(int dtype, const void* y_perm, const int32_t* rowmap_et,
                              const float* probs_et, int64_t T, int E, int64_t C, int d, void* y,
                              int32_t* token_experts, int32_t* unrouted, cudaStream_t stream);

// C1: y[t] = sum_j w[t,j] * y_perm[slot_row[t,j]] in slot order.
cudaError_t launch_combine(int dtype, const void* y_perm, const int32_t* slot_row,
                           const float* topk_w, int64_t T, int d, int k, void* y, int* flags,
                           cudaStream_t stream);

// Grouped GEMM operands.  Rows of A for group g are [offsets[g], offsets[g+1]) (or
// [0, m_rows) with one group when offsets == nullptr); B is [G][N][K] (K-major);
// out[row, n] = act(sum_k A[row,k] * B[g][n][k] + bias[g][n]).
struct GemmArgs {
  const void* A;          // [rows_alloc, K]
  int64_t rows_alloc;     // rows of the A / out buffers
  const void* B;          // [G, N, K]
  const void* bias;       // [G, N] in the operand dtype, or fp32 [N] (router), or nullptr
  void* out;              // [rows_alloc, N]
  const int32_t* offsets; // [G+1] device, or nullptr
  int64_t m_rows;         // rows when offsets == nullptr
  int G, N, K;
  int max_group;          // upper bound on any group's rows (sizes the token tile)
  int ksplit;             // router: K splits; split s writes out + s * split_stride
  int64_t split_stride;
  int* flags;
  void* pre_out;          // EPI_BIAS_SILU: also writes the pre-activation (before SiLU), or nullptr
  // Backward: EPI_DSILU multiplies by SiLU'(aux_in[row, n]) (the saved pre-activation).
  const void* aux_in;
  int64_t b_rows;  // backward B [G][b_rows][N] when b_rows differs from K (rows past it read 0)
  // Weights-as-M expert GEMM (groups <= 128 rows), whose (tile, k-block) iterations are
  // split evenly over the CTAs: kSplitCounters zeroed ints (left zeroed again) and
  // split_part_floats(max_group) floats for the pieces of split tiles.
  int* sk_ctr;
  float* sk_part;
  // Expert GEMM 1 only: when gather_rows is given, the token rows of row r are read
  // straight from gather_src [gather_src_rows, K] at row gather_rows[r] (the dispatch's
  // row -> token map) instead of from A, which is then not read.
  const int32_t* gather_rows;
  const void* gather_src;
  int64_t gather_src_rows;
  // The combine of a top-1 layer folded into the weights-as-M expert GEMMs (comb_token
  // given; comb_out is the layer output [comb_rows, comb_cols]).  GEMM 2: row r's output
  // goes to comb_out at row comb_token[r] (the row -> token map), scaled by that token's
  // gate weight comb_w[token] exactly as the combine scales its one slot (fma(w, output
  // rounded to bf16, 0), rounded to bf16), instead of to out.  GEMM 1: its epilogue warps
  // first set to zero the comb_out rows of the tokens whose slot comb_slot[token] was
  // dropped (-1), while the first tiles' operands stream in.
  const int32_t* comb_token;
  const float* comb_w;
  const int32_t* comb_slot;
  void* comb_out;
  int64_t comb_rows;
  int comb_cols;
};

// K splits of the bf16 router contraction for T tokens, E experts, model width d on a
// GPU with `sms` SMs: enough (tile, split) work units to fill the GPU, at least four
// 64-deep k-blocks per split.  Depends only on its arguments, so the workspace size
// can bound it with an upper limit on the SM count.
int router_splits(int64_t T, int E, int d, int sms);
constexpr int kMaxSmsForSizing = 160;

// Largest expert group (rows) for which the expert GEMMs use the weights-as-M kernel
// (token tiles of 32, 64 or 128 rows); larger groups use 128-row tiles of tokens.
constexpr int kSmallGroup = 128;
// Counters of the weights-as-M expert GEMM's split tiles: one per (CTA, TMEM lane
// quadrant).  Each GEMM of a layer has its own set.
constexpr int kSplitCounters = 4 * kMaxSmsForSizing;
// Floats for the parked pieces of that GEMM's split tiles: two [128 x token tile]
// pieces per CTA; none when the groups are too large for that kernel.
inline int64_t split_part_floats(int64_t max_group) {
  if (max_group > kSmallGroup) return 0;
  const int64_t tb = max_group <= 32 ? 32 : max_group <= 64 ? 64 : 128;
  return int64_t{kMaxSmsForSizing} * 2 * 128 * tb;
}

enum Epilogue {
  EPI_BIAS_SILU = 0,
  EPI_BIAS = 1,
  EPI_ROUTER_F32 = 2,
  EPI_DSILU = 3,  // out = acc * SiLU'(pre)
  EPI_PLAIN = 4   // out = acc
};

// Backward GEMMs on row tiles (bf16): A [rows, K] K-major as in the forward, B stored
// [G][K][N] (N contiguous: the forward weights read transposed, MN-major), epilogue
// EPI_DSILU or EPI_PLAIN, bf16 output [rows, N].  offsets == nullptr: one dense group
// of m_rows rows.
cudaError_t launch_tc_bwd_rows(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream);

// Weight gradients: for each group g with rows [offsets[g], offsets[g+1]) (or one
// group of m_rows rows when offsets == nullptr):
//   out[g][m][n] = sum_{r in g} A[r][m] * B[r][n],  m < Mdim, n < Ndim,
// A [rows, Mdim] and B [rows, Ndim] bf16 row-major (both read MN-major), fp32
// accumulation, out bf16 or fp32; a group without rows gets zeros.
struct WgradArgs {
  const void* A;
  int Mdim;
  const void* B;
  int Ndim;
  const int32_t* offsets;
  int64_t m_rows;
  int64_t rows_alloc;  // rows of the A and B buffers
  int G;
  void* out;
  bool out_f32;
  int* flags;
  // With offsets: each group's last k-block when it is partial, zero-padded to 64 rows
  // ([G, 64, Mdim] and [G, 64, Ndim], see launch_pack_tails).
  const void* tailA;
  const void* tailB;
};
cudaError_t launch_tc_wgrad(const WgradArgs& a, int sm_count, cudaStream_t stream);

// For every group with rows [offsets[g], offsets[g+1]) whose last 64-row block is partial:
// tail[g][r] = A[offsets[g] + 64*(nkb-1) + r] for r < the block's rows, 0 up to 64 rows
// (bf16, [G, 64, cols]); other groups' slots are not written.
cudaError_t launch_pack_tails(const void* A, int cols, const int32_t* offsets, int G, void* tail,
                              cudaStream_t stream);

// Backward of the combine: for kept slot (t,j) in row r = slot_row[t,j]:
//   dy_perm[r] = topk_w[t,j] * dy[t] (bf16),  dw[t,j] = <dy[t], y_perm[r]> (fp32);
// a dropped slot gets dw = 0.
cudaError_t launch_bwd_combine(const void* dy, const void* y_perm, const int32_t* slot_row,
                               const float* topk_w, int64_t T, int d, int k, void* dy_perm,
                               float* dw, cudaStream_t stream);

// Backward of the gate and the balance loss to the logits: dl [T,E] fp32 and its bf16
// copy dl16 [T,Epad] (columns E..Epad-1 zero, Epad <= 256).
cudaError_t launch_bwd_gate(const float* logits, const int32_t* topk_idx, const float* topk_w,
                            const float* dw, const int32_t* counts, float d_aux, int64_t T,
                            int E, int Epad, int k, float* dl, void* dl16, cudaStream_t stream);

// dx[t] = dxr[t] + sum_j dXp[slot_row[t,j]] (slots in order, dropped slots skipped),
// fp32 sums rounded once to bf16.
cudaError_t launch_bwd_dx(const void* dxr, const void* dxp, const int32_t* slot_row, int64_t T,
                          int d, int k, void* dx, cudaStream_t stream);

// Column sums per group: out[g][c] = sum over rows r of group g of A[r][c] (rows in
// order within 64-row slices, slices in order), A bf16 (a_f32 = false) or fp32.
// partial: workspace of colsum_partial_floats(...) floats.
int64_t colsum_partial_floats(int64_t rows_alloc, int G, int C);
cudaError_t launch_colsum(const void* A, bool a_f32, int C, const int32_t* offsets, int64_t m_rows,
                          int64_t rows_alloc, int G, float* partial, float* out,
                          cudaStream_t stream);

// fp32 SIMT grouped GEMM (fp32 operands, fp32 bias and output).
cudaError_t launch_simt_gemm_f32(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream);

// bf16 tcgen05 grouped GEMM (bf16 operands).  EPI_BIAS_SILU / EPI_BIAS take a bf16
// bias and write bf16; EPI_ROUTER_F32 takes an fp32 [N] bias and writes fp32.
cudaError_t launch_tc_gemm_bf16(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream);

}  // namespace moe
