// C ABI of the MoE FFN forward (include/moe.h): argument validation, workspace
// carving and the launch sequence of every entry point.  Nothing here allocates
// device memory, synchronises (except moe_device_error) or keeps per-call state.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "../../include/moe.h"
#include "common.cuh"
#include "entry.h"
#include "kernels.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

// Trace ranges, compiled in only with MOE_NVTX (python -m sparse_mixture_experts_61_b300.build
// --force with MOE_NVTX=1 in the environment): each stage of moe_forward's enqueue becomes
// an NVTX range on the calling host thread, which a timeline tool shows over that stage's
// kernel launches.  Without the switch the macro expands to nothing.
#ifdef MOE_NVTX
#include <nvtx3/nvToolsExt.h>
namespace moe {
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};
}  // namespace moe
#define MOE_TRACE(name) ::moe::TraceRange moe_trace_range_(name)
#else
#define MOE_TRACE(name) static_cast<void>(0)
#endif

namespace moe {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Workspace layout: [flags | per-chunk hist | chunk bases | per-chunk softmax sums |
// router output] = the stage workspace, then the forward-only intermediates.  The
// router output region holds the [T,E] fp32 logits (fp32 layers) or the K-split
// partial sums of the bf16 router GEMM.
struct Layout {
  size_t flags, split_ctr, hist, chunk_base, psum, logits, split_part, stage_end;
  size_t idx, w, counts, aux, offsets, kept, slot_row, row_token, dropped, x_perm, h_buf, y_perm;
  size_t total;
  int64_t nchunks;
};

int64_t capacity_of(const moe_config& c);

// Largest expert group a valid top-k routing can produce: T (one row per token), or C
// under a capacity below T.
int64_t max_group_of(const moe_config& c) {
  const int64_t C = capacity_of(c);
  return C >= 0 && C < c.T ? C : c.T;
}

// Top-1 bf16 layers whose expert groups fit the weights-as-M GEMMs get the combine folded
// into the expert GEMMs in moe_forward (with k = 1 the combine only scales and moves rows):
// GEMM 1 zeroes the output rows of dropped tokens, GEMM 2 writes the others.
bool fused_top1_combine(const moe_config& c) {
  return c.k == 1 && c.dtype == MOE_BF16 && max_group_of(c) <= kSmallGroup;
}

struct TopOneCombine {
  const int32_t* row_token;  // [T*k] row -> token
  const float* w;            // [T] gate weights
  const int32_t* slot_row;   // [T] token -> row, -1 when dropped
  void* y;                   // [T, d] layer output
};

Layout make_layout(const moe_config& c) {
  Layout L{};
  const int64_t T = c.T, E = c.E, k = c.k;
  const size_t s = c.dtype == MOE_F32 ? 4 : 2;
  L.nchunks = (T + kChunk - 1) / kChunk;
  size_t o = 0;
  L.flags = o; o += kAlign;
  L.split_ctr = o; o = align_up(o + 2 * kSplitCounters * sizeof(int));
  L.hist = o; o = align_up(o + L.nchunks * E * 4);
  L.chunk_base = o; o = align_up(o + L.nchunks * E * 4);
  L.psum = o; o = align_up(o + L.nchunks * E * 4);
  const int64_t splits =
      c.dtype == MOE_BF16 ? router_splits(c.T, c.E, c.d, kMaxSmsForSizing) : 1;
  L.logits = o; o = align_up(o + splits * T * E * 4);
  L.split_part = o;
  if (c.dtype == MOE_BF16) o = align_up(o + split_part_floats(max_group_of(c)) * 4);
  L.stage_end = o;
  L.idx = o; o = align_up(o + T * k * 4);
  L.w = o; o = align_up(o + T * k * 4);
  L.counts = o; o = align_up(o + E * 4);
  L.aux = o; o = align_up(o + 4);
  L.offsets = o; o = align_up(o + (E + 1) * 4);
  L.kept = o; o = align_up(o + E * 4);
  L.slot_row = o; o = align_up(o + T * k * 4);
  L.row_token = o; o = align_up(o + T * k * 4);
  L.dropped = o; o = align_up(o + 4);
  L.x_perm = o; if (!c.fused_gather) o = align_up(o + T * k * c.d * s);
  L.h_buf = o; o = align_up(o + T * k * c.h * s);
  L.y_perm = o; o = align_up(o + T * k * c.d * s);
  L.total = o;
  return L;
}
static_assert(kAlign + 2 * kSplitCounters * sizeof(int) == kFlagRegionBytes,
              "the flag word and the split counters open every forward workspace");

}  // namespace

// Shared with moe_dispatch_static (entry.h).
moe_status check_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARGUMENT;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARGUMENT;
  if (c->gate != MOE_GATE_TOPK_SOFTMAX && c->gate != MOE_GATE_SOFTMAX_TOPK_RENORM)
    return MOE_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARGUMENT;
  if (c->noise < MOE_NOISE_NONE || c->noise > MOE_NOISE_LOGIT_SOFTMAX)
    return MOE_ERR_INVALID_ARGUMENT;
  if (c->fused_gather != 0 && c->fused_gather != 1) return MOE_ERR_INVALID_ARGUMENT;
  if (c->fused_gather && c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->T < 0 || c->k < 1 || c->k > kMaxK || c->E < c->k || c->E > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (c->d < 8 || c->d % 8 != 0 || c->h < 8 || c->h % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (c->T * static_cast<int64_t>(c->k) >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

namespace {

int64_t capacity_of(const moe_config& c) {
  if (!(c.capacity_factor > 0.0)) return -1;
  return static_cast<int64_t>(
      std::ceil(static_cast<double>(c.T) * c.capacity_factor / static_cast<double>(c.E)));
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
// Required 16-byte-aligned buffer.
bool need16(const void* p) { return p != nullptr && al16(p); }
// Required 4-byte-aligned array.
bool need4(const void* p) { return p != nullptr && al4(p); }
// Optional arrays: NULL or aligned.
bool opt16(const void* p) { return p == nullptr || al16(p); }
bool opt4(const void* p) { return p == nullptr || al4(p); }
// Token-indexed buffers are required unless the batch is empty (T = 0), where they
// hold no element and may be NULL.
bool tok16(const moe_config& c, const void* p) { return c.T == 0 ? opt16(p) : need16(p); }
bool tok4(const moe_config& c, const void* p) { return c.T == 0 ? opt4(p) : need4(p); }

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

#define MOE_CUDA(call)                            \
  do {                                            \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// R1 + R2 + R3: the router contraction, then softmax / top-k / weights / per-chunk
// histogram and softmax sums.  fp32 layers: a SIMT GEMM writes the biased logits
// (into `logits`, or the workspace).  bf16 layers: the tensor-core GEMM writes
// K-split partial sums into the workspace; the top-k kernel adds them and the logit
// bias and writes the logits to `logits` when given.
moe_status run_router(const moe_config& c, const Layout& L, void* ws, const void* x,
                      const void* w_gate, const float* logit_bias, const float* noise,
                      float* logits, int32_t* topk_idx, float* topk_w, int* flags, int sms,
                      cudaStream_t st) {
  GemmArgs g{};
  g.A = x;
  g.rows_alloc = c.T;
  g.B = w_gate;
  g.offsets = nullptr;
  g.m_rows = c.T;
  g.G = 1;
  g.N = c.E;
  g.K = c.d;
  g.flags = flags;
  float* region = at<float>(ws, L.logits);
  int32_t* hist = at<int32_t>(ws, L.hist);
  float* psum = at<float>(ws, L.psum);
  if (c.dtype == MOE_F32) {
    // Without noise the GEMM's biased logits are the output; with noise the output is
    // the selection scores, written by the top-k kernel.
    const bool noisy = c.noise != MOE_NOISE_NONE;
    float* lg = (logits && !noisy) ? logits : region;
    g.bias = logit_bias;
    g.out = lg;
    MOE_CUDA(launch_simt_gemm_f32(g, EPI_ROUTER_F32, sms, st));
    MOE_CUDA(launch_route_topk(lg, 1, 0, nullptr, noise, c.noise, noisy ? logits : nullptr, c.T,
                               c.E, c.k, c.gate, topk_idx, topk_w, hist, psum, flags, st));
  } else {
    g.bias = nullptr;
    g.out = region;
    g.ksplit = router_splits(c.T, c.E, c.d, sms < kMaxSmsForSizing ? sms : kMaxSmsForSizing);
    g.split_stride = c.T * c.E;
    MOE_CUDA(launch_tc_gemm_bf16(g, EPI_ROUTER_F32, sms, st));
    MOE_CUDA(launch_route_topk(region, g.ksplit, g.split_stride, logit_bias, noise, c.noise,
                               logits, c.T, c.E, c.k, c.gate, topk_idx, topk_w, hist, psum, flags,
                               st));
  }
  return MOE_OK;
}

// G1 + G2 over the expert-contiguous rows: `rows_alloc` rows in the buffers, no
// expert with more than `max_group` rows.
// sk_ctr: the two GEMMs' split counters (2 * kSplitCounters zeroed ints); sk_part:
// split_part_floats(max_group) floats.
moe_status run_expert_ffn_rows(const moe_config& c, int64_t rows_alloc, int64_t max_group,
                               const void* x_perm, const int32_t* offsets, const void* w1,
                               const void* b1, const void* w2, const void* b2, void* h_buf,
                               void* y_perm, int* flags, int* sk_ctr, float* sk_part, int sms,
                               cudaStream_t st, void* h_pre = nullptr,
                               const int32_t* gather_rows = nullptr, const void* x = nullptr,
                               const TopOneCombine* top1 = nullptr) {
  GemmArgs g1{};
  g1.A = x_perm;
  g1.pre_out = h_pre;
  g1.rows_alloc = rows_alloc;
  g1.B = w1;
  g1.bias = b1;
  g1.out = h_buf;
  g1.offsets = offsets;
  g1.G = c.E;
  g1.N = c.h;
  g1.K = c.d;
  g1.max_group = static_cast<int>(max_group);
  g1.flags = flags;
  g1.sk_ctr = sk_ctr;
  g1.sk_part = sk_part;
  g1.gather_rows = gather_rows;
  g1.gather_src = x;
  g1.gather_src_rows = c.T;
  if (top1) {
    g1.comb_token = top1->row_token;
    g1.comb_w = top1->w;
    g1.comb_slot = top1->slot_row;
    g1.comb_out = top1->y;
    g1.comb_rows = c.T;
    g1.comb_cols = c.d;
  }
  GemmArgs g2 = g1;
  g2.sk_ctr = sk_ctr + kSplitCounters;
  g2.gather_rows = nullptr;
  g2.gather_src = nullptr;
  g2.A = h_buf;
  g2.pre_out = nullptr;
  g2.B = w2;
  g2.bias = b2;
  g2.out = y_perm;
  g2.N = c.d;
  g2.K = c.h;
  if (c.dtype == MOE_F32) {
    MOE_CUDA(launch_simt_gemm_f32(g1, EPI_BIAS_SILU, sms, st));
    MOE_CUDA(launch_simt_gemm_f32(g2, EPI_BIAS, sms, st));
  } else {
    MOE_CUDA(launch_tc_gemm_bf16(g1, EPI_BIAS_SILU, sms, st));
    MOE_CUDA(launch_tc_gemm_bf16(g2, EPI_BIAS, sms, st));
  }
  return MOE_OK;
}

// Top-k routing: a valid routing gives an expert at most T rows (one per token), and
// at most C with a capacity; the tile height follows this bound.
moe_status run_expert_ffn(const moe_config& c, const Layout& L, void* ws, const void* x_perm,
                          const int32_t* offsets, const void* w1, const void* b1, const void* w2,
                          const void* b2, void* h_buf, void* y_perm, int* flags, int sms,
                          cudaStream_t st, void* h_pre = nullptr,
                          const int32_t* gather_rows = nullptr, const void* x = nullptr,
                          const TopOneCombine* top1 = nullptr) {
  return run_expert_ffn_rows(c, c.T * c.k, max_group_of(c), x_perm, offsets, w1, b1, w2, b2, h_buf,
                             y_perm, flags, at<int>(ws, L.split_ctr), at<float>(ws, L.split_part),
                             sms, st, h_pre, gather_rows, x, top1);
}

// ---------------------------------------------------------------- expert choice
// Workspace: [flags | router output | probs [E,T] | row map [E,T] | offsets |
// sel_token | sel_w | token rows x_perm, h_buf, y_perm of E*C rows].
struct EcLayout {
  size_t flags, split_ctr, logits, probs_et, rowmap, offsets, sel_token, sel_w, split_part, x_perm,
      h_buf, y_perm, total;
  int64_t C;
};

int64_t ec_capacity_of(const moe_config& c) {
  const int64_t C = static_cast<int64_t>(
      std::ceil(static_cast<double>(c.T) * c.capacity_factor / static_cast<double>(c.E)));
  return C < c.T ? C : c.T;
}

moe_status check_ec_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARGUMENT;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(c->capacity_factor) || !(c->capacity_factor > 0.0))
    return MOE_ERR_INVALID_ARGUMENT;
  if (c->noise != MOE_NOISE_NONE) return MOE_ERR_INVALID_ARGUMENT;
  if (c->fused_gather != 0 && c->fused_gather != 1) return MOE_ERR_INVALID_ARGUMENT;
  if (c->fused_gather) return MOE_ERR_UNSUPPORTED;  // top-k layers only
  if (c->T < 0 || c->T >= (int64_t{1} << 31) || c->E < 1 || c->E > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  if (c->d < 8 || c->d % 8 != 0 || c->h < 8 || c->h % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (ec_capacity_of(*c) * c->E >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

EcLayout make_ec_layout(const moe_config& c) {
  EcLayout L{};
  const int64_t T = c.T, E = c.E;
  const size_t s = c.dtype == MOE_F32 ? 4 : 2;
  L.C = ec_capacity_of(c);
  const int64_t rows = E * L.C;
  size_t o = 0;
  L.flags = o; o += kAlign;
  L.split_ctr = o; o = align_up(o + 2 * kSplitCounters * sizeof(int));
  const int64_t splits =
      c.dtype == MOE_BF16 ? router_splits(c.T, c.E, c.d, kMaxSmsForSizing) : 1;
  L.logits = o; o = align_up(o + splits * T * E * 4);
  L.probs_et = o; o = align_up(o + T * E * 4);
  L.rowmap = o; o = align_up(o + T * E * 4);
  L.offsets = o; o = align_up(o + (E + 1) * 4);
  L.sel_token = o; o = align_up(o + rows * 4);
  L.sel_w = o; o = align_up(o + rows * 4);
  L.split_part = o;
  if (c.dtype == MOE_BF16) o = align_up(o + split_part_floats(L.C) * 4);
  L.x_perm = o; o = align_up(o + rows * c.d * s);
  L.h_buf = o; o = align_up(o + rows * c.h * s);
  L.y_perm = o; o = align_up(o + rows * c.d * s);
  L.total = o;
  return L;
}

moe_status zero_async(void* p, size_t bytes, cudaStream_t st) {
  if (p && bytes) MOE_CUDA(cudaMemsetAsync(p, 0, bytes, st));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_EXPORT const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARGUMENT: return "MOE_ERR_INVALID_ARGUMENT";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

MOE_EXPORT moe_status moe_capacity(const moe_config* cfg, int64_t* capacity) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!capacity) return MOE_ERR_INVALID_ARGUMENT;
  *capacity = capacity_of(*cfg);
  return MOE_OK;
}

MOE_EXPORT moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  *bytes = make_layout(*cfg).total;
  return MOE_OK;
}

MOE_EXPORT moe_status moe_stage_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  *bytes = make_layout(*cfg).stage_end;
  return MOE_OK;
}

MOE_EXPORT moe_status moe_route(const moe_config* cfg, const void* x, const void* w_gate,
                                const float* logit_bias, const float* noise, float* logits,
                                int32_t* topk_idx,
                                float* topk_w, int32_t* counts, float* aux_loss,
                                float* routing_stats, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!tok16(c, x) || !need16(w_gate) || !opt4(logit_bias) || !opt16(logits) ||
      !tok4(c, topk_idx) || !tok4(c, topk_w) || !opt4(counts) || !opt4(aux_loss) ||
      !opt4(routing_stats) || (c.noise != MOE_NOISE_NONE ? !tok4(c, noise) : !opt4(noise)))
    return MOE_ERR_INVALID_ARGUMENT;
  const Layout L = make_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.stage_end) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = at<int>(ws, L.flags);
  MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  if (c.T == 0) {
    if ((s = zero_async(counts, sizeof(int32_t) * c.E, st)) != MOE_OK) return s;
    if ((s = zero_async(routing_stats, sizeof(float) * MOE_ROUTING_STATS, st)) != MOE_OK) return s;
    return zero_async(aux_loss, sizeof(float), st);
  }
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  if ((s = run_router(c, L, ws, x, w_gate, logit_bias, noise, logits, topk_idx, topk_w, flags,
                      sms, st)) != MOE_OK)
    return s;
  if (counts || aux_loss || routing_stats)
    MOE_CUDA(launch_route_finalize(at<int32_t>(ws, L.hist), at<float>(ws, L.psum),
                                   static_cast<int>(L.nchunks), c.E, c.T, -1, counts, aux_loss,
                                   nullptr, nullptr, nullptr, nullptr, routing_stats, st));
  return MOE_OK;
}

MOE_EXPORT moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                   int32_t* offsets, int32_t* kept_counts, int32_t* slot_row,
                                   int32_t* row_token, int32_t* dropped, void* x_perm, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!tok16(c, x) || !tok4(c, topk_idx) || !need4(offsets) || !opt4(kept_counts) ||
      !tok4(c, slot_row) || !tok4(c, row_token) || !opt4(dropped) || !tok16(c, x_perm))
    return MOE_ERR_INVALID_ARGUMENT;
  const Layout L = make_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.stage_end) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = at<int>(ws, L.flags);
  MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  if (c.T == 0) {
    if ((s = zero_async(offsets, sizeof(int32_t) * (c.E + 1), st)) != MOE_OK) return s;
    if ((s = zero_async(kept_counts, sizeof(int32_t) * c.E, st)) != MOE_OK) return s;
    return zero_async(dropped, sizeof(int32_t), st);
  }
  int32_t* hist = at<int32_t>(ws, L.hist);
  int32_t* chunk_base = at<int32_t>(ws, L.chunk_base);
  MOE_CUDA(launch_dispatch_hist(topk_idx, c.T, c.E, c.k, hist, flags, st));
  MOE_CUDA(launch_route_finalize(hist, nullptr, static_cast<int>(L.nchunks), c.E, c.T,
                                 capacity_of(c), nullptr, nullptr, chunk_base, kept_counts, offsets,
                                 dropped, nullptr, st));
  MOE_CUDA(launch_dispatch_place(c.dtype, topk_idx, c.T, c.E, c.k, capacity_of(c), chunk_base,
                                 offsets, slot_row, row_token, x, x_perm, c.d, flags, st));
  return MOE_OK;
}

MOE_EXPORT moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm,
                                     const int32_t* offsets, const void* w1, const void* b1,
                                     const void* w2, const void* b2, void* h_buf, void* y_perm,
                                     void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!tok16(c, x_perm) || !need4(offsets) || !need16(w1) || !opt16(b1) || !need16(w2) ||
      !opt16(b2) || !tok16(c, h_buf) || !tok16(c, y_perm))
    return MOE_ERR_INVALID_ARGUMENT;
  const Layout L = make_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.stage_end) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = at<int>(ws, L.flags);
  MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  if (c.T == 0) return MOE_OK;
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  return run_expert_ffn(c, L, ws, x_perm, offsets, w1, b1, w2, b2, h_buf, y_perm, flags, sms, st);
}

MOE_EXPORT moe_status moe_combine(const moe_config* cfg, const void* y_perm,
                                  const int32_t* slot_row, const float* topk_w, void* y, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  const moe_config& c = *cfg;
  if (!tok16(c, y_perm) || !tok4(c, slot_row) || !tok4(c, topk_w) || !tok16(c, y))
    return MOE_ERR_INVALID_ARGUMENT;
  const Layout L = make_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.stage_end) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = at<int>(ws, L.flags);
  MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  if (c.T == 0) return MOE_OK;
  MOE_CUDA(launch_combine(c.dtype, y_perm, slot_row, topk_w, c.T, c.d, c.k, y, flags, st));
  return MOE_OK;
}

moe_status moe::forward_entry(const moe_config* cfg, const moe_forward_args* a, void* ws,
                              size_t ws_bytes, cudaStream_t st, EntryMode mode) {
  moe_status s = check_config(cfg);
  if (s != MOE_OK) return s;
  if (!a) return MOE_ERR_INVALID_ARGUMENT;
  const moe_config& c = *cfg;
  if (!tok16(c, a->x) || !need16(a->w_gate) || !opt4(a->logit_bias) || !need16(a->w1) ||
      !opt16(a->b1) || !need16(a->w2) || !opt16(a->b2) || !tok16(c, a->y) || !opt16(a->logits) ||
      !opt4(a->topk_idx) || !opt4(a->topk_w) || !opt4(a->counts) || !opt4(a->aux_loss) ||
      !opt4(a->offsets) || !opt4(a->kept_counts) || !opt4(a->slot_row) || !opt4(a->row_token) ||
      !opt4(a->dropped) || !opt4(a->routing_stats) || !opt16(a->x_perm) || !opt16(a->h_act) ||
      !opt16(a->y_perm) || !opt16(a->h_pre) ||
      (c.noise != MOE_NOISE_NONE ? !tok4(c, a->noise) : !opt4(a->noise)))
    return MOE_ERR_INVALID_ARGUMENT;
  const Layout L = make_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (mode == EntryMode::kValidate) return MOE_OK;
  int* flags = at<int>(ws, L.flags);
  if (mode == EntryMode::kRun) MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  int32_t* idx = a->topk_idx ? a->topk_idx : at<int32_t>(ws, L.idx);
  float* w = a->topk_w ? a->topk_w : at<float>(ws, L.w);
  int32_t* counts = a->counts ? a->counts : at<int32_t>(ws, L.counts);
  float* aux = a->aux_loss ? a->aux_loss : at<float>(ws, L.aux);
  int32_t* offsets = a->offsets ? a->offsets : at<int32_t>(ws, L.offsets);
  int32_t* kept = a->kept_counts ? a->kept_counts : at<int32_t>(ws, L.kept);
  int32_t* slot_row = a->slot_row ? a->slot_row : at<int32_t>(ws, L.slot_row);
  int32_t* row_token = a->row_token ? a->row_token : at<int32_t>(ws, L.row_token);
  int32_t* dropped = a->dropped ? a->dropped : at<int32_t>(ws, L.dropped);
  if (c.T == 0) {
    if ((s = zero_async(counts, sizeof(int32_t) * c.E, st)) != MOE_OK) return s;
    if ((s = zero_async(aux, sizeof(float), st)) != MOE_OK) return s;
    if ((s = zero_async(offsets, sizeof(int32_t) * (c.E + 1), st)) != MOE_OK) return s;
    if ((s = zero_async(kept, sizeof(int32_t) * c.E, st)) != MOE_OK) return s;
    if ((s = zero_async(a->routing_stats, sizeof(float) * MOE_ROUTING_STATS, st)) != MOE_OK)
      return s;
    return zero_async(dropped, sizeof(int32_t), st);
  }
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  int32_t* hist = at<int32_t>(ws, L.hist);
  int32_t* chunk_base = at<int32_t>(ws, L.chunk_base);
  float* psum = at<float>(ws, L.psum);
  void* x_perm = a->x_perm ? a->x_perm : at<void>(ws, L.x_perm);
  void* h_buf = a->h_act ? a->h_act : at<void>(ws, L.h_buf);
  void* y_perm = a->y_perm ? a->y_perm : at<void>(ws, L.y_perm);
  const int64_t C = capacity_of(c);

  {
    MOE_TRACE("moe_forward: route");
    if ((s = run_router(c, L, ws, a->x, a->w_gate, a->logit_bias, a->noise, a->logits, idx, w,
                        flags, sms, st)) != MOE_OK)
      return s;
    MOE_CUDA(launch_route_finalize(hist, psum, static_cast<int>(L.nchunks), c.E, c.T, C, counts,
                                   aux, chunk_base, kept, offsets, dropped, a->routing_stats, st));
  }
  // cfg->fused_gather: GEMM1 reads the token rows from x by row_token, and no expert-ordered
  // copy exists (unless the caller asked for one in x_perm).
  const bool gather = c.fused_gather && a->x_perm == nullptr;
  // A bf16 top-1 layer on the weights-as-M GEMMs: GEMM2 writes each kept token's output row
  // itself (the combine's one-slot arithmetic), GEMM1 zeroes the other tokens' rows, and
  // there is no combine pass -- unless the caller asked for Yp in y_perm.
  const bool fuse_combine = fused_top1_combine(c) && a->y_perm == nullptr;
  {
    MOE_TRACE("moe_forward: dispatch");
    MOE_CUDA(launch_dispatch_place(c.dtype, idx, c.T, c.E, c.k, C, chunk_base, offsets, slot_row,
                                   row_token, a->x, gather ? nullptr : x_perm, c.d, flags, st));
  }
  {
    MOE_TRACE("moe_forward: expert_ffn");
    const TopOneCombine top1{row_token, w, slot_row, a->y};
    if ((s = run_expert_ffn(c, L, ws, x_perm, offsets, a->w1, a->b1, a->w2, a->b2, h_buf, y_perm,
                            flags, sms, st, a->h_pre, gather ? row_token : nullptr,
                            gather ? a->x : nullptr, fuse_combine ? &top1 : nullptr)) != MOE_OK)
      return s;
  }
  if (!fuse_combine) {
    MOE_TRACE("moe_forward: combine");
    MOE_CUDA(launch_combine(c.dtype, y_perm, slot_row, w, c.T, c.d, c.k, a->y, flags, st));
  }
  return MOE_OK;
}

MOE_EXPORT moe_status moe_forward(const moe_config* cfg, const moe_forward_args* a, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
  return forward_entry(cfg, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream),
                       EntryMode::kRun);
}

MOE_EXPORT moe_status moe_device_error(const void* ws, moe_stream_t stream, int32_t* flags) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (flags) *flags = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

MOE_EXPORT moe_status moe_expert_choice_capacity(const moe_config* cfg, int64_t* capacity) {
  moe_status s = check_ec_config(cfg);
  if (s != MOE_OK) return s;
  if (!capacity) return MOE_ERR_INVALID_ARGUMENT;
  *capacity = ec_capacity_of(*cfg);
  return MOE_OK;
}

MOE_EXPORT moe_status moe_expert_choice_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_ec_config(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  *bytes = make_ec_layout(*cfg).total;
  return MOE_OK;
}

moe_status moe::ec_forward_entry(const moe_config* cfg, const moe_expert_choice_args* a,
                                 void* ws, size_t ws_bytes, cudaStream_t st, EntryMode mode) {
  moe_status s = check_ec_config(cfg);
  if (s != MOE_OK) return s;
  if (!a) return MOE_ERR_INVALID_ARGUMENT;
  const moe_config& c = *cfg;
  if (!tok16(c, a->x) || !need16(a->w_gate) || !opt4(a->logit_bias) || !need16(a->w1) ||
      !opt16(a->b1) || !need16(a->w2) || !opt16(a->b2) || !tok16(c, a->y) || !opt16(a->logits) ||
      !opt16(a->probs) || !opt4(a->sel_token) || !opt4(a->sel_w) || !opt4(a->token_experts) ||
      !opt4(a->unrouted))
    return MOE_ERR_INVALID_ARGUMENT;
  const EcLayout L = make_ec_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (mode == EntryMode::kValidate) return MOE_OK;
  int* flags = at<int>(ws, L.flags);
  if (mode == EntryMode::kRun) MOE_CUDA(cudaMemsetAsync(ws, 0, kFlagRegionBytes, st));
  if ((s = zero_async(a->unrouted, sizeof(int32_t), st)) != MOE_OK) return s;
  if (c.T == 0) return MOE_OK;
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const int64_t C = L.C;
  float* region = at<float>(ws, L.logits);
  float* probs_et = at<float>(ws, L.probs_et);
  int32_t* rowmap = at<int32_t>(ws, L.rowmap);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* sel_token = a->sel_token ? a->sel_token : at<int32_t>(ws, L.sel_token);
  float* sel_w = a->sel_w ? a->sel_w : at<float>(ws, L.sel_w);
  void* x_perm = at<void>(ws, L.x_perm);
  void* h_buf = at<void>(ws, L.h_buf);
  void* y_perm = at<void>(ws, L.y_perm);

  // EC1: router contraction and softmax (fp32: SIMT GEMM with the bias in its
  // epilogue; bf16: tensor-core K-split partials, added with the bias in EC1).
  GemmArgs g{};
  g.A = a->x;
  g.rows_alloc = c.T;
  g.B = a->w_gate;
  g.m_rows = c.T;
  g.G = 1;
  g.N = c.E;
  g.K = c.d;
  g.flags = flags;
  if (c.dtype == MOE_F32) {
    float* lg = a->logits ? a->logits : region;
    g.bias = a->logit_bias;
    g.out = lg;
    MOE_CUDA(launch_simt_gemm_f32(g, EPI_ROUTER_F32, sms, st));
    MOE_CUDA(launch_ec_softmax(lg, 1, 0, nullptr, nullptr, a->probs, probs_et, c.T, c.E, flags,
                               st));
  } else {
    g.out = region;
    g.ksplit = router_splits(c.T, c.E, c.d, sms < kMaxSmsForSizing ? sms : kMaxSmsForSizing);
    g.split_stride = c.T * c.E;
    MOE_CUDA(launch_tc_gemm_bf16(g, EPI_ROUTER_F32, sms, st));
    MOE_CUDA(launch_ec_softmax(region, g.ksplit, g.split_stride, a->logit_bias, a->logits,
                               a->probs, probs_et, c.T, c.E, flags, st));
  }
  // EC2: each expert's C tokens; then the rows in expert order and the expert FFN.
  MOE_CUDA(launch_ec_select(probs_et, c.T, c.E, C, sel_token, sel_w, rowmap, offsets, st));
  MOE_CUDA(launch_gather_rows(c.dtype, sel_token, offsets, c.E, a->x, x_perm, c.d, c.E * C, st));
  if ((s = run_expert_ffn_rows(c, c.E * C, C, x_perm, offsets, a->w1, a->b1, a->w2, a->b2, h_buf,
                               y_perm, flags, at<int>(ws, L.split_ctr),
                               at<float>(ws, L.split_part), sms, st)) != MOE_OK)
    return s;
  // EC3: per-token combine over the experts that took the token.
  MOE_CUDA(launch_ec_combine(c.dtype, y_perm, rowmap, probs_et, c.T, c.E, C, c.d, a->y,
                             a->token_experts, a->unrouted, st));
  return MOE_OK;
}

MOE_EXPORT moe_status moe_expert_choice_forward(const moe_config* cfg,
                                                const moe_expert_choice_args* a, void* ws,
                                                size_t ws_bytes, moe_stream_t stream) {
  return ec_forward_entry(cfg, a, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream),
                          EntryMode::kRun);
}

// ---------------------------------------------------------------- backward
namespace moe {
namespace {

struct BwdLayout {
  size_t flags, dyp, da, dxp, dxr, dw, dl, dl16, dwg, tail_a, tail_b, partial, total;
  int Epad;
};

BwdLayout make_bwd_layout(const moe_config& c) {
  BwdLayout L{};
  const int64_t T = c.T, E = c.E, k = c.k, rows = T * k;
  L.Epad = (c.E + 63) & ~63;  // dl16 rows span whole 64-column boxes
  int64_t pf = colsum_partial_floats(rows, c.E, c.d);
  pf = std::max<int64_t>(pf, colsum_partial_floats(rows, c.E, c.h));
  pf = std::max<int64_t>(pf, colsum_partial_floats(T, 1, c.E));
  size_t o = 0;
  L.flags = o; o += kAlign;
  L.dyp = o; o = align_up(o + rows * c.d * 2);
  L.da = o; o = align_up(o + rows * c.h * 2);
  L.dxp = o; o = align_up(o + rows * c.d * 2);
  L.dxr = o; o = align_up(o + T * c.d * 2);
  L.dw = o; o = align_up(o + T * k * 4);
  L.dl = o; o = align_up(o + T * E * 4);
  L.dl16 = o; o = align_up(o + T * L.Epad * 2);
  L.dwg = o; o = align_up(o + static_cast<int64_t>(L.Epad) * c.d * 4);
  const int64_t tail_bytes = E * 64 * std::max(c.d, c.h) * 2;
  L.tail_a = o; o = align_up(o + tail_bytes);
  L.tail_b = o; o = align_up(o + tail_bytes);
  L.partial = o; o = align_up(o + pf * 4);
  L.total = o;
  return L;
}

moe_status check_bwd_config(const moe_config* c) {
  moe_status s = check_config(c);
  if (s != MOE_OK) return s;
  if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->noise != MOE_NOISE_NONE) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

MOE_EXPORT moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
  moe_status s = check_bwd_config(cfg);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARGUMENT;
  *bytes = make_bwd_layout(*cfg).total;
  return MOE_OK;
}

MOE_EXPORT moe_status moe_backward(const moe_config* cfg, const moe_backward_args* a, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_bwd_config(cfg);
  if (s != MOE_OK) return s;
  if (!a) return MOE_ERR_INVALID_ARGUMENT;
  const moe_config& c = *cfg;
  if (!tok16(c, a->dy) || !tok16(c, a->x) || !need16(a->w_gate) || !need16(a->w1) ||
      !need16(a->w2) || !tok4(c, a->logits) || !tok4(c, a->topk_idx) || !tok4(c, a->topk_w) ||
      !need4(a->counts) || !need4(a->offsets) || !tok4(c, a->slot_row) || !tok16(c, a->x_perm) ||
      !tok16(c, a->h_pre) || !tok16(c, a->h_act) || !tok16(c, a->y_perm) || !tok16(c, a->dx) ||
      !opt4(a->dw_gate) || !opt4(a->dlogit_bias) || !opt16(a->dw1) || !opt4(a->db1) ||
      !opt16(a->dw2) || !opt4(a->db2) || !std::isfinite(a->d_aux))
    return MOE_ERR_INVALID_ARGUMENT;
  const BwdLayout L = make_bwd_layout(c);
  if (!ws || !al16(ws) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = at<int>(ws, L.flags);
  MOE_CUDA(cudaMemsetAsync(flags, 0, sizeof(int), st));
  const int64_t rows = c.T * c.k;
  if (c.T == 0) {
    // No tokens: every parameter gradient is zero.
    if ((s = zero_async(a->dw_gate, sizeof(float) * c.E * c.d, st)) != MOE_OK) return s;
    if ((s = zero_async(a->dlogit_bias, sizeof(float) * c.E, st)) != MOE_OK) return s;
    if ((s = zero_async(a->dw1, size_t{2} * c.E * c.h * c.d, st)) != MOE_OK) return s;
    if ((s = zero_async(a->db1, sizeof(float) * c.E * c.h, st)) != MOE_OK) return s;
    if ((s = zero_async(a->dw2, size_t{2} * c.E * c.d * c.h, st)) != MOE_OK) return s;
    return zero_async(a->db2, sizeof(float) * c.E * c.d, st);
  }
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  void* dyp = at<void>(ws, L.dyp);
  void* da = at<void>(ws, L.da);
  void* dxp = at<void>(ws, L.dxp);
  float* dw = at<float>(ws, L.dw);
  float* dl = at<float>(ws, L.dl);
  void* dl16 = at<void>(ws, L.dl16);
  float* partial = at<float>(ws, L.partial);

  // Combine and gate backward: dYp, dw, then dl (gate + balance loss).
  MOE_CUDA(launch_bwd_combine(a->dy, a->y_perm, a->slot_row, a->topk_w, c.T, c.d, c.k, dyp, dw, st));
  MOE_CUDA(launch_bwd_gate(a->logits, a->topk_idx, a->topk_w, dw, a->counts, a->d_aux, c.T, c.E,
                           L.Epad, c.k, dl, dl16, st));
  // Data gradients: dA = (dYp W2) * SiLU'(A), dXp = dA W1, dx = dl W_g + sum_j dXp.
  GemmArgs g{};
  g.A = dyp;
  g.rows_alloc = rows;
  g.B = a->w2;
  g.offsets = a->offsets;
  g.G = c.E;
  g.N = c.h;
  g.K = c.d;
  g.out = da;
  g.aux_in = a->h_pre;
  g.flags = flags;
  MOE_CUDA(launch_tc_bwd_rows(g, EPI_DSILU, sms, st));
  g.A = da;
  g.B = a->w1;
  g.N = c.d;
  g.K = c.h;
  g.out = dxp;
  g.aux_in = nullptr;
  MOE_CUDA(launch_tc_bwd_rows(g, EPI_PLAIN, sms, st));
  GemmArgs r{};
  r.A = dl16;
  r.m_rows = c.T;
  r.B = a->w_gate;
  r.G = 1;
  r.N = c.d;
  r.K = L.Epad;
  r.b_rows = c.E;
  r.out = at<void>(ws, L.dxr);
  r.flags = flags;
  MOE_CUDA(launch_tc_bwd_rows(r, EPI_PLAIN, sms, st));
  MOE_CUDA(launch_bwd_dx(at<void>(ws, L.dxr), dxp, a->slot_row, c.T, c.d, c.k, a->dx, st));
  // Weight gradients.
  WgradArgs wg{};
  wg.offsets = a->offsets;
  wg.rows_alloc = rows;
  wg.G = c.E;
  wg.flags = flags;
  wg.tailA = at<void>(ws, L.tail_a);
  wg.tailB = at<void>(ws, L.tail_b);
  if (a->dw2) {
    wg.A = dyp;
    wg.Mdim = c.d;
    wg.B = a->h_act;
    wg.Ndim = c.h;
    wg.out = a->dw2;
    MOE_CUDA(launch_pack_tails(wg.A, wg.Mdim, a->offsets, c.E, at<void>(ws, L.tail_a), st));
    MOE_CUDA(launch_pack_tails(wg.B, wg.Ndim, a->offsets, c.E, at<void>(ws, L.tail_b), st));
    MOE_CUDA(launch_tc_wgrad(wg, sms, st));
  }
  if (a->dw1) {
    wg.A = da;
    wg.Mdim = c.h;
    wg.B = a->x_perm;
    wg.Ndim = c.d;
    wg.out = a->dw1;
    MOE_CUDA(launch_pack_tails(wg.A, wg.Mdim, a->offsets, c.E, at<void>(ws, L.tail_a), st));
    MOE_CUDA(launch_pack_tails(wg.B, wg.Ndim, a->offsets, c.E, at<void>(ws, L.tail_b), st));
    MOE_CUDA(launch_tc_wgrad(wg, sms, st));
  }
  if (a->dw_gate) {
    WgradArgs rg{};
    rg.A = dl16;
    rg.Mdim = L.Epad;
    rg.B = a->x;
    rg.Ndim = c.d;
    rg.m_rows = c.T;
    rg.rows_alloc = c.T;
    rg.G = 1;
    rg.out = at<float>(ws, L.dwg);
    rg.out_f32 = true;
    rg.flags = flags;
    MOE_CUDA(launch_tc_wgrad(rg, sms, st));
    MOE_CUDA(cudaMemcpyAsync(a->dw_gate, at<float>(ws, L.dwg), sizeof(float) * c.E * c.d,
                             cudaMemcpyDeviceToDevice, st));
  }
  // Bias gradients: column sums per expert (fixed order).
  if (a->db2)
    MOE_CUDA(launch_colsum(dyp, false, c.d, a->offsets, 0, rows, c.E, partial, a->db2, st));
  if (a->db1)
    MOE_CUDA(launch_colsum(da, false, c.h, a->offsets, 0, rows, c.E, partial, a->db1, st));
  if (a->dlogit_bias)
    MOE_CUDA(launch_colsum(dl, true, c.E, nullptr, c.T, c.T, 1, partial, a->dlogit_bias, st));
  return MOE_OK;
}
