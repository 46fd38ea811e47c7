// moe_forward_host (include/moe.h): the layer over a sequence of batches whose x
// and y live in host memory, with the copies overlapped with the layer.
//
// Three streams: `in` copies batch i's x into device slot i%2, the caller's stream
// runs the layer on that slot (the same enqueue as moe_forward /
// moe_expert_choice_forward), and `out` copies the slot's y (and the balance
// statistic) back.  Events carry the three hand-offs of each slot:
//   x_ready[s]  in  -> layer   x of the batch is in slot s
//   done[s]     layer -> in, out   the layer finished: slot s's x may be
//               overwritten, its y may be read
//   y_free[s]   out -> layer   slot s's y (and statistic) reached the host
// A slot is reused two batches later, after both of those waits.  No host
// synchronisation: everything is enqueued up front.
//
// A single batch, or batches of less than kSmallBatchBytes of x, run copy in, layer,
// copy out on the caller's stream alone: one batch has nothing to overlap with, and
// small copies are latency-bound, so the cross-stream hand-offs cost more host time
// per batch than the overlap hides (measured on a 256 x 128 fp32 layer: 104 us per
// batch pipelined, host-bound, against 75 us in order on one stream).

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "entry.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t kAlign = 256;
constexpr size_t kSmallBatchBytes = 256 << 10;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

struct HostLayout {
  size_t fwd, xs[2], ys[2], aux, total;
};

moe_status host_layout(const moe_config* cfg, int32_t routing, HostLayout* L) {
  size_t fwd = 0;
  moe_status s = routing == MOE_ROUTING_TOPK ? moe_workspace_size(cfg, &fwd)
                                             : moe_expert_choice_workspace_size(cfg, &fwd);
  if (s != MOE_OK) return s;
  const size_t batch = static_cast<size_t>(cfg->T) * cfg->d * (cfg->dtype == MOE_F32 ? 4 : 2);
  size_t o = align_up(fwd);
  L->fwd = fwd;
  for (int i = 0; i < 2; ++i) { L->xs[i] = o; o = align_up(o + batch); }
  for (int i = 0; i < 2; ++i) { L->ys[i] = o; o = align_up(o + batch); }
  L->aux = o; o = align_up(o + 2 * sizeof(float));
  L->total = o;
  return MOE_OK;
}

// Streams and events of one call, released on every return path.  Destroying a
// stream or event with work still pending is allowed; CUDA frees it afterwards.
struct Resources {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t x_ready[2] = {}, done[2] = {}, y_free[2] = {};

  cudaError_t create() {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    cudaEvent_t* all[] = {&start, &end, &x_ready[0], &x_ready[1], &done[0], &done[1],
                          &y_free[0], &y_free[1]};
    for (cudaEvent_t* ev : all)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    return cudaSuccess;
  }
  ~Resources() {
    cudaEvent_t all[] = {start, end, x_ready[0], x_ready[1], done[0], done[1], y_free[0],
                         y_free[1]};
    for (cudaEvent_t ev : all)
      if (ev) cudaEventDestroy(ev);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
};

#define HP_CUDA(call)                               \
  do {                                              \
    if ((call) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// The layer for one batch: x and y in workspace slots, weights shared.  `mode`
// kValidate checks the arguments without enqueueing anything.
moe_status run_layer(const moe_config* cfg, int32_t routing, const moe_weights& w, void* ws,
                     const HostLayout& L, int slot, cudaStream_t st, moe::EntryMode mode) {
  char* base = static_cast<char*>(ws);
  void* x = base + L.xs[slot];
  void* y = base + L.ys[slot];
  if (routing == MOE_ROUTING_TOPK) {
    moe_forward_args a{};
    a.x = x;
    a.w_gate = w.w_gate;
    a.logit_bias = w.logit_bias;
    a.w1 = w.w1;
    a.b1 = w.b1;
    a.w2 = w.w2;
    a.b2 = w.b2;
    a.y = y;
    a.aux_loss = reinterpret_cast<float*>(base + L.aux) + slot;
    return moe::forward_entry(cfg, &a, ws, L.fwd, st, mode);
  }
  moe_expert_choice_args a{};
  a.x = x;
  a.w_gate = w.w_gate;
  a.logit_bias = w.logit_bias;
  a.w1 = w.w1;
  a.b1 = w.b1;
  a.w2 = w.w2;
  a.b2 = w.b2;
  a.y = y;
  return moe::ec_forward_entry(cfg, &a, ws, L.fwd, st, mode);
}

}  // namespace

MOE_EXPORT moe_status moe_forward_host_workspace_size(const moe_config* cfg, int32_t routing,
                                                      size_t* bytes) {
  if (!cfg || !bytes || (routing != MOE_ROUTING_TOPK && routing != MOE_ROUTING_EXPERT_CHOICE))
    return MOE_ERR_INVALID_ARGUMENT;
  HostLayout L;
  moe_status s = host_layout(cfg, routing, &L);
  if (s != MOE_OK) return s;
  *bytes = L.total;
  return MOE_OK;
}

MOE_EXPORT moe_status moe_forward_host(const moe_config* cfg, int32_t routing,
                                       const moe_weights* weights,
                                       const moe_host_batches* b, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
  if (!cfg || !weights || !b || (routing != MOE_ROUTING_TOPK &&
                                 routing != MOE_ROUTING_EXPERT_CHOICE))
    return MOE_ERR_INVALID_ARGUMENT;
  HostLayout L;
  moe_status s = host_layout(cfg, routing, &L);
  if (s != MOE_OK) return s;
  if (cfg->noise != MOE_NOISE_NONE) return MOE_ERR_UNSUPPORTED;
  if (b->n < 1 || !b->x || !b->y) return MOE_ERR_INVALID_ARGUMENT;
  if (routing == MOE_ROUTING_EXPERT_CHOICE && b->aux_loss) return MOE_ERR_INVALID_ARGUMENT;
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 16 != 0 || ws_bytes < L.total)
    return MOE_ERR_WORKSPACE;
  const int64_t T = cfg->T;
  if (T > 0)
    for (int64_t i = 0; i < b->n; ++i)
      if (!b->x[i] || !b->y[i]) return MOE_ERR_INVALID_ARGUMENT;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The layer's own checks of the weights (the slots are valid by construction).
  if ((s = run_layer(cfg, routing, *weights, ws, L, 0, st, moe::EntryMode::kValidate)) != MOE_OK)
    return s;

  // The flag word and the expert GEMMs' split counters, once: the counters are left
  // zeroed by every layer that completes.
  HP_CUDA(cudaMemsetAsync(ws, 0, moe::kFlagRegionBytes, st));
  if (T == 0) {
    if (b->aux_loss)
      for (int64_t i = 0; i < b->n; ++i) b->aux_loss[i] = 0.f;
    return MOE_OK;
  }
  const size_t bytes = static_cast<size_t>(T) * cfg->d * (cfg->dtype == MOE_F32 ? 4 : 2);
  char* base = static_cast<char*>(ws);
  const float* aux_dev = reinterpret_cast<const float*>(base + L.aux);

  if (b->n == 1 || bytes < kSmallBatchBytes) {
    for (int64_t i = 0; i < b->n; ++i) {
      HP_CUDA(cudaMemcpyAsync(base + L.xs[0], b->x[i], bytes, cudaMemcpyHostToDevice, st));
      if ((s = run_layer(cfg, routing, *weights, ws, L, 0, st,
                         moe::EntryMode::kRunKeepFlags)) != MOE_OK)
        return s;
      HP_CUDA(cudaMemcpyAsync(b->y[i], base + L.ys[0], bytes, cudaMemcpyDeviceToHost, st));
      if (b->aux_loss)
        HP_CUDA(cudaMemcpyAsync(b->aux_loss + i, aux_dev, sizeof(float),
                                cudaMemcpyDeviceToHost, st));
    }
    return MOE_OK;
  }

  Resources r;
  HP_CUDA(r.create());
  HP_CUDA(cudaEventRecord(r.start, st));
  HP_CUDA(cudaStreamWaitEvent(r.in, r.start, 0));
  HP_CUDA(cudaStreamWaitEvent(r.out, r.start, 0));
  for (int64_t i = 0; i < b->n; ++i) {
    const int slot = static_cast<int>(i & 1);
    if (i >= 2) HP_CUDA(cudaStreamWaitEvent(r.in, r.done[slot], 0));
    HP_CUDA(cudaMemcpyAsync(base + L.xs[slot], b->x[i], bytes, cudaMemcpyHostToDevice, r.in));
    HP_CUDA(cudaEventRecord(r.x_ready[slot], r.in));

    HP_CUDA(cudaStreamWaitEvent(st, r.x_ready[slot], 0));
    if (i >= 2) HP_CUDA(cudaStreamWaitEvent(st, r.y_free[slot], 0));
    if ((s = run_layer(cfg, routing, *weights, ws, L, slot, st,
                       moe::EntryMode::kRunKeepFlags)) != MOE_OK)
      return s;
    HP_CUDA(cudaEventRecord(r.done[slot], st));

    HP_CUDA(cudaStreamWaitEvent(r.out, r.done[slot], 0));
    HP_CUDA(cudaMemcpyAsync(b->y[i], base + L.ys[slot], bytes, cudaMemcpyDeviceToHost, r.out));
    if (b->aux_loss)
      HP_CUDA(cudaMemcpyAsync(b->aux_loss + i, aux_dev + slot, sizeof(float),
                              cudaMemcpyDeviceToHost, r.out));
    HP_CUDA(cudaEventRecord(r.y_free[slot], r.out));
  }
  HP_CUDA(cudaEventRecord(r.end, r.out));
  HP_CUDA(cudaStreamWaitEvent(st, r.end, 0));
  return MOE_OK;
}
