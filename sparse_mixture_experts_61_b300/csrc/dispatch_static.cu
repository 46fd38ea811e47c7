// moe_dispatch_static: the dispatch stage with its scratch held by the library.
//
// moe_dispatch needs a caller workspace for two per-chunk tables (the expert
// histogram of each 64-token chunk and each chunk's first position per expert)
// and the device flag word.  Some callers cannot provide one: code running under
// a host framework that owns all device memory and forbids allocating once it is
// serving, or a plugin whose call site has no allocator at all.  This entry point
// keeps those tables in one file-scope device array instead, so the caller passes
// only inputs and outputs.  It launches exactly the kernels moe_dispatch launches.
//
// The array is sized for ceil(T/64) * E <= MOE_DISPATCH_STATIC_MAX_CELLS table
// cells; it lives in every GPU that loads the library until the process exits.
// Every call shares it and it keeps the last call's contents: both tables are fully
// rewritten by each call before they are read, and the flag word is cleared at the
// start of each call.  Calls whose work overlaps on the GPU (different streams, or
// different host threads) race on the array and must be serialised by the caller.
//
// Its device address is looked up (cudaGetSymbolAddress) by the first call made in a
// given CUDA context -- the device's primary context, for runtime-API callers -- and
// kept for as long as that context is current: a call made in a new context (after
// cudaDeviceReset, say) looks it up again.  Make the first call in a context before any
// stream capture begins.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "entry.h"
#include "kernels.h"

namespace {

constexpr int64_t kCells = MOE_DISPATCH_STATIC_MAX_CELLS;
constexpr int64_t kFlagInts = 64;  // flag word, padded to 256 bytes

// [flag word | per-chunk histogram (kCells) | per-chunk position bases (kCells)]
static __device__ __align__(256) int32_t g_dispatch_scratch[kFlagInts + 2 * kCells];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// Per device: the address and the unique id of the context it was looked up in.
int32_t* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Unique id of the calling thread's current context (ids are never reused within a
// process), from the driver entry points cuCtxGetCurrent and cuCtxGetId.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
         get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_dispatch_scratch in the current context (looked up once per
// context).
moe_status scratch_address(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!have_ctx || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    // The lookup also makes the device's primary context current when no context is.
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    if (!current_context_id(&ctx)) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
// Required unless the batch is empty; always aligned when given.
bool token_buf(const moe_config& c, const void* p, uintptr_t a) {
  return (p == nullptr) ? c.T == 0 : aligned(p, a);
}

}  // namespace

extern "C" __attribute__((visibility("default"))) moe_status moe_dispatch_static(
    const moe_config* cfg, const void* x, const int32_t* topk_idx, int32_t* offsets,
    int32_t* kept_counts, int32_t* slot_row, int32_t* row_token, int32_t* dropped, void* x_perm,
    int32_t* device_flags, moe_stream_t stream) {
  // The same validation as moe_dispatch.
  const moe_status valid = moe::check_config(cfg);
  if (valid != MOE_OK) return valid;
  const moe_config& c = *cfg;
  const int64_t nchunks = (c.T + moe::kChunk - 1) / moe::kChunk;
  if (nchunks * c.E > kCells) return MOE_ERR_UNSUPPORTED;  // beyond the static scratch
  if (!token_buf(c, x, 16) || !token_buf(c, topk_idx, 4) || !offsets || !aligned(offsets, 4) ||
      !aligned(kept_counts, 4) || !token_buf(c, slot_row, 4) || !token_buf(c, row_token, 4) ||
      !aligned(dropped, 4) || !token_buf(c, x_perm, 16) || !aligned(device_flags, 4))
    return MOE_ERR_INVALID_ARGUMENT;

  int32_t* scratch = nullptr;
  moe_status s = scratch_address(&scratch);
  if (s != MOE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* flags = device_flags ? device_flags : scratch;
  if (cudaMemsetAsync(flags, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  if (c.T == 0) {
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (c.E + 1), st) != cudaSuccess ||
        (kept_counts && cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * c.E, st) != cudaSuccess) ||
        (dropped && cudaMemsetAsync(dropped, 0, sizeof(int32_t), st) != cudaSuccess))
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const int64_t C = (c.capacity_factor > 0.0)
                        ? static_cast<int64_t>(std::ceil(static_cast<double>(c.T) *
                                                         c.capacity_factor /
                                                         static_cast<double>(c.E)))
                        : -1;
  int32_t* hist = scratch + kFlagInts;
  int32_t* chunk_base = hist + kCells;
  if (moe::launch_dispatch_hist(topk_idx, c.T, c.E, c.k, hist, flags, st) != cudaSuccess ||
      moe::launch_route_finalize(hist, nullptr, static_cast<int>(nchunks), c.E, c.T, C, nullptr,
                                 nullptr, chunk_base, kept_counts, offsets, dropped, nullptr,
                                 st) != cudaSuccess ||
      moe::launch_dispatch_place(c.dtype, topk_idx, c.T, c.E, c.k, C, chunk_base, offsets,
                                 slot_row, row_token, x, x_perm, c.d, flags, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
