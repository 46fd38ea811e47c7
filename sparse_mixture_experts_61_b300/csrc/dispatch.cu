// Dispatch: capacity drop and expert-contiguous placement of the token rows.
//
// Assignments (t, j) are visited token by token, slot by slot; expert e hands out
// positions 0, 1, 2, ... in that order and an assignment is kept iff capacity is
// off or its position is below C ("Expert Choice routing and capacity-factor
// tuning": capacity = tokens / experts * capacity_factor, overflow tokens are
// rejected and pass through the residual).  Kept rows of expert e occupy
// [offsets[e], offsets[e+1]) in token order, the grouping by expert id that
// "Breaking the MoE trilemma" 3.3 describes.
//
// Parallel form of that sequential walk: tokens are cut into chunks of kChunk;
// a per-chunk expert histogram is scanned over chunks (route.cu, finalize) to
// give each chunk's first position per expert, and inside a chunk the position
// of an assignment is that base plus the number of earlier assignments of the
// chunk (in token-then-slot order) with the same expert.  The row copy into the
// expert-contiguous buffer is a separate grid-stride kernel (over the tokens for
// top-k routing, over the rows for expert choice), so that it uses the whole GPU
// whatever the number of chunks.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    dispatch_hist_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int E, int k,
                         int32_t* __restrict__ hist, int* flags) {
  pdl_enter();
  __shared__ int s_hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kChunk * k;
  const int64_t total = T * k;
  for (int a = threadIdx.x; a < kChunk * k; a += blockDim.x) {
    if (base + a >= total) break;
    const int e = topk_idx[base + a];
    if (e < 0 || e >= E)
      raise_flag(flags, MOE_DEVERR_BAD_INDEX);
    else
      atomicAdd(&s_hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[static_cast<int64_t>(blockIdx.x) * E + e] = s_hist[e];
}

__global__ void __launch_bounds__(kThreads)
    dispatch_place_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int E, int k, int64_t C,
                          const int32_t* __restrict__ chunk_base,
                          const int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
                          int32_t* __restrict__ row_token, int* flags) {
  pdl_enter();
  __shared__ int s_idx[kChunk * kMaxK];
  const int c = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(c) * kChunk;
  const int ntok = static_cast<int>(T - t0 < kChunk ? T - t0 : kChunk);
  const int npairs = ntok * k;
  const int64_t base = t0 * k;
  for (int a = threadIdx.x; a < npairs; a += blockDim.x) s_idx[a] = topk_idx[base + a];
  __syncthreads();

  for (int a = threadIdx.x; a < npairs; a += blockDim.x) {
    const int e = s_idx[a];
    int row = -1;
    if (e >= 0 && e < E) {
      int rank = 0;
      for (int b = 0; b < a; ++b) rank += (s_idx[b] == e);
      const int64_t pos = static_cast<int64_t>(chunk_base[static_cast<int64_t>(c) * E + e]) + rank;
      if (C < 0 || pos < C) row = offsets[e] + static_cast<int>(pos);
    } else {
      raise_flag(flags, MOE_DEVERR_BAD_INDEX);
    }
    slot_row[base + a] = row;
    if (row >= 0) row_token[row] = static_cast<int32_t>(t0 + a / k);
  }

  // Rows past the kept total carry no token.
  const int64_t M = offsets[E];
  for (int64_t r = M + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < T * k;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x)
    row_token[r] = -1;
}

// Row gather Xp[r, :] = x[row_token[r], :] for r < M = offsets[E]: one warp per row,
// grid-stride over rows, four independent 16-byte loads in flight per lane.  Used by
// expert-choice routing, whose selection lists each expert's rows by token; top-k
// dispatch copies token by token instead (scatter_rows_kernel below).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    gather_rows_kernel(const int32_t* __restrict__ row_token, const int32_t* __restrict__ offsets,
                       int E, const Tin* __restrict__ x, Tin* __restrict__ x_perm, int d) {
  pdl_enter();
  const int64_t M = offsets[E];
  const int nvec = d * static_cast<int>(sizeof(Tin)) / 16;
  const int lane = threadIdx.x & 31;
  const int64_t wpb = kThreads / 32;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); r < M;
       r += static_cast<int64_t>(gridDim.x) * wpb) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row_token[r]) * d);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + r * d);
    int v = lane;
    for (; v + 96 < nvec; v += 128) {
      const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                  e = __ldg(src + v + 96);
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = e;
    }
    for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

// Row scatter Xp[slot_row[t, j], :] = x[t, :] for every kept slot.  Work unit =
// (token, 128 consecutive 16-byte vectors), one warp per unit, grid-stride: each lane
// loads its 4 vectors once and stores them to each of the token's kept rows (the
// gather above reads a row once per slot: k times the reads when the rows do not
// stay in L2); a token with no kept slot costs one slot_row read.  Every row below M
// is some kept slot's, so all are written.
constexpr int kScatterVecs = 128;

__global__ void __launch_bounds__(kThreads)
    scatter_rows_kernel(const int32_t* __restrict__ slot_row, int64_t T, int k,
                        const uint4* __restrict__ x, uint4* __restrict__ x_perm, int nvec) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t wpb = kThreads / 32;
  const int chunks = (nvec + kScatterVecs - 1) / kScatterVecs;
  const int64_t units = T * chunks;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); u < units;
       u += static_cast<int64_t>(gridDim.x) * wpb) {
    const int64_t t = chunks == 1 ? u : u / chunks;
    const int v0 = static_cast<int>(u - t * chunks) * kScatterVecs;
    const int my_row = lane < k ? slot_row[t * k + lane] : -1;
    // A token whose every slot was dropped has no row to fill: its x row is not read.
    if (!__any_sync(0xffffffffu, my_row >= 0)) continue;
    int64_t dst[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      const int r = __shfl_sync(0xffffffffu, my_row, j);
      dst[j] = (j < k && r >= 0) ? static_cast<int64_t>(r) * nvec : -1;
    }
    const uint4* src = x + t * nvec;
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int v = v0 + lane + 32 * i;
      if (v < nvec) q[i] = __ldg(src + v);
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (dst[j] < 0) continue;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int v = v0 + lane + 32 * i;
        if (v < nvec) x_perm[dst[j] + v] = q[i];
      }
    }
  }
}

}  // namespace

cudaError_t launch_dispatch_hist(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* hist,
                                 int* flags, cudaStream_t stream) {
  const int64_t nchunks = (T + kChunk - 1) / kChunk;
  if (nchunks == 0) return cudaSuccess;
  launch_pdl(dispatch_hist_kernel, static_cast<unsigned>(nchunks), kThreads, 0, stream, topk_idx, T, E, k,
                                                                               hist, flags);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_place(int dtype, const int32_t* topk_idx, int64_t T, int E, int k,
                                  int64_t C, const int32_t* chunk_base, const int32_t* offsets,
                                  int32_t* slot_row, int32_t* row_token, const void* x,
                                  void* x_perm, int d, int* flags, cudaStream_t stream) {
  const int64_t nchunks = (T + kChunk - 1) / kChunk;
  if (nchunks == 0) return cudaSuccess;
  launch_pdl(dispatch_place_kernel, static_cast<unsigned>(nchunks), kThreads, 0, stream, 
      topk_idx, T, E, k, C, chunk_base, offsets, slot_row, row_token, flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || x_perm == nullptr) return e;
  // Xp by scatter from the tokens (each x row read once).
  const int nvec = d * (dtype == MOE_F32 ? 4 : 2) / 16;
  const int64_t units = T * ((nvec + kScatterVecs - 1) / kScatterVecs);
  const unsigned grid = static_cast<unsigned>(
      std::min<int64_t>((units + kThreads / 32 - 1) / (kThreads / 32), 4096));
  launch_pdl(scatter_rows_kernel, grid, kThreads, 0, stream, slot_row, T, k,
             static_cast<const uint4*>(x), static_cast<uint4*>(x_perm), nvec);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(int dtype, const int32_t* row_token, const int32_t* offsets, int E,
                               const void* x, void* x_perm, int d, int64_t rows,
                               cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  // Enough warps for every possible row, capped; the kernel strides over the rest.
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>((rows + kThreads / 32 - 1) / (kThreads / 32), 4096));
  if (dtype == MOE_F32)
    launch_pdl(gather_rows_kernel<float>, grid, kThreads, 0, stream, 
        row_token, offsets, E, static_cast<const float*>(x), static_cast<float*>(x_perm), d);
  else
    launch_pdl(gather_rows_kernel<__nv_bfloat16>, grid, kThreads, 0, stream, 
        row_token, offsets, E, static_cast<const __nv_bfloat16*>(x),
        static_cast<__nv_bfloat16*>(x_perm), d);
  return cudaGetLastError();
}

}  // namespace moe
