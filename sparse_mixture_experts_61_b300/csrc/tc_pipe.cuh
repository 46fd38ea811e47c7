// The warp-specialised tcgen05 GEMM pipeline shared by the forward GEMMs (gemm_tc.cu)
// and the backward GEMMs (gemm_bwd.cu): shared-memory stage ring, barrier set-up and
// TMEM allocation, the per-group tile prefix, the TMA producer and MMA issuer loops
// with bounded waits, teardown, and the host-side tensor-map and launch helpers.
// Included by exactly those translation units; everything has internal linkage.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int TC_BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int TC_THREADS = 192;
// The row-tile expert GEMM runs two epilogue warps per TMEM lane quadrant (each takes
// half of the tile's columns): 64 + 256 threads.
constexpr int ROWS_EPI_WARPS = 8;
constexpr int ROWS_THREADS = 64 + 32 * ROWS_EPI_WARPS;
constexpr int TILE_M = 128;

template <int A_BYTES, int B_BYTES, int STAGES>
struct PipeSmem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int pref[kMaxExperts + 1];  // per-group prefix of tile units
};

// Wait used only while unwinding: bounded by time, ignores the abort flag.
__device__ __forceinline__ void mbar_wait_unwind(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return;
}

// Set-up that touches no global memory, so it runs before the kernel waits for its
// predecessor in the stream: barrier initialisation, tensor-map prefetch and TMEM
// allocation.  All threads call.
template <class Smem, int STAGES>
__device__ __forceinline__ void pipe_setup(Smem& S, uint32_t tmem_cols, const void* tmA,
                                           const void* tmB, uint32_t epi_threads = 128) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.tfull[i]), 1);
      mbar_init(smem_u32(&S.tempty[i]), epi_threads);
    }
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(tmA);
    tma_prefetch_desc(tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), tmem_cols);
    tmem_relinquish();
  }
}

// After the grid-dependency wait: the per-group prefix of ceil(rows_g / unit) (rows_g
// from the offsets, or m_rows for a single dense group), then the CTA-wide barrier that
// publishes it together with the set-up.  All threads call.  Every offset is loaded
// before any is used, so the prefix costs one memory latency, not one per 32 groups.
template <class Smem>
__device__ __forceinline__ void pipe_prefix(Smem& S, const GemmArgs& p, int G, int unit) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    constexpr int kChunks = kMaxExperts / 32;
    int units[kChunks];
    if (p.offsets) {
      int lo[kChunks], hi[kChunks];
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int g = i * 32 + lane;
        lo[i] = g < G ? p.offsets[g] : 0;
        hi[i] = g < G ? p.offsets[g + 1] : 0;
      }
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int64_t rows = static_cast<int64_t>(hi[i]) - lo[i];
        units[i] = rows > 0 ? static_cast<int>((rows + unit - 1) / unit) : 0;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kChunks; ++i)
        units[i] = (i == 0 && lane == 0 && G >= 1 && p.m_rows > 0)
                       ? static_cast<int>((p.m_rows + unit - 1) / unit)
                       : 0;
    }
    int carry = 0;
    if (lane == 0) S.pref[0] = 0;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      int v = units[i];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      const int g = i * 32 + lane;
      if (g < G) S.pref[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// The whole prologue: set-up, grid-dependency wait, prefix.  All threads call.
template <class Smem, int STAGES>
__device__ __forceinline__ void pipe_prologue(Smem& S, uint32_t tmem_cols, const GemmArgs& p,
                                              int G, int unit, const void* tmA,
                                              const void* tmB, uint32_t epi_threads = 128) {
  pipe_setup<Smem, STAGES>(S, tmem_cols, tmA, tmB, epi_threads);
  pdl_enter();
  pipe_prefix(S, p, G, unit);
}

// Group of a tile: the g with pref[g]*per <= tile < pref[g+1]*per.
__device__ __forceinline__ int find_group(const int* pref, int G, int per, int tile) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] * per <= tile) lo = mid; else hi = mid;
  }
  return lo;
}

// Warp 0, lane 0, over tiles first, first + step, ...  decode(tile) -> coordinates
// with the stage's byte count in .bytes and the tile's k-blocks [.kb0, .kb1);
// load(coords, kb, smem_a, smem_b, bar).
template <int STAGES, class Smem, class Decode, class Load>
__device__ __forceinline__ void run_producer(Smem& S, int first, int step, int total,
                                             Decode decode, Load load, volatile int* abort,
                                             int* flags) {
  int s = 0;
  uint32_t ph = 0, issued = 0, issued_par = 0;
  bool ok = true;
  for (int tile = first; ok && tile < total; tile += step) {
    const auto c = decode(tile);
    for (int kb = c.kb0; kb < c.kb1; ++kb) {
      if (!mbar_wait_bounded(smem_u32(&S.empty[s]), ph ^ 1u, abort, flags)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&S.full[s]);
      mbar_arrive_expect_tx(fb, c.bytes);
      load(c, kb, smem_u32(S.a[s]), smem_u32(S.b[s]), fb);
      issued |= 1u << s;
      issued_par = (issued_par & ~(1u << s)) | (ph << s);
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  if (!ok) {
    // Unwinding: let this CTA's copies in flight land before it exits.
    for (int q = 0; q < STAGES; ++q)
      if ((issued >> q) & 1u) mbar_wait_unwind(smem_u32(&S.full[q]), (issued_par >> q) & 1u);
  }
}

// run_producer for the whole warp 0: before each tile's first k-block every lane calls
// prepare(coords, lane) (work spread over the warp, such as fetching a tile's row
// indices into shared memory, finished before lane 0 issues that tile's copies); the
// ring waits and load(coords, kb, smem_a, smem_b, bar) are lane 0's.
template <int STAGES, class Smem, class Decode, class Prepare, class Load>
__device__ __forceinline__ void run_producer_warp(Smem& S, int first, int step, int total,
                                                  Decode decode, Prepare prepare, Load load,
                                                  volatile int* abort, int* flags) {
  const int lane = threadIdx.x & 31;
  int s = 0;
  uint32_t ph = 0, issued = 0, issued_par = 0;
  bool ok = true;
  for (int tile = first; ok && tile < total; tile += step) {
    const auto c = decode(tile);
    __syncwarp();  // lane 0 has issued the previous tile's copies
    prepare(c, lane);
    __syncwarp();
    for (int kb = c.kb0; kb < c.kb1; ++kb) {
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(smem_u32(&S.empty[s]), ph ^ 1u, abort, flags);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        const uint32_t fb = smem_u32(&S.full[s]);
        mbar_arrive_expect_tx(fb, c.bytes);
        load(c, kb, smem_u32(S.a[s]), smem_u32(S.b[s]), fb);
        issued |= 1u << s;
        issued_par = (issued_par & ~(1u << s)) | (ph << s);
      }
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  if (!ok && lane == 0) {
    // Unwinding: let this CTA's copies in flight land before it exits.
    for (int q = 0; q < STAGES; ++q)
      if ((issued >> q) & 1u) mbar_wait_unwind(smem_u32(&S.full[q]), (issued_par >> q) & 1u);
  }
}

// Warp 1, lane 0.  decode(tile) -> coordinates with the k-block range [.kb0, .kb1);
// idesc_of(coords) -> instruction descriptor of the tile's MMAs.  B_MN: the B stage
// holds MN-major boxes of [64 K rows x 64 N] (8 KB apart) instead of one K-major box.
template <int STAGES, int ACC_COLS, bool B_MN = false, class Smem, class Decode, class Idesc>
__device__ __forceinline__ void run_mma(Smem& S, int first, int step, int total,
                                        uint32_t tmem_base, Decode decode, Idesc idesc_of,
                                        volatile int* abort, int* flags) {
  int s = 0, acc = 0;
  uint32_t ph = 0, aph = 0;
  bool ok = true, issued_any = false;
  for (int tile = first; ok && tile < total; tile += step) {
    const auto c = decode(tile);
    const uint32_t idesc = idesc_of(c);
    if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), aph ^ 1u, abort, flags)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
    for (int kb = c.kb0; kb < c.kb1; ++kb) {
      if (!mbar_wait_bounded(smem_u32(&S.full[s]), ph, abort, flags)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(S.a[s]), b0 = smem_u32(S.b[s]);
#pragma unroll
      for (int kk = 0; kk < TC_BK / 16; ++kk)
        tc_mma_bf16(d_tmem, sw128_kmajor_desc(a0 + kk * 32),
                    B_MN ? sw128_mnmajor_desc(b0 + kk * 2048, 8192)
                         : sw128_kmajor_desc(b0 + kk * 32),
                    idesc, (kb != c.kb0 || kk != 0) ? 1u : 0u);
      issued_any = true;
      tc_commit(smem_u32(&S.empty[s]));
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (!ok) break;
    tc_commit(smem_u32(&S.tfull[acc]));
    acc ^= 1;
    if (acc == 0) aph ^= 1u;
  }
  // Unwinding: every MMA issued by this thread completes before TMEM is released.
  // (On the normal path the epilogue has already waited for all of them.)
  if (!ok && issued_any) {
    tc_commit(smem_u32(&S.drain));
    mbar_wait_unwind(smem_u32(&S.drain), 0);
  }
}

template <class Smem>
__device__ __forceinline__ void pipe_teardown(Smem& S, uint32_t tmem_cols) {
  tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(S.tmem_base, tmem_cols);
  }
}

template <class Smem>
__device__ __forceinline__ Smem& smem_aligned() {
  extern __shared__ uint8_t smem_raw[];
  return *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                  ~static_cast<uintptr_t>(1023));
}

// SiLU(x) = x / (1 + e^-x) with the fast division intrinsic (within 2 ulp in fp32, far below
// the bf16 rounding of the result; 0 when e^-x overflows, x when it underflows).  The
// IEEE-rounded division took four times as long in the epilogue.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.f + __expf(-x)); }

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                        strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows, K] bf16 matrix, box [box_rows x box_cols].
bool rows_map(CUtensorMap* m, const void* base, int64_t rows, int K, int box_rows,
              int box_cols = TC_BK) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  return encode_bf16_map(m, base, 2, dims, str, box);
}

// 3-D map over stacked [G, N, K] bf16 weights, box [box_rows x 64] of one group.
bool stacked_map(CUtensorMap* m, const void* base, int G, int N, int K, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(G)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(N) * K * 2};
  const cuuint32_t box[3] = {TC_BK, static_cast<cuuint32_t>(box_rows), 1};
  return encode_bf16_map(m, base, 3, dims, str, box);
}

template <class Kern>
cudaError_t launch_pipe(Kern kern, size_t smem, int grid, const CUtensorMap& a,
                        const CUtensorMap& b, const GemmArgs& args, cudaStream_t stream,
                        int threads = TC_THREADS) {
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  launch_pdl(kern, grid, threads, smem, stream, a, b, args);
  return cudaGetLastError();
}

}  // namespace
}  // namespace moe
