// Ragged grouped GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   out[r, n] = act( sum_c A[r, c] * B[g][n][c] + bias[g][n] ),  r in group g's rows
//
// It serves the two expert GEMMs of the expert FFN (Expert.forward =
// w2(silu(w1(x))) with nn.Linear biases, "MoE mixture-of-experts routing
// mechanism: principles and sparse activation") -- bias + SiLU fused into the
// first GEMM's epilogue, bias into the second's -- and, with one group and an fp32
// epilogue, the router contraction x . W_g of the gating formula.  Its job is the
// one "Breaking the MoE trilemma" 3.3 gives _grouped_ffn: every expert's token
// group multiplied in one kernel, with no per-expert launch.
//
// Design (one CTA per SM, persistent):
//  * 128 x BN output tiles; a tile never straddles two groups.  Group g owns
//    ceil(rows_g / 128) row tiles.  Tiles are ordered (group, column block, row
//    block) so CTAs running side by side share the same weight tile through L2.
//    The tile list is derived on the device from the group offsets: the number
//    of kept rows never goes to the host.
//  * warp 0: TMA producer.  A tile [128 x 64] from a 2-D tensor map over the row
//    buffer; B tile [BN x 64] from a 3-D map [G, N, K] addressed by group, so
//    no per-group descriptors.  Rows past the buffer are zero-filled by TMA; rows
//    past the group's end are computed and discarded by the epilogue.
//  * warp 1: allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16) from one
//    thread into one of two TMEM accumulators, committing each smem stage back to
//    the producer and each finished accumulator to the epilogue.
//  * warps 2-5: epilogue.  tcgen05.ld drains the accumulator 32 columns at a time
//    (thread = row), adds the bias, applies the activation, rounds and stores.
//    Two accumulators let the epilogue of one tile overlap the next main loop.
//  * Every wait is bounded (common.cuh); on a timeout the CTA records
//    MOE_DEVERR_TIMEOUT, drains its own TMA copies and MMAs, frees TMEM, returns.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
constexpr int TC_THREADS = 192;

template <int BN, int STAGES>
struct TcSmem {
  uint8_t a[STAGES][TC_BM * TC_BK * 2];
  uint8_t b[STAGES][BN * TC_BK * 2];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int mpref[kMaxExperts + 1];
};

// Wait used only while unwinding: bounded by time, ignores the abort flag.
__device__ __forceinline__ void mbar_wait_unwind(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) return;
}

struct TileCoord {
  int g;
  int64_t row0, row_end;
  int n0;
};

__device__ __forceinline__ TileCoord decode_tile(int tile, const int* mpref, int G, int NB,
                                                 const GemmArgs& p, int bn) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mpref[mid] * NB <= tile) lo = mid; else hi = mid;
  }
  TileCoord c;
  c.g = lo;
  const int mt_g = mpref[lo + 1] - mpref[lo];
  const int local = tile - mpref[lo] * NB;
  const int nb = local / mt_g, mt = local % mt_g;
  const int64_t base = p.offsets ? p.offsets[lo] : 0;
  c.row0 = base + static_cast<int64_t>(mt) * TC_BM;
  c.row_end = p.offsets ? p.offsets[lo + 1] : p.m_rows;
  c.n0 = nb * bn;
  return c;
}

template <int EPI, int CH>
__device__ __forceinline__ void epilogue_store(const GemmArgs& p, int g, int64_t row, int n_start,
                                               const float (&v)[CH]) {
  if constexpr (EPI == EPI_ROUTER_F32) {
    float* out = static_cast<float*>(p.out) + row * p.N;
    const float* bias = static_cast<const float*>(p.bias);
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int n = n_start + i;
      if (n < p.N) out[n] = v[i] + (bias ? bias[n] : 0.f);
    }
  } else {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + row * p.N + n_start;
    const __nv_bfloat16* bias =
        p.bias ? static_cast<const __nv_bfloat16*>(p.bias) + static_cast<int64_t>(g) * p.N + n_start
               : nullptr;
    if (n_start + CH <= p.N) {
#pragma unroll
      for (int q = 0; q < CH / 8; ++q) {
        float b[8];
        if (bias) {
          const uint4 bv = __ldg(reinterpret_cast<const uint4*>(bias + 8 * q));
          const __nv_bfloat162* bh = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(bh[i]);
            b[2 * i] = f.x;
            b[2 * i + 1] = f.y;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) b[i] = 0.f;
        }
        uint4 packed;
        __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float x0 = v[8 * q + 2 * i] + b[2 * i];
          float x1 = v[8 * q + 2 * i + 1] + b[2 * i + 1];
          if (EPI == EPI_BIAS_SILU) {
            x0 = x0 / (1.f + __expf(-x0));
            x1 = x1 / (1.f + __expf(-x1));
          }
          ph[i] = __floats2bfloat162_rn(x0, x1);
        }
        *reinterpret_cast<uint4*>(out + 8 * q) = packed;
      }
    } else {
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (n_start + i >= p.N) break;
        float x = v[i] + (bias ? __bfloat162float(bias[i]) : 0.f);
        if (EPI == EPI_BIAS_SILU) x = x / (1.f + __expf(-x));
        out[i] = __float2bfloat16_rn(x);
      }
    }
  }
}

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs p) {
  static_assert(BN >= 16 && BN <= 256 && (BN & (BN - 1)) == 0, "BN: power of two in [16, 256]");
  constexpr uint32_t kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  constexpr uint32_t kIdesc = bf16_idesc(TC_BM, BN);
  constexpr uint32_t kStageBytes = (TC_BM + BN) * TC_BK * 2;
  constexpr int CH = BN < 32 ? BN : 32;
  using Smem = TcSmem<BN, STAGES>;

  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&S.tfull[i]), 1);
      mbar_init(smem_u32(&S.tempty[i]), 128);
    }
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  const int G = p.offsets ? p.G : 1;
  if (warp == 0) {
    // Row-tile prefix over the groups: mpref[g] = sum_{g' < g} ceil(rows_g' / 128).
    int carry = 0;
    if (lane == 0) S.mpref[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int mt = 0;
      if (g < G) {
        const int64_t rows = p.offsets ? (p.offsets[g + 1] - p.offsets[g]) : p.m_rows;
        mt = rows > 0 ? static_cast<int>((rows + TC_BM - 1) / TC_BM) : 0;
      }
      int v = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (g < G) S.mpref[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = S.tmem_base;
  const int NB = (p.N + BN - 1) / BN;
  const int total = S.mpref[G] * NB;
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  volatile int* abort = &S.abort;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, S.mpref, G, NB, p, BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&S.empty[s]), ph ^ 1u, abort, p.flags)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&S.full[s]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d(smem_u32(S.a[s]), &tmA, fb, kb * TC_BK, static_cast<int>(c.row0));
          tma_load_3d(smem_u32(S.b[s]), &tmB, fb, kb * TC_BK, c.n0, c.g);
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
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true, issued_any = false;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), aph ^ 1u, abort, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&S.full[s]), ph, abort, p.flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(S.a[s]), b0 = smem_u32(S.b[s]);
#pragma unroll
          for (int kk = 0; kk < TC_BK / 16; ++kk)
            tc_mma_bf16(d_tmem, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32),
                        kIdesc, (kb | kk) != 0 ? 1u : 0u);
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
  } else {
    // -------------------------------------------------- epilogue (warps 2..5)
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    const int r_in = quad * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const TileCoord c = decode_tile(tile, S.mpref, G, NB, p, BN);
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;  // the warp-collective loads need every lane
      tc_fence_after();
      const int64_t row = c.row0 + r_in;
      const bool valid = row < c.row_end;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int col = 0; col < BN; col += CH) {
        float v[CH];
        if constexpr (CH == 32)
          tmem_ld_32cols(t_row + col, v);
        else
          tmem_ld_16cols(t_row + col, v);
        tc_wait_ld();
        if (valid) epilogue_store<EPI, CH>(p, c.g, row, c.n0 + col, v);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&S.tempty[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

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

template <int BN, int STAGES, int EPI>
cudaError_t launch_tc(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  CUtensorMap tmA, tmB;
  const int64_t a_rows = a.offsets ? a.rows_alloc : a.m_rows;
  const cuuint64_t a_dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a_rows)};
  const cuuint64_t a_str[1] = {static_cast<cuuint64_t>(a.K) * 2};
  const cuuint32_t a_box[2] = {TC_BK, TC_BM};
  const int G = a.offsets ? a.G : 1;
  const cuuint64_t b_dims[3] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.N),
                                static_cast<cuuint64_t>(G)};
  const cuuint64_t b_str[2] = {static_cast<cuuint64_t>(a.K) * 2,
                               static_cast<cuuint64_t>(a.N) * a.K * 2};
  const cuuint32_t b_box[3] = {TC_BK, BN, 1};
  if (!encode_bf16_map(&tmA, a.A, 2, a_dims, a_str, a_box) ||
      !encode_bf16_map(&tmB, a.B, 3, b_dims, b_str, b_box))
    return cudaErrorInvalidValue;

  const int64_t mtiles = a.offsets ? (a.rows_alloc + TC_BM - 1) / TC_BM + G
                                   : (a.m_rows + TC_BM - 1) / TC_BM;
  const int64_t bound = mtiles * ((a.N + BN - 1) / BN);
  const int grid = static_cast<int>(std::min<int64_t>(bound, sm_count));
  if (grid <= 0) return cudaSuccess;
  const size_t smem = sizeof(TcSmem<BN, STAGES>) + 1024;
  auto kern = tc_gemm_kernel<BN, STAGES, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, TC_THREADS, smem, stream>>>(tmA, tmB, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_gemm_bf16(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream) {
  switch (epi) {
    case EPI_BIAS_SILU:
      return launch_tc<256, 4, EPI_BIAS_SILU>(a, sm_count, stream);
    case EPI_BIAS:
      return launch_tc<256, 4, EPI_BIAS>(a, sm_count, stream);
    default:
      // Router: N = E columns; the narrowest power-of-two tile that covers them, at most 128.
      if (a.N <= 16) return launch_tc<16, 8, EPI_ROUTER_F32>(a, sm_count, stream);
      if (a.N <= 32) return launch_tc<32, 8, EPI_ROUTER_F32>(a, sm_count, stream);
      if (a.N <= 64) return launch_tc<64, 8, EPI_ROUTER_F32>(a, sm_count, stream);
      return launch_tc<128, 6, EPI_ROUTER_F32>(a, sm_count, stream);
  }
}

}  // namespace moe
