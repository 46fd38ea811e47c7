// Backward GEMMs of the expert FFN and the router on the 5th-generation tensor cores.
//
// The layer's backward is the chain rule through Expert.forward = w2(silu(w1(x))) and
// the router contraction of "MoE mixture-of-experts routing mechanism: principles and
// sparse activation" (the pages print no backward).  With dYp = w * dy per kept slot:
//   data gradients (row tiles, like the forward, but reading the forward weights
//   transposed, i.e. as MN-major B operands):
//     dA  = (dYp . W2[g]) * SiLU'(pre)     per expert, K = d, N = h   (EPI_DSILU)
//     dXp = dA . W1[g]                     per expert, K = h, N = d   (EPI_PLAIN)
//     dxr = dl . W_g                       dense, K = E, N = d        (EPI_PLAIN)
//   (dx = dxr + sum_j dXp[slot j] is summed per token in backward.cu)
//   weight gradients (both operands MN-major, K = the expert's rows):
//     dW2[g] = dYp_g^T . H_g,  dW1[g] = dA_g^T . Xp_g,  dW_g = dl^T . x.
//
// The data-gradient kernel is the forward's row-tile pipeline (tc_pipe.cuh) with B
// loaded as four 64-column boxes of the [G][K][N] weights.  The weight-gradient kernel
// tiles each expert's output [Mdim x Ndim] in 128 x 256 blocks and walks the expert's
// rows in 64-row k-blocks; the last k-block of an expert usually runs into the next
// expert's rows, so it is read from zero-padded copies of each expert's last rows
// (backward.cu packs them before the launch).

#include "tc_pipe.cuh"

namespace moe {
namespace {

constexpr int kBoxBytes = 64 * TC_BK * 2;  // one [64 x 64] bf16 box: 8 KB

__device__ __forceinline__ float silu_grad(float a) {
  const float sg = 1.f / (1.f + __expf(-a));
  return sg * (1.f + a * (1.f - sg));
}

__device__ __forceinline__ void unpack8(const uint4& q, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

// ------------------------------------------------------------- data gradients
// A = rows [128 x 64] K-major (2-D map over [rows_alloc, K]); B = [64 K x 256 N] as four
// MN-major boxes of the 3-D map over [G, K, N]; D[128 x 256] in TMEM.
template <int EPI>
__global__ void __launch_bounds__(ROWS_THREADS, 1)
    tc_bwd_rows_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const GemmArgs p) {
  static_assert(EPI == EPI_DSILU || EPI == EPI_PLAIN, "backward epilogues");
  constexpr int BN = 256, STAGES = 4;
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = bf16_idesc(TILE_M, BN) | kIdescBMnMajor;
  constexpr uint32_t kStageBytes = (TILE_M + BN) * TC_BK * 2;
  using Smem = PipeSmem<TILE_M * TC_BK * 2, BN * TC_BK * 2, STAGES>;
  Smem& S = smem_aligned<Smem>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.offsets ? p.G : 1;
  pipe_prologue<Smem, STAGES>(S, kTmemCols, p, G, TILE_M, &tmA, &tmB, 32 * ROWS_EPI_WARPS);

  const int NB = (p.N + BN - 1) / BN;
  const int total = S.pref[G] * NB;
  const int KB = (p.K + TC_BK - 1) / TC_BK;
  volatile int* abort = &S.abort;

  struct Coord {
    int g, n0, kb0, kb1;
    uint32_t bytes;
    int64_t row0, row_end;
  };
  auto decode = [&](int tile) {
    Coord c;
    c.g = find_group(S.pref, G, NB, tile);
    const int mt = S.pref[c.g + 1] - S.pref[c.g];
    const int local = tile - S.pref[c.g] * NB;
    c.n0 = (local / mt) * BN;
    const int64_t base = p.offsets ? p.offsets[c.g] : 0;
    c.row0 = base + static_cast<int64_t>(local % mt) * TILE_M;
    c.row_end = p.offsets ? p.offsets[c.g + 1] : p.m_rows;
    c.bytes = kStageBytes;
    c.kb0 = 0;
    c.kb1 = KB;
    return c;
  };

  if (warp == 0) {
    if (lane == 0)
      run_producer<STAGES>(
          S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), total, decode,
          [&](const Coord& c, int kb, uint32_t sa, uint32_t sb, uint32_t bar) {
            tma_load_2d(sa, &tmA, bar, kb * TC_BK, static_cast<int>(c.row0));
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(sb + j * kBoxBytes, &tmB, bar, c.n0 + 64 * j, kb * TC_BK, c.g);
          },
          abort, p.flags);
  } else if (warp == 1) {
    if (lane == 0)
      run_mma<STAGES, BN, true>(S, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                                   total, S.tmem_base, decode, [](const Coord&) { return kIdesc; },
                                   abort, p.flags);
  } else {
    const int quad = warp & 3;  // TMEM lanes this warp may read: 32*quad .. 32*quad+31
    constexpr int kColsPerWarp = BN * 4 / ROWS_EPI_WARPS;
    const int col_lo = ((warp - 2) / 4) * kColsPerWarp;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    const __nv_bfloat16* aux = static_cast<const __nv_bfloat16*>(p.aux_in);
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = static_cast<int>(blockIdx.x); tile < total; tile += static_cast<int>(gridDim.x)) {
      const Coord c = decode(tile);
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;  // the warp-collective loads need every lane
      tc_fence_after();
      const int64_t row = c.row0 + quad * 32 + lane;
      const bool valid = row < c.row_end;
      const uint32_t t_row = S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int col = col_lo; col < col_lo + kColsPerWarp; col += 32) {
        float v[32];
        tmem_ld_32cols(t_row + col, v);
        tc_wait_ld();
        if (!valid || c.n0 + col >= p.N) continue;
        const int64_t o = row * p.N + c.n0 + col;
        const bool whole = c.n0 + col + 32 <= p.N;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = v[8 * q + i];
          if (EPI == EPI_DSILU) {
            float a[8];
            if (whole) {
              unpack8(__ldg(reinterpret_cast<const uint4*>(aux + o + 8 * q)), a);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                a[i] = (c.n0 + col + 8 * q + i < p.N) ? __bfloat162float(aux[o + 8 * q + i]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= silu_grad(a[i]);
          }
          uint4 packed;
          __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
          for (int i = 0; i < 4; ++i) ph[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
          if (whole) {
            *reinterpret_cast<uint4*>(out + o + 8 * q) = packed;
          } else {
            const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(&packed);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (c.n0 + col + 8 * q + i < p.N) out[o + 8 * q + i] = pv[i];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&S.tempty[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }
  pipe_teardown(S, kTmemCols);
}

// ------------------------------------------------------------- weight gradients
constexpr int WG_BM = 128, WG_BN = 256, WG_BK = 64;  // output tile; rows per k-block
constexpr int WG_STAGES = 4;
constexpr int WG_THREADS = 192;        // producer, MMA, 4 epilogue warps
constexpr int WG_STG_BOX = 32 * 128;   // one staged store box: 32 rows x 64 bf16

// bf16 outputs leave through shared memory and TMA stores (whole 128-byte lines of the
// gradient, which is as large as the weights and the bulk of this kernel's traffic), a
// half tile at a time: each epilogue warp stages its 32 rows x 128 columns (two boxes).
struct WgradSmem {
  uint8_t a[WG_STAGES][WG_BM * WG_BK * 2];  // two MN-major boxes [64 rows x 64 m]
  uint8_t b[WG_STAGES][WG_BN * WG_BK * 2];  // four MN-major boxes [64 rows x 64 n]
  uint8_t stg[4][2][WG_STG_BOX];            // [epilogue warp][box]
  uint64_t full[WG_STAGES];
  uint64_t empty[WG_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2-5 = epilogue.  The K loop
// of group g covers its rows in 64-row k-blocks.  A last k-block that would run into the
// next group's rows is read instead from the zero-padded copies of each group's last
// rows (tmAt / tmBt, [G, 64, cols], filled by the tail-packing kernel), and only its K
// steps holding rows of the group are issued.  Without offsets (one dense group), rows
// past the end lie outside the tensor and TMA fills them with zeros.
template <bool OUT_F32>
__global__ void __launch_bounds__(WG_THREADS, 1)
    tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmAt,
                    const __grid_constant__ CUtensorMap tmBt,
                    const __grid_constant__ CUtensorMap tmO, const WgradArgs p) {
  constexpr uint32_t kTmemCols = 2 * WG_BN;
  constexpr uint32_t kIdesc = bf16_idesc(WG_BM, WG_BN) | kIdescAMnMajor | kIdescBMnMajor;
  constexpr uint32_t kStageBytes = (WG_BM + WG_BN) * WG_BK * 2;
  WgradSmem& S = smem_aligned<WgradSmem>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_STAGES; ++s) {
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
    if (p.offsets) {
      tma_prefetch_desc(&tmAt);
      tma_prefetch_desc(&tmBt);
    }
    if (!OUT_F32) tma_prefetch_desc(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  // Nothing above touches global memory; wait for the predecessor here.
  pdl_enter();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int G = p.offsets ? p.G : 1;
  const int MB = (p.Mdim + WG_BM - 1) / WG_BM, NB = (p.Ndim + WG_BN - 1) / WG_BN;
  const int total = G * MB * NB;
  const int first = static_cast<int>(blockIdx.x), step = static_cast<int>(gridDim.x);
  volatile int* abort = &S.abort;

  struct Coord {
    int g, m0, n0, nkb, tail;  // tail: valid rows of the last k-block (64 = full)
    int64_t row0;
  };
  auto decode = [&](int tile) {
    Coord c;
    c.g = tile / (MB * NB);
    const int r = tile % (MB * NB);
    c.m0 = (r / NB) * WG_BM;
    c.n0 = (r % NB) * WG_BN;
    c.row0 = p.offsets ? p.offsets[c.g] : 0;
    const int64_t n = p.offsets ? p.offsets[c.g + 1] - c.row0 : p.m_rows;
    c.nkb = n > 0 ? static_cast<int>((n + WG_BK - 1) / WG_BK) : 0;
    c.tail = n > 0 ? static_cast<int>(n - static_cast<int64_t>(c.nkb - 1) * WG_BK) : WG_BK;
    return c;
  };

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_par = 0;
      bool ok = true;
      for (int tile = first; ok && tile < total; tile += step) {
        const Coord c = decode(tile);
        for (int kb = 0; kb < c.nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&S.empty[s]), ph ^ 1u, abort, p.flags)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&S.full[s]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          if (p.offsets && kb == c.nkb - 1 && c.tail < WG_BK) {
#pragma unroll
            for (int j = 0; j < WG_BM / 64; ++j)
              tma_load_3d(smem_u32(S.a[s]) + j * kBoxBytes, &tmAt, fb, c.m0 + 64 * j, 0, c.g);
#pragma unroll
            for (int j = 0; j < WG_BN / 64; ++j)
              tma_load_3d(smem_u32(S.b[s]) + j * kBoxBytes, &tmBt, fb, c.n0 + 64 * j, 0, c.g);
          } else {
            const int row = static_cast<int>(c.row0) + kb * WG_BK;
#pragma unroll
            for (int j = 0; j < WG_BM / 64; ++j)
              tma_load_2d(smem_u32(S.a[s]) + j * kBoxBytes, &tmA, fb, c.m0 + 64 * j, row);
#pragma unroll
            for (int j = 0; j < WG_BN / 64; ++j)
              tma_load_2d(smem_u32(S.b[s]) + j * kBoxBytes, &tmB, fb, c.n0 + 64 * j, row);
          }
          issued |= 1u << s;
          issued_par = (issued_par & ~(1u << s)) | (ph << s);
          if (++s == WG_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int q = 0; q < WG_STAGES; ++q)
          if ((issued >> q) & 1u) mbar_wait_unwind(smem_u32(&S.full[q]), (issued_par >> q) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true, issued_any = false;
      for (int tile = first; ok && tile < total; tile += step) {
        const Coord c = decode(tile);
        if (!mbar_wait_bounded(smem_u32(&S.tempty[acc]), aph ^ 1u, abort, p.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = S.tmem_base + static_cast<uint32_t>(acc * WG_BN);
        for (int kb = 0; kb < c.nkb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&S.full[s]), ph, abort, p.flags)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K steps of 16 rows that hold rows of the group (the rest are zero).
          const int ksteps = kb == c.nkb - 1 ? (c.tail + 15) / 16 : WG_BK / 16;
          const uint32_t a0 = smem_u32(S.a[s]), b0 = smem_u32(S.b[s]);
          for (int kk = 0; kk < ksteps; ++kk)
            tc_mma_bf16(d_tmem, sw128_mnmajor_desc(a0 + kk * 2048, kBoxBytes),
                        sw128_mnmajor_desc(b0 + kk * 2048, kBoxBytes), kIdesc,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          issued_any = true;
          tc_commit(smem_u32(&S.empty[s]));
          if (++s == WG_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(&S.tfull[acc]));  // with no MMA (empty group) it arrives at once
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      if (!ok && issued_any) {
        tc_commit(smem_u32(&S.drain));
        mbar_wait_unwind(smem_u32(&S.drain), 0);
      }
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31 = output rows of the tile
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = first; tile < total; tile += step) {
      const Coord c = decode(tile);
      const bool got = mbar_wait_bounded(smem_u32(&S.tfull[acc]), aph, abort, p.flags);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int m = c.m0 + quad * 32 + lane;
      const uint32_t t_row = S.tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * WG_BN);
      if (OUT_F32) {
        const bool valid = m < p.Mdim;
        const int64_t o = (static_cast<int64_t>(c.g) * p.Mdim + m) * p.Ndim + c.n0;
#pragma unroll 1
        for (int col = 0; col < WG_BN; col += 32) {
          float v[32];
          tmem_ld_32cols(t_row + col, v);
          tc_wait_ld();
          if (!valid || c.n0 + col >= p.Ndim) continue;
          if (c.nkb == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          float* out = static_cast<float*>(p.out) + o + col;
          if (c.n0 + col + 32 <= p.Ndim) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(out + 4 * q) =
                  make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c.n0 + col + i < p.Ndim) out[i] = v[i];
          }
        }
      } else {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          // The previous stores must have finished reading this warp's staging.
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
#pragma unroll 1
          for (int col = half * 128; col < half * 128 + 128; col += 32) {
            float v[32];
            tmem_ld_32cols(t_row + col, v);
            tc_wait_ld();
            if (c.nkb == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            // Box (col%128)/64, row lane; 16-byte chunk (col%64)/8 + q, 128-byte swizzled.
            uint8_t* box = S.stg[quad][(col % 128) / 64] + lane * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 packed;
              __nv_bfloat162* ph2 = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ph2[i] = __floats2bfloat162_rn(v[8 * q + 2 * i], v[8 * q + 2 * i + 1]);
              const int chunk = ((col % 64) / 8 + q) ^ (lane & 7);
              *reinterpret_cast<uint4*>(box + chunk * 16) = packed;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_store_3d(&tmO, smem_u32(S.stg[quad][j]), c.n0 + half * 128 + 64 * j,
                           c.m0 + quad * 32, c.g);
            bulk_commit_group();
          }
        }
      }
      // TMEM drained: the accumulator can take the next tile while the stores run.
      tc_fence_before();
      mbar_arrive(smem_u32(&S.tempty[acc]));
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (!OUT_F32 && lane == 0) bulk_wait_group0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(S.tmem_base, kTmemCols);
  }
}

template <int EPI>
cudaError_t launch_bwd_rows_epi(const GemmArgs& a, int sm_count, cudaStream_t stream) {
  CUtensorMap tmA, tmB;
  const int64_t rows = a.offsets ? a.rows_alloc : a.m_rows;
  // B [G][K][N] read as MN-major boxes of 64 N columns x 64 K rows.
  if (!rows_map(&tmA, a.A, rows, a.K, TILE_M) ||
      !stacked_map(&tmB, a.B, a.offsets ? a.G : 1, /*rows=*/static_cast<int>(a.b_rows ? a.b_rows : a.K),
                   /*cols=*/a.N, 64))
    return cudaErrorInvalidValue;
  const int G = a.offsets ? a.G : 1;
  const int64_t bound = ((rows + TILE_M - 1) / TILE_M + G) * ((a.N + 255) / 256);
  const int grid = static_cast<int>(std::min<int64_t>(bound, sm_count));
  using Smem = PipeSmem<TILE_M * TC_BK * 2, 256 * TC_BK * 2, 4>;
  return launch_pipe(tc_bwd_rows_kernel<EPI>, sizeof(Smem) + 1024, grid, tmA, tmB, a, stream,
                     ROWS_THREADS);
}

}  // namespace

cudaError_t launch_tc_bwd_rows(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream) {
  switch (epi) {
    case EPI_DSILU: return launch_bwd_rows_epi<EPI_DSILU>(a, sm_count, stream);
    case EPI_PLAIN: return launch_bwd_rows_epi<EPI_PLAIN>(a, sm_count, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc_wgrad(const WgradArgs& a, int sm_count, cudaStream_t stream) {
  CUtensorMap tmA, tmB, tmAt{}, tmBt{}, tmO{};
  // [rows, Mdim] and [rows, Ndim] row-major, read as 64-column x 64-row boxes (the tail
  // copies [G, 64, cols] likewise); a bf16 output [G, Mdim, Ndim] is written as
  // 64-column x 32-row boxes.
  const int G = a.offsets ? a.G : 1;
  if (!rows_map(&tmA, a.A, a.rows_alloc, a.Mdim, 64) || !rows_map(&tmB, a.B, a.rows_alloc, a.Ndim, 64))
    return cudaErrorInvalidValue;
  if (a.offsets && (!a.tailA || !a.tailB || !stacked_map(&tmAt, a.tailA, G, 64, a.Mdim, 64) ||
                    !stacked_map(&tmBt, a.tailB, G, 64, a.Ndim, 64)))
    return cudaErrorInvalidValue;
  if (!a.out_f32 && !stacked_map(&tmO, a.out, G, a.Mdim, a.Ndim, 32)) return cudaErrorInvalidValue;
  const int64_t tiles = static_cast<int64_t>(G) * ((a.Mdim + WG_BM - 1) / WG_BM) *
                        ((a.Ndim + WG_BN - 1) / WG_BN);
  const int grid = static_cast<int>(std::min<int64_t>(tiles, sm_count));
  if (grid <= 0) return cudaSuccess;
  const size_t smem = sizeof(WgradSmem) + 1024;
  auto kern = a.out_f32 ? tc_wgrad_kernel<true> : tc_wgrad_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  launch_pdl(kern, grid, WG_THREADS, smem, stream, tmA, tmB, tmAt, tmBt, tmO, a);
  return cudaGetLastError();
}

}  // namespace moe
