// fp32 grouped GEMM on the CUDA cores, for fp32 layers: the tensor cores have no
// fp32-exact mode (kind::tf32 keeps a 10-bit mantissa), so fp32 operands stay on
// FFMA.  Used for both the router contraction and the two expert GEMMs of an
// fp32 layer:  out[r, n] = act(sum_c A[r, c] * B[g][n][c] + bias),  act = SiLU
// for the first expert GEMM ("MoE mixture-of-experts routing mechanism",
// Expert.forward = w2(silu(w1(x)))).
//
// Output tiles of (16*TM) x (16*TN), TM x TN outputs per thread of 256; 32-deep K
// slices staged in shared memory, double-buffered: the next slice is loaded into
// registers while the current one is multiplied.  64x64 tiles when they fill the
// GPU, 32x32 otherwise (small layers are latency-bound: more CTAs, fewer slices in
// flight per CTA).  Tiles never straddle two groups: group g owns ceil(rows_g/BM)
// row tiles, ordered (group, column block, row block) and walked grid-stride.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BK = 32;
constexpr int kSimtThreads = 256;

template <int EPI, int TM, int TN>
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_f32_kernel(GemmArgs p) {
  constexpr int BM = 16 * TM, BN = 16 * TN;
  constexpr int KV = BK / 4;                      // float4 per row of a slice
  constexpr int VA = (BM * KV + kSimtThreads - 1) / kSimtThreads;  // A vectors per thread
  constexpr int VB = (BN * KV + kSimtThreads - 1) / kSimtThreads;
  pdl_enter();
  __shared__ float As[2][BK][BM + 4];
  __shared__ float Bs[2][BK][BN + 4];
  __shared__ int s_mpref[kMaxExperts + 1];
  const int tid = threadIdx.x;
  const int G = p.offsets ? p.G : 1;
  if (tid < 32) {
    int carry = 0;
    if (tid == 0) s_mpref[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + tid;
      int mt = 0;
      if (g < G) {
        const int64_t rows = p.offsets ? (p.offsets[g + 1] - p.offsets[g]) : p.m_rows;
        mt = rows > 0 ? static_cast<int>((rows + BM - 1) / BM) : 0;
      }
      int v = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (tid >= o) v += n;
      }
      if (g < G) s_mpref[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const int NB = (p.N + BN - 1) / BN;
  const int total = s_mpref[G] * NB;
  const float* A = static_cast<const float*>(p.A);
  const float* B = static_cast<const float*>(p.B);
  const float* bias = static_cast<const float*>(p.bias);
  float* out = static_cast<float*>(p.out);
  const int ty = tid >> 4, tx = tid & 15;
  const int nslices = (p.K + BK - 1) / BK;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_mpref[mid] * NB <= tile) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int mt_g = s_mpref[g + 1] - s_mpref[g];
    const int local = tile - s_mpref[g] * NB;
    const int nb = local / mt_g, mt = local % mt_g;
    const int64_t gbase = p.offsets ? p.offsets[g] : 0;
    const int64_t row_end = p.offsets ? p.offsets[g + 1] : p.m_rows;
    const int64_t row0 = gbase + static_cast<int64_t>(mt) * BM;
    const int n0 = nb * BN;
    const float* Bg = B + static_cast<int64_t>(g) * p.N * p.K;

    // Slice loads: vector v of A covers row v / KV, columns 4 * (v % KV) .. +3.
    float4 ra[VA], rb[VB];
    auto load = [&](int k0) {
#pragma unroll
      for (int i = 0; i < VA; ++i) {
        const int v = tid + i * kSimtThreads;
        const int r = v / KV, kq = 4 * (v % KV);
        ra[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < BM * KV && row0 + r < row_end && k0 + kq < p.K)
          ra[i] = *reinterpret_cast<const float4*>(A + (row0 + r) * p.K + k0 + kq);
      }
#pragma unroll
      for (int i = 0; i < VB; ++i) {
        const int v = tid + i * kSimtThreads;
        const int r = v / KV, kq = 4 * (v % KV);
        rb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < BN * KV && n0 + r < p.N && k0 + kq < p.K)
          rb[i] = *reinterpret_cast<const float4*>(Bg + static_cast<int64_t>(n0 + r) * p.K + k0 +
                                                   kq);
      }
    };
    auto stage = [&](int buf) {
#pragma unroll
      for (int i = 0; i < VA; ++i) {
        const int v = tid + i * kSimtThreads;
        if (v < BM * KV) {
          const int r = v / KV, kq = 4 * (v % KV);
          As[buf][kq + 0][r] = ra[i].x; As[buf][kq + 1][r] = ra[i].y;
          As[buf][kq + 2][r] = ra[i].z; As[buf][kq + 3][r] = ra[i].w;
        }
      }
#pragma unroll
      for (int i = 0; i < VB; ++i) {
        const int v = tid + i * kSimtThreads;
        if (v < BN * KV) {
          const int r = v / KV, kq = 4 * (v % KV);
          Bs[buf][kq + 0][r] = rb[i].x; Bs[buf][kq + 1][r] = rb[i].y;
          Bs[buf][kq + 2][r] = rb[i].z; Bs[buf][kq + 3][r] = rb[i].w;
        }
      }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    load(0);
    stage(0);
    __syncthreads();
    for (int s = 0; s < nslices; ++s) {
      const int buf = s & 1;
      if (s + 1 < nslices) load((s + 1) * BK);  // in flight during this slice's FMAs
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float a[TM], b[TN];
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = As[buf][kk][ty * TM + i];
#pragma unroll
        for (int j = 0; j < TN; ++j) b[j] = Bs[buf][kk][tx * TN + j];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      // The other buffer was last read in slice s-1, before the barrier that ended it.
      if (s + 1 < nslices) stage(buf ^ 1);
      __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int64_t r = row0 + ty * TM + i;
      if (r >= row_end) continue;
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const int n = n0 + tx * TN + j;
        if (n >= p.N) continue;
        float v = acc[i][j];
        if (bias) v += (EPI == EPI_ROUTER_F32) ? bias[n] : bias[static_cast<int64_t>(g) * p.N + n];
        if (EPI == EPI_BIAS_SILU) {
          if (p.pre_out) static_cast<float*>(p.pre_out)[r * p.N + n] = v;
          v = v / (1.f + expf(-v));
        }
        out[r * p.N + n] = v;
      }
    }
  }
}

}  // namespace

template <int TM, int TN>
void launch_simt_tiles(const GemmArgs& a, int epi, int64_t bound, int sm_count,
                       cudaStream_t stream) {
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(bound, static_cast<int64_t>(sm_count) * 8));
  switch (epi) {
    case EPI_BIAS_SILU:
      launch_pdl(simt_gemm_f32_kernel<EPI_BIAS_SILU, TM, TN>, grid, kSimtThreads, 0, stream, a);
      break;
    case EPI_BIAS:
      launch_pdl(simt_gemm_f32_kernel<EPI_BIAS, TM, TN>, grid, kSimtThreads, 0, stream, a);
      break;
    default:
      launch_pdl(simt_gemm_f32_kernel<EPI_ROUTER_F32, TM, TN>, grid, kSimtThreads, 0, stream, a);
      break;
  }
}

cudaError_t launch_simt_gemm_f32(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream) {
  const int G = a.offsets ? a.G : 1;
  const int64_t rows = a.offsets ? a.rows_alloc : a.m_rows;
  // Upper bound on the tiles of a tile shape (each group adds at most one partial tile).
  auto bound = [&](int bm, int bn) {
    return ((rows + bm - 1) / bm + (a.offsets ? G : 0)) * ((a.N + bn - 1) / bn);
  };
  const int64_t b64 = bound(64, 64);
  if (b64 <= 0) return cudaSuccess;
  if (b64 >= sm_count)
    launch_simt_tiles<4, 4>(a, epi, b64, sm_count, stream);
  else
    launch_simt_tiles<2, 2>(a, epi, bound(32, 32), sm_count, stream);
  return cudaGetLastError();
}

}  // namespace moe
