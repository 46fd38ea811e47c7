// fp32 grouped GEMM on the CUDA cores, for fp32 layers: the tensor cores have no
// fp32-exact mode (kind::tf32 keeps a 10-bit mantissa), so fp32 operands stay on
// FFMA.  Used for both the router contraction and the two expert GEMMs of an
// fp32 layer:  out[r, n] = act(sum_c A[r, c] * B[g][n][c] + bias),  act = SiLU
// for the first expert GEMM ("MoE mixture-of-experts routing mechanism",
// Expert.forward = w2(silu(w1(x)))).
//
// 64x64 output tiles, 16-deep K slices staged in shared memory, 4x4 outputs per
// thread.  Tiles never straddle two groups: group g owns ceil(rows_g/64) row
// tiles, ordered (group, column block, row block) and walked grid-stride.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_f32_kernel(GemmArgs p) {
  pdl_enter();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
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
  const int lr = tid >> 2, lk = (tid & 3) * 4;

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

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < p.K; k0 += BK) {
      float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
      const int64_t ar = row0 + lr;
      if (ar < row_end && k0 + lk < p.K)
        va = *reinterpret_cast<const float4*>(A + ar * p.K + k0 + lk);
      const int bn = n0 + lr;
      if (bn < p.N && k0 + lk < p.K)
        vb = *reinterpret_cast<const float4*>(Bg + static_cast<int64_t>(bn) * p.K + k0 + lk);
      As[lk + 0][lr] = va.x; As[lk + 1][lr] = va.y; As[lk + 2][lr] = va.z; As[lk + 3][lr] = va.w;
      Bs[lk + 0][lr] = vb.x; Bs[lk + 1][lr] = vb.y; Bs[lk + 2][lr] = vb.z; Bs[lk + 3][lr] = vb.w;
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        float a4[4], b4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a4[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b4[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a4[i], b4[j], acc[i][j]);
      }
      __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = row0 + ty * 4 + i;
      if (r >= row_end) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx * 4 + j;
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

cudaError_t launch_simt_gemm_f32(const GemmArgs& a, int epi, int sm_count, cudaStream_t stream) {
  const int G = a.offsets ? a.G : 1;
  const int64_t rows = a.offsets ? a.rows_alloc : a.m_rows;
  const int64_t bound = ((rows + BM - 1) / BM + (a.offsets ? G : 0)) * ((a.N + BN - 1) / BN);
  const int64_t grid = std::min<int64_t>(bound, static_cast<int64_t>(sm_count) * 8);
  if (grid <= 0) return cudaSuccess;
  switch (epi) {
    case EPI_BIAS_SILU:
      launch_pdl(simt_gemm_f32_kernel<EPI_BIAS_SILU>, static_cast<unsigned>(grid), 256, 0, stream, a);
      break;
    case EPI_BIAS:
      launch_pdl(simt_gemm_f32_kernel<EPI_BIAS>, static_cast<unsigned>(grid), 256, 0, stream, a);
      break;
    default:
      launch_pdl(simt_gemm_f32_kernel<EPI_ROUTER_F32>, static_cast<unsigned>(grid), 256, 0, stream, a);
      break;
  }
  return cudaGetLastError();
}

}  // namespace moe
