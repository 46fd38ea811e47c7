// Combine: y[t,:] = sum_{j kept} w[t,j] * y_perm[slot_row[t,j], :]
// ("MoE mixture-of-experts routing mechanism": y = sum_{i<=K} G(x)_i E_i(x); the
// MoELayer listing adds each slot's weighted expert output in slot order).
// One warp per token; each lane owns 16-byte column vectors; the k slot
// contributions are added in slot order in fp32 and rounded once.  No atomics.

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 8;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = q;
  }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32)
    combine_kernel(const T* __restrict__ y_perm, const int32_t* __restrict__ slot_row,
                   const float* __restrict__ topk_w, int64_t ntok, int d, int k, int64_t rows,
                   T* __restrict__ y, int* flags) {
  constexpr int V = Vec<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (t >= ntok) return;
  int r[kMaxK];
  float w[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    r[j] = -1;
    w[j] = 0.f;
    if (j < k) {
      int q = slot_row[t * k + j];
      if (q < -1 || q >= rows) {
        if (lane == 0) raise_flag(flags, MOE_DEVERR_BAD_ROW);
        q = -1;
      }
      r[j] = q;
      w[j] = topk_w[t * k + j];
    }
  }
  const int nvec = d / V;
  for (int v = lane; v < nvec; v += 32) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k && r[j] >= 0) {
        float val[V];
        Vec<T>::load(y_perm + static_cast<int64_t>(r[j]) * d + v * V, val);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(w[j], val[i], acc[i]);
      }
    }
    Vec<T>::store(y + t * d + v * V, acc);
  }
}

}  // namespace

cudaError_t launch_combine(int dtype, const void* y_perm, const int32_t* slot_row,
                           const float* topk_w, int64_t T, int d, int k, void* y, int* flags,
                           cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((T + kWarps - 1) / kWarps);
  const int64_t rows = T * k;
  if (dtype == MOE_F32)
    combine_kernel<float><<<grid, kWarps * 32, 0, stream>>>(
        static_cast<const float*>(y_perm), slot_row, topk_w, T, d, k, rows,
        static_cast<float*>(y), flags);
  else
    combine_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(y_perm), slot_row, topk_w, T, d, k, rows,
        static_cast<__nv_bfloat16*>(y), flags);
  return cudaGetLastError();
}

}  // namespace moe
