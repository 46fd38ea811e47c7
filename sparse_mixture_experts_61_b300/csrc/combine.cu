// Combine: y[t,:] = sum_{j kept} w[t,j] * y_perm[slot_row[t,j], :]
// ("MoE mixture-of-experts routing mechanism": y = sum_{i<=K} G(x)_i E_i(x); the
// MoELayer listing adds each slot's weighted expert output in slot order).
// Each 16-byte output vector is computed by one lane: the k slot contributions are
// added in slot order in fp32 and rounded once.  No atomics.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {


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

// Work unit = (token, `uv` consecutive 16-byte column vectors); one warp per unit,
// grid-stride.  Lanes 0..k-1 read the token's slots, the warp shares them by shuffles,
// then each lane walks the unit's vectors two at a time, issuing all 2k loads before
// adding.  A unit is the whole row when there are enough tokens to fill the GPU
// (cutting rows up then only repeats the slot reads: measured slower on the prefill
// layers), and a slice of it when there are few (decode), so every SM has work.  No
// shared memory or barrier.
constexpr int kCombineWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const T* __restrict__ y_perm, const int32_t* __restrict__ slot_row,
                   const float* __restrict__ topk_w, int64_t ntok, int d, int k, int64_t rows,
                   int uv, T* __restrict__ y, int* flags) {
  pdl_enter();
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  const int chunks = (nvec + uv - 1) / uv;
  const int64_t units = ntok * chunks;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kCombineWarps;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
       u < units; u += nwarps) {
    const int64_t t = chunks == 1 ? u : u / chunks;
    const int c = static_cast<int>(u - t * chunks);
    int my_q = -1;
    float my_w = 0.f;
    if (lane < k) {
      my_q = slot_row[t * k + lane];
      if (my_q < -1 || my_q >= rows) {
        if (c == 0) raise_flag(flags, MOE_DEVERR_BAD_ROW);
        my_q = -1;
      }
      my_w = topk_w[t * k + lane];
    }
    int64_t src[kMaxK];
    float wj[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      const int q = __shfl_sync(0xffffffffu, my_q, j);
      wj[j] = __shfl_sync(0xffffffffu, my_w, j);
      src[j] = (j < k && q >= 0) ? static_cast<int64_t>(q) * d : -1;
    }
    T* dst = y + t * d;
    const int vend = min(nvec, (c + 1) * uv);
    int v = c * uv + lane;
    for (; v + 32 < vend; v += 64) {
      float a0[V], a1[V];
#pragma unroll
      for (int i = 0; i < V; ++i) a0[i] = a1[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (src[j] >= 0) {
          float x0[V], x1[V];
          Vec<T>::load(y_perm + src[j] + v * V, x0);
          Vec<T>::load(y_perm + src[j] + (v + 32) * V, x1);
#pragma unroll
          for (int i = 0; i < V; ++i) {
            a0[i] = fmaf(wj[j], x0[i], a0[i]);
            a1[i] = fmaf(wj[j], x1[i], a1[i]);
          }
        }
      }
      Vec<T>::store(dst + v * V, a0);
      Vec<T>::store(dst + (v + 32) * V, a1);
    }
    if (v < vend) {
      float a0[V];
#pragma unroll
      for (int i = 0; i < V; ++i) a0[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (src[j] >= 0) {
          float x0[V];
          Vec<T>::load(y_perm + src[j] + v * V, x0);
#pragma unroll
          for (int i = 0; i < V; ++i) a0[i] = fmaf(wj[j], x0[i], a0[i]);
        }
      }
      Vec<T>::store(dst + v * V, a0);
    }
  }
}

// Expert-choice combine ("Expert Choice routing and capacity-factor tuning" section
// of the same page): y[t] = sum over the experts e that took t, in ascending e, of
// p[t,e] * y_perm[e*C + c]; a token no expert took gets 0.  One CTA per token: thread
// e reads the [E,T] row map, the chosen experts are compacted in expert order into
// shared memory, then the CTA's threads stride over the 16-byte column vectors.
constexpr int kEcThreads = kMaxExperts;

template <typename T>
__global__ void __launch_bounds__(kEcThreads)
    ec_combine_kernel(const T* __restrict__ y_perm, const int32_t* __restrict__ rowmap_et,
                      const float* __restrict__ probs_et, int64_t ntok, int E, int64_t C, int d,
                      T* __restrict__ y, int32_t* __restrict__ token_experts,
                      int32_t* __restrict__ unrouted) {
  pdl_enter();
  constexpr int V = Vec<T>::N;
  __shared__ int64_t s_row[kMaxExperts];
  __shared__ float s_w[kMaxExperts];
  __shared__ int s_cnt[kEcThreads / 32];
  const int64_t t = blockIdx.x;
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int c = -1;
  float w = 0.f;
  if (e < E) {
    c = rowmap_et[static_cast<int64_t>(e) * ntok + t];
    if (c >= 0) w = probs_et[static_cast<int64_t>(e) * ntok + t];
  }
  const unsigned b = __ballot_sync(0xffffffffu, c >= 0);
  if (lane == 0) s_cnt[warp] = __popc(b);
  __syncthreads();
  int before = 0, n = 0;
#pragma unroll
  for (int i = 0; i < kEcThreads / 32; ++i) {
    before += (i < warp) ? s_cnt[i] : 0;
    n += s_cnt[i];
  }
  if (c >= 0) {
    const int pos = before + __popc(b & ((1u << lane) - 1u));
    s_row[pos] = static_cast<int64_t>(e) * C + c;
    s_w[pos] = w;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (token_experts) token_experts[t] = n;
    if (n == 0 && unrouted) atomicAdd(unrouted, 1);
  }
  const int nvec = d / V;
  for (int v = threadIdx.x; v < nvec; v += kEcThreads) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int j = 0; j < n; ++j) {
      float val[V];
      Vec<T>::load(y_perm + s_row[j] * d + v * V, val);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(s_w[j], val[i], acc[i]);
    }
    Vec<T>::store(y + t * d + v * V, acc);
  }
}

}  // namespace

cudaError_t launch_ec_combine(int dtype, const void* y_perm, const int32_t* rowmap_et,
                              const float* probs_et, int64_t T, int E, int64_t C, int d, void* y,
                              int32_t* token_experts, int32_t* unrouted, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(T));
  if (dtype == MOE_F32)
    launch_pdl(ec_combine_kernel<float>, grid, kEcThreads, 0, stream, 
        static_cast<const float*>(y_perm), rowmap_et, probs_et, T, E, C, d,
        static_cast<float*>(y), token_experts, unrouted);
  else
    launch_pdl(ec_combine_kernel<__nv_bfloat16>, grid, kEcThreads, 0, stream, 
        static_cast<const __nv_bfloat16*>(y_perm), rowmap_et, probs_et, T, E, C, d,
        static_cast<__nv_bfloat16*>(y), token_experts, unrouted);
  return cudaGetLastError();
}

cudaError_t launch_combine(int dtype, const void* y_perm, const int32_t* slot_row,
                           const float* topk_w, int64_t T, int d, int k, void* y, int* flags,
                           cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  // Vectors per unit: whole rows when T alone gives every SM 16 warps, else rows cut
  // into slices (multiples of 64 vectors) until it does.
  const int vec = dtype == MOE_F32 ? Vec<float>::N : Vec<__nv_bfloat16>::N;
  const int nvec = d / vec;
  const int64_t want = static_cast<int64_t>(sms) * 16;
  const int split = static_cast<int>(std::min<int64_t>((want + T - 1) / T, (nvec + 63) / 64));
  const int uv = ((nvec + split - 1) / split + 63) / 64 * 64;
  const int64_t units = T * ((nvec + uv - 1) / uv);
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(
      (units + kCombineWarps - 1) / kCombineWarps, static_cast<int64_t>(sms) * 8));
  const int64_t rows = T * k;
  if (dtype == MOE_F32)
    launch_pdl(combine_kernel<float>, grid, kCombineWarps * 32, 0, stream,
               static_cast<const float*>(y_perm), slot_row, topk_w, T, d, k, rows, uv,
               static_cast<float*>(y), flags);
  else
    launch_pdl(combine_kernel<__nv_bfloat16>, grid, kCombineWarps * 32, 0, stream,
               static_cast<const __nv_bfloat16*>(y_perm), slot_row, topk_w, T, d, k, rows, uv,
               static_cast<__nv_bfloat16*>(y), flags);
  return cudaGetLastError();
}

}  // namespace moe
