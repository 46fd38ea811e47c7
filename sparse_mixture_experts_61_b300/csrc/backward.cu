// Element-wise and reduction stages of the layer's backward (the chain rule through
// the gate, the balance loss and the combine of "MoE mixture-of-experts routing
// mechanism: principles and sparse activation"; the pages print no backward):
//   combine:  dYp[r] = w[t,j] dy[t],  dw[t,j] = <dy[t], Yp[r]>   for kept slot (t,j) -> r
//   gate:     dl[t,j-th expert] = w_j (dw_j - sum_i w_i dw_i)   (softmax over the TopK set)
//   balance:  dl[t,c] += d_aux (E/T) p[t,c] (P_c - sum_e P_e p[t,e]),  P_e = counts_e / T
//   bias gradients as column sums per expert group.
// Every reduction has a fixed order, so results are bitwise reproducible.

#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCbThreads = 256;

// One CTA per token; the k slots in order.
__global__ void __launch_bounds__(kCbThreads)
    bwd_combine_kernel(const __nv_bfloat16* __restrict__ dy, const __nv_bfloat16* __restrict__ y_perm,
                       const int32_t* __restrict__ slot_row, const float* __restrict__ topk_w, int d,
                       int k, __nv_bfloat16* __restrict__ dy_perm, float* __restrict__ dw) {
  pdl_enter();
  __shared__ float s_red[kCbThreads / 32];
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = d / 8;
  const uint4* g = reinterpret_cast<const uint4*>(dy + t * d);
  for (int j = 0; j < k; ++j) {
    const int r = slot_row[t * k + j];
    if (r < 0) {
      if (threadIdx.x == 0) dw[t * k + j] = 0.f;
      continue;
    }
    const float w = topk_w[t * k + j];
    const uint4* z = reinterpret_cast<const uint4*>(y_perm + static_cast<int64_t>(r) * d);
    uint4* o = reinterpret_cast<uint4*>(dy_perm + static_cast<int64_t>(r) * d);
    float part = 0.f;
    for (int v = threadIdx.x; v < nvec; v += kCbThreads) {
      const uint4 gq = __ldg(g + v), zq = __ldg(z + v);
      const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gq);
      const __nv_bfloat162* zh = reinterpret_cast<const __nv_bfloat162*>(&zq);
      uint4 oq;
      __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&oq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 gf = __bfloat1622float2(gh[i]), zf = __bfloat1622float2(zh[i]);
        part = fmaf(gf.x, zf.x, part);
        part = fmaf(gf.y, zf.y, part);
        oh[i] = __floats2bfloat162_rn(w * gf.x, w * gf.y);
      }
      o[v] = oq;
    }
    part = warp_sum(part);
    if (lane == 0) s_red[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
      float acc = 0.f;
      for (int i = 0; i < kCbThreads / 32; ++i) acc += s_red[i];
      dw[t * k + j] = acc;
    }
    __syncthreads();
  }
}

constexpr int kGateWarps = 8;

// One warp per token; lane l holds experts l, l+32, ... (EPL of them).
template <int EPL>
__global__ void __launch_bounds__(kGateWarps * 32)
    bwd_gate_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                    const float* __restrict__ topk_w, const float* __restrict__ dw,
                    const int32_t* __restrict__ counts, float d_aux, int64_t T, int E, int Epad,
                    int k, float* __restrict__ dl, __nv_bfloat16* __restrict__ dl16) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kGateWarps + warp;
  if (t >= T) return;
  float l[EPL], g[EPL];
  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane + 32 * q;
    l[q] = e < E ? logits[t * E + e] : -INFINITY;
    m = fmaxf(m, l[q]);
  }
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    l[q] = (lane + 32 * q < E) ? expf(l[q] - m) : 0.f;
    s += l[q];
  }
  s = warp_sum(s);
  // balance loss: d_aux (E/T) p_c (P_c - sum_e P_e p_e)
  const float invT = 1.f / static_cast<float>(T);
  float pp = 0.f;
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane + 32 * q;
    l[q] = l[q] / s;  // p
    if (e < E) pp += static_cast<float>(counts[e]) * invT * l[q];
  }
  pp = warp_sum(pp);
  const float scale = d_aux * static_cast<float>(E) * invT;
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane + 32 * q;
    g[q] = (e < E) ? scale * l[q] * (static_cast<float>(counts[e]) * invT - pp) : 0.f;
  }
  // gate: softmax over the TopK set, slots in order
  int my_e = 0;
  float my_w = 0.f, my_dw = 0.f;
  if (lane < k) {
    my_e = topk_idx[t * k + lane];
    my_w = topk_w[t * k + lane];
    my_dw = dw[t * k + lane];
  }
  float inner = 0.f;
  for (int j = 0; j < k; ++j) inner += __shfl_sync(0xffffffffu, my_w * my_dw, j);
  for (int j = 0; j < k; ++j) {
    const int e = __shfl_sync(0xffffffffu, my_e, j);
    const float c = __shfl_sync(0xffffffffu, my_w * (my_dw - inner), j);
#pragma unroll
    for (int q = 0; q < EPL; ++q)
      if (e == lane + 32 * q) g[q] += c;
  }
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane + 32 * q;
    if (e < E) dl[t * E + e] = g[q];
    if (e < Epad) dl16[t * Epad + e] = __float2bfloat16_rn(e < E ? g[q] : 0.f);
  }
}

// dx: one thread per 16-byte vector of a token; the router term, then the slots in order.
constexpr int kDxThreads = 128;

__global__ void __launch_bounds__(kDxThreads)
    bwd_dx_kernel(const __nv_bfloat16* __restrict__ dxr, const __nv_bfloat16* __restrict__ dxp,
                  const int32_t* __restrict__ slot_row, int d, int k,
                  __nv_bfloat16* __restrict__ dx) {
  pdl_enter();
  __shared__ int s_row[kMaxK];
  const int64_t t = blockIdx.x;
  if (threadIdx.x < k) s_row[threadIdx.x] = slot_row[t * k + threadIdx.x];
  __syncthreads();
  const int v = blockIdx.y * kDxThreads + threadIdx.x;
  if (v >= d / 8) return;
  float acc[8], a[8];
  const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(dxr + t * d) + v);
  const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&q0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h0[i]);
    acc[2 * i] = f.x;
    acc[2 * i + 1] = f.y;
  }
  for (int j = 0; j < k; ++j) {
    const int r = s_row[j];
    if (r < 0) continue;
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(dxp + static_cast<int64_t>(r) * d) + v);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      a[2 * i] = f.x;
      a[2 * i + 1] = f.y;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += a[i];
  }
  uint4 o;
  __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) oh[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  reinterpret_cast<uint4*>(dx + t * d)[v] = o;
}

// Tail packing: CTA (g, r) writes row r of group g's zero-padded last k-block.
constexpr int kPackThreads = 128;

__global__ void __launch_bounds__(kPackThreads)
    pack_tails_kernel(const __nv_bfloat16* __restrict__ A, int cols,
                      const int32_t* __restrict__ offsets, __nv_bfloat16* __restrict__ tail) {
  pdl_enter();
  const int g = blockIdx.x, r = blockIdx.y;
  const int64_t base = offsets[g], n = offsets[g + 1] - base;
  if (n <= 0) return;
  const int64_t nkb = (n + 63) / 64;
  const int valid = static_cast<int>(n - (nkb - 1) * 64);
  if (valid == 64) return;  // the group's last k-block is whole: read in place
  uint4* dst = reinterpret_cast<uint4*>(tail + (static_cast<int64_t>(g) * 64 + r) * cols);
  const uint4* src = reinterpret_cast<const uint4*>(A + (base + (nkb - 1) * 64 + r) * cols);
  for (int v = threadIdx.x; v < cols / 8; v += kPackThreads)
    dst[v] = r < valid ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
}

// Per-group prefix of 64-row slices; thread 0..31 of the block compute it.
constexpr int kSlice = 64;
constexpr int kColThreads = 256;

__device__ void slice_prefix(const int32_t* offsets, int64_t m_rows, int G, int* pref) {
  const int lane = threadIdx.x;
  if (lane < 32) {
    int carry = 0;
    if (lane == 0) pref[0] = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      int n = 0;
      if (g < G) {
        const int64_t rows = offsets ? offsets[g + 1] - offsets[g] : m_rows;
        n = rows > 0 ? static_cast<int>((rows + kSlice - 1) / kSlice) : 0;
      }
      int v = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += x;
      }
      if (g < G) pref[g + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

template <typename Tin>
__global__ void __launch_bounds__(kColThreads)
    colsum_partial_kernel(const Tin* __restrict__ A, int C, const int32_t* __restrict__ offsets,
                          int64_t m_rows, int G, float* __restrict__ partial) {
  pdl_enter();
  __shared__ int pref[kMaxExperts + 1];
  slice_prefix(offsets, m_rows, G, pref);
  const int sl = blockIdx.y;
  if (sl >= pref[G]) return;
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= sl) lo = mid; else hi = mid;
  }
  const int g = lo;
  const int64_t base = offsets ? offsets[g] : 0;
  const int64_t end = offsets ? offsets[g + 1] : m_rows;
  const int64_t r0 = base + static_cast<int64_t>(sl - pref[g]) * kSlice;
  const int64_t r1 = r0 + kSlice < end ? r0 + kSlice : end;
  const int c = blockIdx.x * kColThreads + threadIdx.x;
  if (c >= C) return;
  float acc = 0.f;
  for (int64_t r = r0; r < r1; ++r) acc += to_f32(A[r * C + c]);
  partial[static_cast<int64_t>(sl) * C + c] = acc;
}

__global__ void __launch_bounds__(kColThreads)
    colsum_final_kernel(const float* __restrict__ partial, int C, const int32_t* __restrict__ offsets,
                        int64_t m_rows, int G, float* __restrict__ out) {
  pdl_enter();
  __shared__ int pref[kMaxExperts + 1];
  slice_prefix(offsets, m_rows, G, pref);
  const int g = blockIdx.y;
  const int c = blockIdx.x * kColThreads + threadIdx.x;
  if (c >= C) return;
  float acc = 0.f;
  for (int sl = pref[g]; sl < pref[g + 1]; ++sl) acc += partial[static_cast<int64_t>(sl) * C + c];
  out[static_cast<int64_t>(g) * C + c] = acc;
}

}  // namespace

cudaError_t launch_bwd_combine(const void* dy, const void* y_perm, const int32_t* slot_row,
                               const float* topk_w, int64_t T, int d, int k, void* dy_perm,
                               float* dw, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  launch_pdl(bwd_combine_kernel, static_cast<unsigned>(T), kCbThreads, 0, stream, 
      static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(y_perm), slot_row,
      topk_w, d, k, static_cast<__nv_bfloat16*>(dy_perm), dw);
  return cudaGetLastError();
}

cudaError_t launch_bwd_gate(const float* logits, const int32_t* topk_idx, const float* topk_w,
                            const float* dw, const int32_t* counts, float d_aux, int64_t T,
                            int E, int Epad, int k, float* dl, void* dl16, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>((T + kGateWarps - 1) / kGateWarps);
  __nv_bfloat16* d16 = static_cast<__nv_bfloat16*>(dl16);
#define MOE_GATE_BWD(EPL)                                                                       \
  launch_pdl(bwd_gate_kernel<EPL>, grid, kGateWarps * 32, 0, stream, logits, topk_idx, topk_w, dw, counts, \
                                                             d_aux, T, E, Epad, k, dl, d16)
  if (Epad <= 32)
    MOE_GATE_BWD(1);
  else if (Epad <= 64)
    MOE_GATE_BWD(2);
  else if (Epad <= 128)
    MOE_GATE_BWD(4);
  else
    MOE_GATE_BWD(8);
#undef MOE_GATE_BWD
  return cudaGetLastError();
}

cudaError_t launch_bwd_dx(const void* dxr, const void* dxp, const int32_t* slot_row, int64_t T,
                          int d, int k, void* dx, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((d / 8 + kDxThreads - 1) / kDxThreads));
  launch_pdl(bwd_dx_kernel, grid, kDxThreads, 0, stream, 
      static_cast<const __nv_bfloat16*>(dxr), static_cast<const __nv_bfloat16*>(dxp), slot_row, d,
      k, static_cast<__nv_bfloat16*>(dx));
  return cudaGetLastError();
}

cudaError_t launch_pack_tails(const void* A, int cols, const int32_t* offsets, int G, void* tail,
                              cudaStream_t stream) {
  if (G <= 0) return cudaSuccess;
  launch_pdl(pack_tails_kernel, dim3(static_cast<unsigned>(G), 64), kPackThreads, 0, stream,
             static_cast<const __nv_bfloat16*>(A), cols, offsets,
             static_cast<__nv_bfloat16*>(tail));
  return cudaGetLastError();
}

int64_t colsum_partial_floats(int64_t rows_alloc, int G, int C) {
  return (rows_alloc / kSlice + G + 1) * static_cast<int64_t>(C);
}

cudaError_t launch_colsum(const void* A, bool a_f32, int C, const int32_t* offsets, int64_t m_rows,
                          int64_t rows_alloc, int G, float* partial, float* out,
                          cudaStream_t stream) {
  if (C <= 0 || G <= 0) return cudaSuccess;
  const unsigned cb = static_cast<unsigned>((C + kColThreads - 1) / kColThreads);
  const int64_t slices = rows_alloc / kSlice + G + 1;
  const dim3 g1(cb, static_cast<unsigned>(slices)), g2(cb, static_cast<unsigned>(G));
  if (a_f32)
    launch_pdl(colsum_partial_kernel<float>, g1, kColThreads, 0, stream, static_cast<const float*>(A), C,
                                                                 offsets, m_rows, G, partial);
  else
    launch_pdl(colsum_partial_kernel<__nv_bfloat16>, g1, kColThreads, 0, stream, 
        static_cast<const __nv_bfloat16*>(A), C, offsets, m_rows, G, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(colsum_final_kernel, g2, kColThreads, 0, stream, partial, C, offsets, m_rows, G, out);
  return cudaGetLastError();
}

}  // namespace moe
