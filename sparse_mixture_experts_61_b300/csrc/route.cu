// Router stages after the logits contraction:
//   R2  softmax over the experts, top-k selection on the logits (value desc,
//       lower expert index on equality) and the gate weights of the kept experts,
//   R3  per-chunk expert histogram and per-chunk softmax column sums,
//   R4  balance loss E * sum_e f_e P_e, the routing statistics of the counts, and
//       (shared with dispatch) D1: capacity, kept counts, exclusive-scan offsets and
//       the per-chunk position bases.
// Formulas: gating formula G(x)=softmax(TopK(x.W_g)) and TopKRouter.forward /
// load_balancing_loss of "MoE mixture-of-experts routing mechanism: principles
// and sparse activation"; capacity from its "Expert Choice routing and
// capacity-factor tuning" section.
//
// Every reduction has a fixed order (butterfly shuffles, per-warp partials summed
// in warp order, per-chunk partials summed in chunk order), so repeated runs give
// bitwise-identical results.  Integer histograms use shared-memory atomics, whose
// result does not depend on order.

#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {


// s += v with the rounding error carried in c (Kahan); order-fixed, so deterministic.
__device__ __forceinline__ void kahan_add(float& s, float& c, float v) {
  const float y = v - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

constexpr int kRouteWarps = 32;
constexpr int kTokensPerWarp = kChunk / kRouteWarps;

// One CTA per chunk of kChunk tokens, one warp per token at a time.  Lane l holds
// experts l, l+32, ... (EPL of them); K = k, so the per-slot loops have exact trip
// counts instead of kMaxK predicated iterations.
template <int EPL, int K>
__global__ void __launch_bounds__(kRouteWarps * 32)
    route_topk_kernel(const float* __restrict__ src, int nsplit, int64_t split_stride,
                      const float* __restrict__ bias, const float* __restrict__ noise,
                      int noise_mode, float* __restrict__ logits_out, int64_t T, int E,
                      int gate, int32_t* __restrict__ topk_idx,
                      float* __restrict__ topk_w, int32_t* __restrict__ hist,
                      float* __restrict__ psum, int* flags) {
  pdl_enter();
  __shared__ int s_hist[kMaxExperts];
  __shared__ float s_ps[kRouteWarps][kMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();

  float ps[EPL];
#pragma unroll
  for (int q = 0; q < EPL; ++q) ps[q] = 0.f;

  const int64_t t_first = static_cast<int64_t>(blockIdx.x) * kChunk + warp * kTokensPerWarp;
  // The router logits (split partials added in split order, then the bias) of TP
  // tokens at a time, loaded before any of them is processed so that their loads are
  // in flight together; U splits' loads are issued at a time.  TP * EPL * (U + 1)
  // values stay within the 64 registers a thread of this 1024-thread CTA has.
  constexpr int TP = EPL >= 8 ? 1 : kTokensPerWarp;
  constexpr int U = EPL >= 4 ? 2 : 4;
  for (int i0 = 0; i0 < kTokensPerWarp; i0 += TP) {
    float vv[TP][EPL];
#pragma unroll
    for (int i = 0; i < TP; ++i)
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        const int64_t t = t_first + i0 + i;
        const int e = lane + 32 * q;
        vv[i][q] = (t < T && e < E) ? src[t * E + e] : -INFINITY;
      }
    int sp = 1;
    for (; sp + U - 1 < nsplit; sp += U) {
      float part[U][TP][EPL];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < TP; ++i)
#pragma unroll
          for (int q = 0; q < EPL; ++q) {
            const int64_t t = t_first + i0 + i;
            const int e = lane + 32 * q;
            part[u][i][q] = (t < T && e < E) ? src[(sp + u) * split_stride + t * E + e] : 0.f;
          }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < TP; ++i)
#pragma unroll
          for (int q = 0; q < EPL; ++q) vv[i][q] += part[u][i][q];
    }
    for (; sp < nsplit; ++sp)
#pragma unroll
      for (int i = 0; i < TP; ++i)
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          const int64_t t = t_first + i0 + i;
          const int e = lane + 32 * q;
          if (t < T && e < E) vv[i][q] += src[sp * split_stride + t * E + e];
        }

#pragma unroll
    for (int i = 0; i < TP; ++i) {
      const int64_t t = t_first + i0 + i;
      if (t >= T) break;  // warp-uniform
      float v[EPL];
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        v[q] = vv[i][q];
        if (e < E && bias) v[q] += bias[e];
      }
      // sc: the selection scores (the logits themselves without noise).
      float sc[EPL];
      if (noise_mode == MOE_NOISE_PROB_GAUSS || noise_mode == MOE_NOISE_LOGIT_SOFTMAX) {
        float mc = -INFINITY;
#pragma unroll
        for (int q = 0; q < EPL; ++q)
          if (lane + 32 * q < E) mc = fmaxf(mc, v[q]);
        mc = warp_max(mc);
        float sc_sum = 0.f;
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          sc[q] = (lane + 32 * q < E) ? expf(v[q] - mc) : 0.f;
          sc_sum += sc[q];
        }
        sc_sum = warp_sum(sc_sum);
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          const int e = lane + 32 * q;
          if (e < E) {
            const float pc = sc[q] / sc_sum;
            const float n = noise[t * E + e];
            sc[q] = (noise_mode == MOE_NOISE_PROB_GAUSS) ? pc + n : v[q] + n * pc;
          } else {
            sc[q] = -INFINITY;
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
          const int e = lane + 32 * q;
          sc[q] = v[q];
          if (noise_mode == MOE_NOISE_GUMBEL && e < E) {
            // g = -log(-log(u + 1e-9) + 1e-9).  For u > 1/2, u - 1 is exact and
            // log1p keeps -log(u + 1e-9) accurate where it is tiny (u near 1).
            const float u = noise[t * E + e];
            const float a = (u > 0.5f) ? -log1pf((u - 1.0f) + 1e-9f) : -logf(u + 1e-9f);
            sc[q] = v[q] - logf(a + 1e-9f);
          }
        }
      }
      bool bad = false;
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        const int e = lane + 32 * q;
        if (e < E) {
          if (logits_out) logits_out[t * E + e] = sc[q];
          if (!isfinite(sc[q])) bad = true;
        }
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(flags, MOE_DEVERR_NONFINITE);
      // b: the logits the gate weights and f use -- the clean ones when the noise was
      // added to the probabilities, the scores otherwise.
      const bool clean_base = noise_mode == MOE_NOISE_PROB_GAUSS;

      // softmax of b: m = max, s = sum exp(b - m)
      float m = -INFINITY;
#pragma unroll
      for (int q = 0; q < EPL; ++q)
        if (lane + 32 * q < E) m = fmaxf(m, clean_base ? v[q] : sc[q]);
      m = warp_max(m);
      float ex[EPL];
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        ex[q] = (lane + 32 * q < E) ? expf((clean_base ? v[q] : sc[q]) - m) : 0.f;
        s += ex[q];
      }
      s = warp_sum(s);
      const float inv_s = 1.f / s;
#pragma unroll
      for (int q = 0; q < EPL; ++q) ps[q] += ex[q] * inv_s;

      // top-k on the scores: k rounds of a warp arg-max under (value desc, index asc).
      // Each candidate carries its b value for the weights.
      uint32_t taken = 0;
      int sel_e[K];
      float sel_b[K];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        {
          float bv = -INFINITY, bb = 0.f;
          int be = E;  // sentinel: larger than any valid index
#pragma unroll
          for (int q = 0; q < EPL; ++q) {
            const int e = lane + 32 * q;
            if (e < E && !((taken >> q) & 1u) && (sc[q] > bv || (sc[q] == bv && e < be))) {
              bv = sc[q];
              be = e;
              bb = clean_base ? v[q] : sc[q];
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float ob = __shfl_xor_sync(0xffffffffu, bb, o);
            if (ov > bv || (ov == bv && oe < be)) {
              bv = ov;
              be = oe;
              bb = ob;
            }
          }
          if (be >= E) be = 0;  // only reachable with NaN scores, already flagged
          if ((be & 31) == lane) taken |= 1u << (be >> 5);
          sel_e[j] = be;
          sel_b[j] = bb;
        }
      }

      // gate weights of the kept experts
      float bmax = sel_b[0];
#pragma unroll
      for (int j = 1; j < K; ++j) bmax = fmaxf(bmax, sel_b[j]);
      float w[K];
      float den = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        // mode 0: softmax over the kept logits, shifted by the largest kept one;
        // mode 1: the full-softmax probability p_j = exp(b_j - m) / s.
        w[j] = (gate == 0) ? expf(sel_b[j] - bmax) : expf(sel_b[j] - m) / s;
        den += w[j];
      }
      int my_e = 0;
      float my_w = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (j == lane) {
          my_e = sel_e[j];
          my_w = w[j] / den;
        }
      if (lane < K) {
        topk_idx[t * K + lane] = my_e;
        topk_w[t * K + lane] = my_w;
        atomicAdd(&s_hist[my_e], 1);
      }
    }
  }

#pragma unroll
  for (int q = 0; q < EPL; ++q)
    if (lane + 32 * q < E) s_ps[warp][lane + 32 * q] = ps[q];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) acc += s_ps[w][e];
    psum[static_cast<int64_t>(blockIdx.x) * E + e] = acc;
    hist[static_cast<int64_t>(blockIdx.x) * E + e] = s_hist[e];
  }
}

// Single CTA of kFinThreads threads.  The per-chunk tables are reduced by
// kFinThreads / EP slices of consecutive chunks (EP = E rounded up to a power of two,
// at least 32), each slice summing its chunks in order and the slices then added in
// slice order; the rest of the kernel runs on thread e = expert e.
constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads)
    route_finalize_kernel(const int32_t* __restrict__ hist, const float* __restrict__ psum,
                          int nchunks, int E, int64_t T, int64_t C, int32_t* __restrict__ counts,
                          float* __restrict__ aux, int32_t* __restrict__ chunk_base,
                          int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
                          int32_t* __restrict__ dropped, float* __restrict__ stats) {
  pdl_enter();
  __shared__ int s_c[kMaxExperts];
  __shared__ float s_loss[kMaxExperts / 32];
  __shared__ int s_scan[kMaxExperts / 32];
  __shared__ int s_drop;
  __shared__ int s_cnt[kFinThreads];
  __shared__ float s_ps[kFinThreads];
  const int tid = threadIdx.x;
  if (tid == 0) s_drop = 0;
  int EP = 32;
  while (EP < E) EP <<= 1;
  const int nslices = kFinThreads / EP;
  const int per = (nchunks + nslices - 1) / nslices;
  {
    // Slice sl of expert ex: chunks [c_lo, c_hi), summed in order.
    const int sl = tid / EP, ex = tid % EP;
    const int c_lo = sl * per, c_hi = min(nchunks, c_lo + per);
    int cnt = 0;
    float ps = 0.f, pc = 0.f;  // compensated (Kahan) sum of the chunks' softmax sums
    // Sixteen chunks at a time: the loads are issued together (one memory latency per
    // batch), then added in order.  The first batch's counts stay in registers for the
    // position bases below, so a slice of at most sixteen chunks is read once.
    constexpr int B = 16;
    int first[B];
#pragma unroll
    for (int i = 0; i < B; ++i) first[i] = 0;
    if (ex < E) {
      for (int c0 = c_lo; c0 < c_hi; c0 += B) {
        int hv[B];
        float pv[B];
#pragma unroll
        for (int i = 0; i < B; ++i) {
          const int c = c0 + i;
          hv[i] = c < c_hi ? hist[static_cast<int64_t>(c) * E + ex] : 0;
          pv[i] = (psum && c < c_hi) ? psum[static_cast<int64_t>(c) * E + ex] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < B; ++i) {
          cnt += hv[i];
          kahan_add(ps, pc, pv[i]);
        }
        if (c0 == c_lo) {
#pragma unroll
          for (int i = 0; i < B; ++i) first[i] = hv[i];
        }
      }
    }
    s_cnt[tid] = cnt;
    s_ps[tid] = ps - pc;
    __syncthreads();
    // Position bases: the counts of the lower slices, then this slice's chunks in order.
    if (chunk_base && ex < E) {
      int base = 0;
      for (int q = 0; q < sl; ++q) base += s_cnt[q * EP + ex];
      for (int c0 = c_lo; c0 < c_hi; c0 += B) {
        int hv[B];
#pragma unroll
        for (int i = 0; i < B; ++i)
          hv[i] = c0 == c_lo ? first[i]
                             : (c0 + i < c_hi ? hist[static_cast<int64_t>(c0 + i) * E + ex] : 0);
#pragma unroll
        for (int i = 0; i < B; ++i) {
          if (c0 + i < c_hi) chunk_base[static_cast<int64_t>(c0 + i) * E + ex] = base;
          base += hv[i];
        }
      }
    }
  }
  // From here thread e handles expert e; warps 0 .. kExpertWarps-1 cover every expert.
  // Reductions over the experts are butterfly sums within each warp, then the warp
  // partials added in warp order: a fixed order, one barrier each.
  constexpr int kExpertWarps = kMaxExperts / 32;
  const int e = tid, lane = tid & 31, warp = tid >> 5;
  int cnt = 0;
  float ps = 0.f, pc = 0.f;
  if (e < E) {
    for (int q = 0; q < nslices; ++q) {
      cnt += s_cnt[q * EP + e];
      kahan_add(ps, pc, s_ps[q * EP + e]);
    }
    if (counts) counts[e] = cnt;
  }
  // balance loss: E * sum_e (psum_e / T) * (count_e / T) = E * sum_e psum_e count_e / T^2.
  // fp32 throughout (this GPU's FP64 rate is a small fraction of its FP32 rate):
  // compensated sums over the chunks, one rounding per product, a 32-term butterfly.
  const float lv = warp_sum((e < E) ? (ps - pc) * static_cast<float>(cnt) : 0.f);
  if (lane == 0 && warp < kExpertWarps) s_loss[warp] = lv;

  // capacity, kept counts and the exclusive scan of the offsets
  int kp = 0;
  if (e < E) kp = (C < 0 || cnt < C) ? cnt : static_cast<int>(C);
  if (kept && e < E) kept[e] = kp;
  if (e < E && cnt > kp) atomicAdd(&s_drop, cnt - kp);
  int incl = kp;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31 && warp < kExpertWarps) s_scan[warp] = incl;
  __syncthreads();
  if (e == 0) {
    if (psum && aux) {
      // fp32: the warp partials in warp order, then one product and one quotient.
      float tot = 0.f;
      for (int w = 0; w < kExpertWarps; ++w) tot += s_loss[w];
      const float Tf = static_cast<float>(T);
      aux[0] = T > 0 ? static_cast<float>(E) * tot / (Tf * Tf) : 0.f;
    }
    if (dropped) dropped[0] = s_drop;
  }
  if (warp < kExpertWarps)
    for (int w = 0; w < warp; ++w) incl += s_scan[w];
  if (offsets) {
    if (e < E) offsets[e] = incl - kp;
    if (e == E - 1) offsets[E] = incl;
  }

  // Routing statistics of the pre-drop counts, in warp 0 once the counts are in shared
  // memory, without FP64 (this GPU's FP64 pipe is thin, and scalar double chains cost
  // microseconds here).  With load_e = count_e / total and S2 = sum_e count_e^2, both
  // sums of squared deviations follow from one exact integer,
  //   N = E * S2 - total^2  (>= 0):   sum_e (load_e - 1/E)^2 = N / (E total^2),
  //                                   sum_e (count_e - total/E)^2 = N / E,
  // computed in 128-bit integer arithmetic (count_e < 2^31, total < 2^31), so only the
  // closing fp32 formulas round.  The total, the maximum and the dead-expert test
  // (load_e < 1e-4  <=>  10^4 * count_e < total) are exact; the entropy's terms
  // -load_e ln(load_e + 1e-10) are non-negative (up to 1e-10 load_e) and summed in fp32.
  // Sample standard deviations (divisor E - 1); mean load = 1/E.
  if (stats) {
    if (e < E) s_c[e] = cnt;
    __syncthreads();
    if (warp == 0) {
      long long tot = 0;
      unsigned long long s2 = 0;
      int mx = 0;
      for (int i = lane; i < E; i += 32) {
        const int c = s_c[i];
        tot += c;
        s2 += static_cast<unsigned long long>(c) * static_cast<unsigned long long>(c);
        mx = max(mx, c);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const float inv = tot > 0 ? 1.f / static_cast<float>(tot) : 0.f;
      float ent = 0.f;
      int dead = 0;
      for (int i = lane; i < E; i += 32) {
        const int c = s_c[i];
        const float load = static_cast<float>(c) * inv;
        ent -= load * logf(load + 1e-10f);
        dead += (static_cast<long long>(c) * 10000 < tot) ? 1 : 0;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ent += __shfl_xor_sync(0xffffffffu, ent, o);
        dead += __shfl_xor_sync(0xffffffffu, dead, o);
      }
      if (lane == 0) {
        if (tot > 0) {
          const unsigned __int128 n128 =
              static_cast<unsigned __int128>(E) * s2 -
              static_cast<unsigned __int128>(tot) * static_cast<unsigned long long>(tot);
          const float Ef = static_cast<float>(E), totf = static_cast<float>(tot);
          // sqrt(N / (E (E - 1))) = the count standard deviation
          const float cstd = E > 1 ? sqrtf(static_cast<float>(n128) / (Ef * (Ef - 1.f))) : 0.f;
          stats[0] = cstd * Ef / totf;  // std(load) / mean(load)
          stats[1] = static_cast<float>(dead) / Ef;
          stats[2] = static_cast<float>(mx) / totf * Ef;
          stats[3] = ent;
          stats[4] = expf(ent);
          stats[5] = cstd / (totf / Ef + 1e-6f);
        } else {
          for (int q = 0; q < 6; ++q) stats[q] = 0.f;
        }
      }
    }
  }
}

// route_topk_kernel<EPL, k> for the runtime k (1..kMaxK).
template <int EPL, typename... Args>
void launch_topk_k(int k, dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
  switch (k) {
    case 1: launch_pdl(route_topk_kernel<EPL, 1>, grid, block, 0, stream, args...); break;
    case 2: launch_pdl(route_topk_kernel<EPL, 2>, grid, block, 0, stream, args...); break;
    case 3: launch_pdl(route_topk_kernel<EPL, 3>, grid, block, 0, stream, args...); break;
    case 4: launch_pdl(route_topk_kernel<EPL, 4>, grid, block, 0, stream, args...); break;
    case 5: launch_pdl(route_topk_kernel<EPL, 5>, grid, block, 0, stream, args...); break;
    case 6: launch_pdl(route_topk_kernel<EPL, 6>, grid, block, 0, stream, args...); break;
    case 7: launch_pdl(route_topk_kernel<EPL, 7>, grid, block, 0, stream, args...); break;
    default: launch_pdl(route_topk_kernel<EPL, 8>, grid, block, 0, stream, args...); break;
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* src, int nsplit, int64_t split_stride,
                              const float* bias, const float* noise, int noise_mode,
                              float* logits_out, int64_t T, int E, int k, int gate,
                              int32_t* topk_idx, float* topk_w, int32_t* hist, float* psum,
                              int* flags, cudaStream_t stream) {
  const int64_t nchunks = (T + kChunk - 1) / kChunk;
  if (nchunks == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(nchunks)), block(kRouteWarps * 32);
  if (k < 1 || k > kMaxK) return cudaErrorInvalidValue;
  if (E <= 32)
    launch_topk_k<1>(k, grid, block, stream, src, nsplit, split_stride, bias, noise, noise_mode,
                     logits_out, T, E, gate, topk_idx, topk_w, hist, psum, flags);
  else if (E <= 64)
    launch_topk_k<2>(k, grid, block, stream, src, nsplit, split_stride, bias, noise, noise_mode,
                     logits_out, T, E, gate, topk_idx, topk_w, hist, psum, flags);
  else if (E <= 128)
    launch_topk_k<4>(k, grid, block, stream, src, nsplit, split_stride, bias, noise, noise_mode,
                     logits_out, T, E, gate, topk_idx, topk_w, hist, psum, flags);
  else
    launch_topk_k<8>(k, grid, block, stream, src, nsplit, split_stride, bias, noise, noise_mode,
                     logits_out, T, E, gate, topk_idx, topk_w, hist, psum, flags);
  return cudaGetLastError();
}

cudaError_t launch_route_finalize(const int32_t* hist, const float* psum, int nchunks, int E,
                                  int64_t T, int64_t C, int32_t* counts, float* aux,
                                  int32_t* chunk_base, int32_t* kept, int32_t* offsets,
                                  int32_t* dropped, float* stats, cudaStream_t stream) {
  launch_pdl(route_finalize_kernel, 1, kFinThreads, 0, stream, hist, psum, nchunks, E, T, C, counts, aux,
                                                       chunk_base, kept, offsets, dropped, stats);
  return cudaGetLastError();
}

}  // namespace moe
