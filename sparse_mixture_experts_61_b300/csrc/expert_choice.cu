// Expert-choice routing: the direction of selection reversed, each expert taking a
// fixed number C of tokens ("MoE mixture-of-experts routing mechanism: principles and
// sparse activation", section "Expert Choice routing and capacity-factor tuning").
//   EC1  softmax over the experts of each token (split partials of the router
//        contraction added in order, then the logit bias), written token-major for
//        the caller and expert-major [E,T] for the selection;
//   EC2  per expert, the C tokens with the largest probability (equal values: lower
//        token first), emitted in ascending token order, plus the [E,T] row map and
//        the expert-contiguous row offsets e*C.
// The combine over the chosen rows is in combine.cu.
//
// EC2 is an exact radix select on the order-preserving 32-bit key of each fp32
// probability: four 8-bit digit passes narrow the candidates to the key of the C-th
// largest value, then one ordered pass takes every larger key and the first R equal
// ones.  Integer counting only, so the result does not depend on thread timing.

#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kSmWarps = 8;
constexpr int kSmTokensPerWarp = 4;
constexpr int kSmTokens = kSmWarps * kSmTokensPerWarp;  // tokens per softmax CTA

// One CTA per kSmTokens tokens, one warp per token at a time; lane l holds experts
// l, l+32, ... (EPL of them).  The block's probabilities are transposed through
// shared memory so the [E,T] copy is written in 128-byte rows.
template <int EPL>
__global__ void __launch_bounds__(kSmWarps * 32)
    ec_softmax_kernel(const float* __restrict__ src, int nsplit, int64_t split_stride,
                      const float* __restrict__ bias, float* __restrict__ logits_out,
                      float* __restrict__ probs_out, float* __restrict__ probs_et, int64_t T,
                      int E, int* flags) {
  pdl_enter();
  __shared__ float s_p[kMaxExperts][kSmTokens + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kSmTokens;
  for (int i = 0; i < kSmTokensPerWarp; ++i) {
    const int tl = warp * kSmTokensPerWarp + i;
    const int64_t t = t0 + tl;
    if (t >= T) break;  // warp-uniform
    float v[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane + 32 * q;
      v[q] = -INFINITY;
      if (e < E) {
        const float* p0 = src + t * E + e;
        float l = p0[0];
        for (int sp = 1; sp < nsplit; ++sp) l += p0[sp * split_stride];
        if (bias) l += bias[e];
        v[q] = l;
      }
    }
    bool bad = false;
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane + 32 * q;
      if (e < E) {
        if (logits_out) logits_out[t * E + e] = v[q];
        if (!isfinite(v[q])) bad = true;
        m = fmaxf(m, v[q]);
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(flags, MOE_DEVERR_NONFINITE);
    m = warp_max(m);
    float ex[EPL];
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      ex[q] = (lane + 32 * q < E) ? expf(v[q] - m) : 0.f;
      s += ex[q];
    }
    s = warp_sum(s);
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane + 32 * q;
      if (e < E) {
        const float p = ex[q] / s;
        if (probs_out) probs_out[t * E + e] = p;
        s_p[e][tl] = p;
      }
    }
  }
  __syncthreads();
  const int64_t t = t0 + lane;
  if (t < T)
    for (int e = warp; e < E; e += kSmWarps) probs_et[static_cast<int64_t>(e) * T + t] = s_p[e][lane];
}

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

// Unsigned key with the order of the float values (negative values reversed).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive count of `flag` over the threads before this one (thread order);
// *total receives the block's count.  s holds kSelWarps + 1 ints.
__device__ __forceinline__ int block_excl_count(bool flag, int* s, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(b & ((1u << lane) - 1u));
  __syncthreads();  // the previous call's readers are done with s
  if (lane == 0) s[warp] = __popc(b);
  __syncthreads();
  if (warp == 0) {
    const int own = s[lane];
    int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    s[lane] = incl - own;
    if (lane == 31) s[kSelWarps] = incl;
  }
  __syncthreads();
  *total = s[kSelWarps];
  return s[warp] + in_warp;
}

// One CTA per expert e: selects from probs_et[e, 0..T) the C largest, lower token
// first on equal values.  Requires 1 <= C <= T.
__global__ void __launch_bounds__(kSelThreads)
    ec_select_kernel(const float* __restrict__ probs_et, int64_t T, int E, int64_t C,
                     int32_t* __restrict__ sel_token, float* __restrict__ sel_w,
                     int32_t* __restrict__ rowmap_et, int32_t* __restrict__ offsets) {
  pdl_enter();
  __shared__ int s_hist[256];
  __shared__ int s_scan[kSelWarps + 1];
  __shared__ int s_bin, s_before;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    s_bin = 0;
    s_before = 0;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* p = probs_et + static_cast<int64_t>(e) * T;

  // Radix select of the C-th largest key.  Candidates: keys whose digits above the
  // current one equal `prefix`; `remaining` is the target's rank among them.
  uint32_t prefix = 0, mask = 0;
  int remaining = static_cast<int>(C);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSelThreads) s_hist[i] = 0;
    __syncthreads();
    for (int64_t base = 0; base < T; base += kSelThreads) {
      const int64_t t = base + threadIdx.x;
      int bin = 256;  // not a candidate
      if (t < T) {
        const uint32_t key = order_key(p[t]);
        if ((key & mask) == prefix) bin = static_cast<int>((key >> shift) & 0xFFu);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[bin], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // Lane l visits bins 255-8l down to 248-8l; lanes in order cover 255 .. 0.
      int cnt[8], local = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = s_hist[255 - 8 * lane - i];
        local += cnt[i];
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int cum = incl - local;  // candidates in higher bins
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (cum < remaining && cum + cnt[i] >= remaining) {
          s_bin = 255 - 8 * lane - i;
          s_before = cum;
        }
        cum += cnt[i];
      }
    }
    __syncthreads();
    remaining -= s_before;
    prefix |= static_cast<uint32_t>(s_bin) << shift;
    mask |= 0xFFu << shift;
  }
  const uint32_t thr = prefix;  // key of the C-th largest value
  const int take_eq = remaining;  // how many keys equal to thr are taken (lowest t first)

  // Ordered emission: every key above thr, and the first take_eq keys equal to it.
  int32_t* my_tok = sel_token + static_cast<int64_t>(e) * C;
  float* my_w = sel_w + static_cast<int64_t>(e) * C;
  int32_t* my_map = rowmap_et + static_cast<int64_t>(e) * T;
  int carry_eq = 0, carry_sel = 0;
  for (int64_t base = 0; base < T; base += kSelThreads) {
    const int64_t t = base + threadIdx.x;
    const bool valid = t < T;
    const float pv = valid ? p[t] : 0.f;
    const uint32_t key = order_key(pv);
    const bool eq = valid && key == thr;
    int total;
    const int eq_rank = carry_eq + block_excl_count(eq, s_scan, &total);
    carry_eq += total;
    const bool sel = (valid && key > thr) || (eq && eq_rank < take_eq);
    const int pos = carry_sel + block_excl_count(sel, s_scan, &total);
    carry_sel += total;
    // pos < C holds by construction (exactly C keys qualify); the check keeps every
    // store inside the [E,C] outputs regardless.
    const bool keep = sel && pos < C;
    if (keep) {
      my_tok[pos] = static_cast<int32_t>(t);
      my_w[pos] = pv;
    }
    if (valid) my_map[t] = keep ? pos : -1;
  }
  if (threadIdx.x == 0) {
    offsets[e] = static_cast<int32_t>(e * C);
    if (e == E - 1) offsets[E] = static_cast<int32_t>(E * C);
  }
}

}  // namespace

cudaError_t launch_ec_softmax(const float* src, int nsplit, int64_t split_stride,
                              const float* bias, float* logits_out, float* probs_out,
                              float* probs_et, int64_t T, int E, int* flags, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((T + kSmTokens - 1) / kSmTokens)), block(kSmWarps * 32);
#define MOE_EC_SOFTMAX(EPL)                                                                  \
  launch_pdl(ec_softmax_kernel<EPL>, grid, block, 0, stream, src, nsplit, split_stride, bias,        \
                                                     logits_out, probs_out, probs_et, T, E, \
                                                     flags)
  if (E <= 32)
    MOE_EC_SOFTMAX(1);
  else if (E <= 64)
    MOE_EC_SOFTMAX(2);
  else if (E <= 128)
    MOE_EC_SOFTMAX(4);
  else
    MOE_EC_SOFTMAX(8);
#undef MOE_EC_SOFTMAX
  return cudaGetLastError();
}

cudaError_t launch_ec_select(const float* probs_et, int64_t T, int E, int64_t C,
                             int32_t* sel_token, float* sel_w, int32_t* rowmap_et,
                             int32_t* offsets, cudaStream_t stream) {
  if (T == 0 || C <= 0) return cudaSuccess;
  launch_pdl(ec_select_kernel, static_cast<unsigned>(E), kSelThreads, 0, stream, 
      probs_et, T, E, C, sel_token, sel_w, rowmap_et, offsets);
  return cudaGetLastError();
}

}  // namespace moe
