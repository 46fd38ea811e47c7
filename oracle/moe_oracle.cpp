// Plain, slow CPU oracle of the top-k Mixture-of-Experts FFN forward.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg may load this library.  The CUDA library never
// links, includes or calls it, and it shares no code with the CUDA library.
//
// Every quantity is accumulated in double with explicit per-token loops in the
// order the formulas are written; there is no blocking, fusion or reordering.
// Inputs are read exactly as the GPU receives them (fp32 or bf16 bit patterns)
// and widened exactly to double.
//
// Sources (page titles as printed; section headings translated):
//   [P5] "MoE mixture-of-experts routing mechanism: principles and sparse
//        activation" (yunthe.com) -- the gating formula G(x)=softmax(TopK(x.W_g)),
//        the output y = sum_{i<=K} G(x)_i E_i(x), the PyTorch TopKRouter /
//        Expert / MoELayer listing, the load-balancing loss, and the capacity
//        factor section ("Expert Choice routing and capacity-factor tuning").
//   [P1] "Breaking the MoE trilemma" (0539edu.com), section 3.2 -- the gating
//        network returns top-k logits' softmax as expert weights (top-k first,
//        softmax over the kept logits) and section 3.3 groups tokens by expert.
//
// Parity status per function (what pins it is listed in the tests):
//   orc_logits, orc_softmax, orc_topk, orc_gate_weights, orc_aux_loss,
//   orc_capacity, orc_dispatch, orc_expert_rows, orc_combine, orc_forward,
//   orc_forward_dense, orc_expert_choice, orc_combine_expert_choice and
//   orc_backward are each pinned by closed forms, invariants, library routines,
//   brute force or (the backward) central differences of the fp64 forward in
//   tests/test_oracle_pins.py.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// dtype codes: 0 = IEEE fp32, 1 = bfloat16 (upper 16 bits of an fp32), 2 = IEEE fp64
// (used by the tests that differentiate the layer numerically).
double elem(const void* p, int dtype, int64_t i) {
  if (dtype == 0) return (double)static_cast<const float*>(p)[i];
  if (dtype == 2) return static_cast<const double*>(p)[i];
  uint32_t bits = (uint32_t)static_cast<const uint16_t*>(p)[i] << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int64_t elem_size(int dtype) { return dtype == 0 ? 4 : dtype == 2 ? 8 : 2; }

// SiLU(a) = a * sigmoid(a) = a / (1 + e^{-a})  ([P5] Expert.forward uses F.silu).
double silu(double a) { return a / (1.0 + std::exp(-a)); }

// d SiLU / da = sigmoid(a) * (1 + a * (1 - sigmoid(a))).
double silu_grad(double a) {
  const double sg = 1.0 / (1.0 + std::exp(-a));
  return sg * (1.0 + a * (1.0 - sg));
}

}  // namespace

extern "C" {

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// O1. Router logits ([P5] gating formula, x . W_g; TopKRouter.gate is an
// nn.Linear(dim, E, bias=False), weight stored [E, d]):
//   logits[t,e] = sum_i x[t,i] * Wg[e,i]  (+ logit_bias[e] when given).
void orc_logits(int64_t T, int d, int E, int dtype, const void* x, const void* wg,
                const float* logit_bias, double* logits) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += elem(x, dtype, t * (int64_t)d + i) * elem(wg, dtype, (int64_t)e * d + i);
      if (logit_bias) acc += (double)logit_bias[e];
      logits[t * E + e] = acc;
    }
  }
}

// O2. Full softmax over the experts ([P5] TopKRouter.forward: F.softmax(logits)):
//   p[t,e] = exp(l[t,e] - m_t) / sum_e' exp(l[t,e'] - m_t),  m_t = max_e l[t,e].
void orc_softmax(int64_t T, int E, const double* logits, double* p) {
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    double m = l[0];
    for (int e = 1; e < E; ++e)
      if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += std::exp(l[e] - m);
    for (int e = 0; e < E; ++e) p[t * E + e] = std::exp(l[e] - m) / s;
  }
}

// O3. Top-k selection on the logits ([P5] TopK keeps the K highest scores; the
// listing takes torch.topk of the softmax, which is monotone in the logits).
// Repeat k times: take the largest not-yet-taken logit, the lower expert index
// winning on equality (IEEE comparison, so -0 == +0).  Slot j holds the j-th pick.
void orc_topk(int64_t T, int E, int k, const double* logits, int32_t* idx) {
  std::vector<char> taken(E);
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    for (int e = 0; e < E; ++e) taken[e] = 0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;
      }
      taken[best] = 1;
      idx[t * k + j] = best;
    }
  }
}

// O3w. Gate weights of the kept experts.
//   mode 0 ([P5] G(x) = softmax(TopK(x.W_g)); [P1] softmax of the top-k logits):
//     w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0)        (l_0 = slot-0 logit)
//   mode 1 ([P5] TopKRouter: softmax, top-k, divide by the kept sum):
//     w_j = p_j / sum_j' p_j'                               (p = full softmax)
void orc_gate_weights(int64_t T, int E, int k, int mode, const double* logits,
                      const int32_t* idx, double* w) {
  std::vector<double> p(E);
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    if (mode == 0) {
      double l0 = l[idx[t * k]];
      double den = 0.0;
      for (int j = 0; j < k; ++j) den += std::exp(l[idx[t * k + j]] - l0);
      for (int j = 0; j < k; ++j) w[t * k + j] = std::exp(l[idx[t * k + j]] - l0) / den;
    } else {
      orc_softmax(1, E, l, p.data());
      double den = 0.0;
      for (int j = 0; j < k; ++j) den += p[idx[t * k + j]];
      for (int j = 0; j < k; ++j) w[t * k + j] = p[idx[t * k + j]] / den;
    }
  }
}

// O2n. Noisy routing scores: the values top-k selects on when routing noise is
// applied.  The random draws are inputs (noise[T,E]), so both implementations see
// the same numbers.
//   mode 1 (the sparse-inference article, section 3.2: Gumbel top-k): noise holds
//          uniform draws u; g = -log(-log(u + 1e-9) + 1e-9); score = logit + g.
//   mode 2 (MoE overview, section 2.1: noise added to the probabilities): noise holds
//          the scaled Gaussian draws n; score = softmax(logits) + n.
//   mode 3 (routing-mechanism page, router collapse: logits + noise * softmax(logits)):
//          noise holds the scaled draws n; score = logit + n * softmax(logits).
void orc_noisy_scores(int64_t T, int E, int mode, const double* logits, const float* noise,
                      double* scores) {
  std::vector<double> p(E);
  for (int64_t t = 0; t < T; ++t) {
    const double* l = logits + t * E;
    const float* n = noise + t * E;
    orc_softmax(1, E, l, p.data());
    for (int e = 0; e < E; ++e) {
      double v;
      if (mode == 1)
        v = l[e] - std::log(-std::log((double)n[e] + 1e-9) + 1e-9);
      else if (mode == 2)
        v = p[e] + (double)n[e];
      else
        v = l[e] + (double)n[e] * p[e];
      scores[t * E + e] = v;
    }
  }
}

// O4. Per-expert counts and the load-balancing loss ([P5] load_balancing_loss):
//   f_e = (1/T) sum_t p[t,e]            (full softmax, every gate mode)
//   P_e = count_e / T                   (top-k assignments before any drop; sum_e P_e = k)
//   loss = E * sum_e f_e * P_e
// counts, f and P may be NULL.  T = 0 gives loss 0 and zero counts.
double orc_aux_loss(int64_t T, int E, int k, const double* p, const int32_t* idx,
                    int64_t* counts, double* f, double* P) {
  std::vector<int64_t> c(E, 0);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) c[idx[t * k + j]] += 1;
  double loss = 0.0;
  for (int e = 0; e < E; ++e) {
    double fe = 0.0, pe = 0.0;
    if (T > 0) {
      for (int64_t t = 0; t < T; ++t) fe += p[t * E + e];
      fe /= (double)T;
      pe = (double)c[e] / (double)T;
    }
    if (counts) counts[e] = c[e];
    if (f) f[e] = fe;
    if (P) P[e] = pe;
    loss += fe * pe;
  }
  return (double)E * loss;
}

// O4s. Routing statistics of the per-expert assignment counts (before any drop),
// from the monitoring script of "LLM MoE guide" section 4.1 and the load loss of
// the sparse-inference article's router (sections 2.3 / 3.2).  With load_e =
// count_e / sum(count), mean = sum(load)/E and the sample standard deviation
// (divisor E - 1, the default of the std the pages call; 0 when E = 1):
//   stats[0] cv                = std(load) / mean(load)
//   stats[1] dead_ratio        = #{e : load_e < 1e-4} / E
//   stats[2] max_over_avg      = max(load) / mean(load)
//   stats[3] entropy           = -sum_e load_e * ln(load_e + 1e-10)
//   stats[4] effective_experts = exp(entropy)
//   stats[5] count_cv_loss     = std(count) / (mean(count) + 1e-6)
// With no assignments at all every statistic is 0.
void orc_routing_stats(int E, const int64_t* counts, double* stats) {
  double total = 0.0;
  for (int e = 0; e < E; ++e) total += (double)counts[e];
  for (int i = 0; i < 6; ++i) stats[i] = 0.0;
  if (total <= 0.0) return;
  std::vector<double> load(E);
  for (int e = 0; e < E; ++e) load[e] = (double)counts[e] / total;
  double lsum = 0.0, csum = 0.0;
  for (int e = 0; e < E; ++e) {
    lsum += load[e];
    csum += (double)counts[e];
  }
  const double lmean = lsum / E, cmean = csum / E;
  double lvar = 0.0, cvar = 0.0, lmax = load[0], dead = 0.0, ent = 0.0;
  for (int e = 0; e < E; ++e) {
    lvar += (load[e] - lmean) * (load[e] - lmean);
    cvar += ((double)counts[e] - cmean) * ((double)counts[e] - cmean);
    if (load[e] > lmax) lmax = load[e];
    if (load[e] < 1e-4) dead += 1.0;
    ent -= load[e] * std::log(load[e] + 1e-10);
  }
  const double lstd = E > 1 ? std::sqrt(lvar / (E - 1)) : 0.0;
  const double cstd = E > 1 ? std::sqrt(cvar / (E - 1)) : 0.0;
  stats[0] = lstd / lmean;
  stats[1] = dead / E;
  stats[2] = lmax / lmean;
  stats[3] = ent;
  stats[4] = std::exp(ent);
  stats[5] = cstd / (cmean + 1e-6);
}

// O5a. Capacity ([P5] capacity = tokens_per_batch / num_experts * capacity_factor),
// rounded up to a whole token.  capacity_factor <= 0 means no limit (returns -1).
int64_t orc_capacity(int64_t T, int E, double capacity_factor) {
  if (!(capacity_factor > 0.0)) return -1;
  return (int64_t)std::ceil((double)T * capacity_factor / (double)E);
}

// O5b. Capacity drop and expert-contiguous placement ([P5] capacity section:
// tokens beyond an expert's capacity are rejected and pass through the residual;
// [P1] 3.3 groups tokens by expert id).  Assignments are visited token by token,
// slot by slot; each expert hands out positions 0,1,2,... in that order and an
// assignment is kept iff its position is below the capacity C (C < 0: no limit).
// offsets = exclusive prefix sum of kept counts; a kept assignment (t,j) of
// expert e lands in row offsets[e] + position; row_token[row] = t; dropped
// assignments get slot_row = -1; rows >= offsets[E] of row_token are -1.
// Returns 0, or 1 if an index is outside [0, E).
int orc_dispatch(int64_t T, int E, int k, int64_t C, const int32_t* idx, int32_t* kept,
                 int32_t* offsets, int32_t* slot_row, int32_t* row_token, int64_t* dropped) {
  for (int64_t a = 0; a < T * k; ++a)
    if (idx[a] < 0 || idx[a] >= E) return 1;
  std::vector<int64_t> next(E, 0), nkept(E, 0), pos(T * k);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      pos[t * k + j] = next[e]++;
      if (C < 0 || pos[t * k + j] < C) nkept[e] += 1;
    }
  int64_t run = 0, drop = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)run;
    kept[e] = (int32_t)nkept[e];
    run += nkept[e];
    drop += next[e] - nkept[e];
  }
  offsets[E] = (int32_t)run;
  for (int64_t r = 0; r < T * k; ++r) row_token[r] = -1;
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      int64_t q = pos[t * k + j];
      if (C < 0 || q < C) {
        int64_t row = offsets[e] + q;
        slot_row[t * k + j] = (int32_t)row;
        row_token[row] = (int32_t)t;
      } else {
        slot_row[t * k + j] = -1;
      }
    }
  if (dropped) *dropped = drop;
  return 0;
}

// O5e. Expert-choice selection ([P5], section "Expert Choice routing and capacity-factor
// tuning": the direction of choice is reversed, each expert takes a fixed number of
// tokens from the batch).  Scores p[T,E]
// (the full softmax of the router logits); each expert e takes the C tokens with the
// largest p[t,e], the lower token index winning on equality, and lists them in
// ascending token order: sel_token[e*C + c], with weight sel_w[e*C + c] = p[t,e].
// C must be in [0, T].
void orc_expert_choice(int64_t T, int E, int64_t C, const double* p, int32_t* sel_token,
                       double* sel_w) {
  std::vector<int64_t> order(T);
  for (int e = 0; e < E; ++e) {
    for (int64_t t = 0; t < T; ++t) order[t] = t;
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
      return p[a * E + e] > p[b * E + e];  // stable: equal scores keep token order
    });
    std::vector<int64_t> chosen(order.begin(), order.begin() + C);
    std::sort(chosen.begin(), chosen.end());
    for (int64_t c = 0; c < C; ++c) {
      sel_token[e * C + c] = (int32_t)chosen[c];
      sel_w[e * C + c] = p[chosen[c] * E + e];
    }
  }
}

// O7e. Expert-choice combine: y_t = sum over experts e (ascending) that chose t of
// w(t,e) * z(t,e), where z holds each expert's output for each of its chosen rows
// (z[(e*C + c)*d]).  Tokens no expert chose get y = 0.
void orc_combine_expert_choice(int64_t T, int d, int E, int64_t C, const int32_t* sel_token,
                               const double* sel_w, const double* z, double* y) {
  for (int64_t i = 0; i < T * d; ++i) y[i] = 0.0;
  for (int e = 0; e < E; ++e)
    for (int64_t c = 0; c < C; ++c) {
      const int64_t t = sel_token[e * C + c];
      const double* zz = z + (e * C + c) * (int64_t)d;
      for (int o = 0; o < d; ++o) y[t * d + o] += sel_w[e * C + c] * zz[o];
    }
}

// O6. One expert on n token rows ([P5] Expert: w2(silu(w1(x))) with nn.Linear
// layers that carry biases):  a = W1 x + b1;  s = SiLU(a);  z = W2 s + b2.
// W1 is [h, d], W2 is [d, h] (nn.Linear orientation); b1, b2 may be NULL (zero).
// Each output element is one sequential sum, so the result does not depend on
// the number of threads.
void orc_expert_rows(int d, int h, int dtype, int64_t n, const void* x_rows, const void* w1,
                     const void* b1, const void* w2, const void* b2, double* z) {
  std::vector<double> s(h);
  for (int64_t r = 0; r < n; ++r) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < h; ++i) {
      double a = 0.0;
      for (int c = 0; c < d; ++c)
        a += elem(w1, dtype, (int64_t)i * d + c) * elem(x_rows, dtype, r * d + c);
      if (b1) a += elem(b1, dtype, i);
      s[i] = silu(a);
    }
#pragma omp parallel for schedule(static)
    for (int o = 0; o < d; ++o) {
      double acc = 0.0;
      for (int i = 0; i < h; ++i) acc += elem(w2, dtype, (int64_t)o * h + i) * s[i];
      if (b2) acc += elem(b2, dtype, o);
      z[r * d + o] = acc;
    }
  }
}

// O7. Gate-weighted combine ([P5] y = sum_{i<=K} G(x)_i E_i(x); the listing adds
// expert outputs slot by slot).  z holds E_{idx[t,j]}(x_t) at z[(t*k + j)*d].
// Dropped slots (slot_row < 0) contribute nothing; a token with every slot
// dropped gets y = 0 (it passes through the residual outside this layer).
void orc_combine(int64_t T, int d, int k, const int32_t* slot_row, const double* w,
                 const double* z, double* y) {
  for (int64_t t = 0; t < T; ++t) {
    for (int o = 0; o < d; ++o) y[t * d + o] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (slot_row[t * k + j] < 0) continue;
      const double* zz = z + (t * k + j) * (int64_t)d;
      for (int o = 0; o < d; ++o) y[t * d + o] += w[t * k + j] * zz[o];
    }
  }
}

// Whole layer, stage by stage (O1 -> O7).  Every output pointer may be NULL
// except y.  Returns 0, or 1 if routing produced an invalid index (cannot happen
// for finite logits).
int orc_forward(int64_t T, int d, int h, int E, int k, int mode, int dtype, double capacity_factor,
                const void* x, const void* wg, const float* logit_bias, const void* w1,
                const void* b1, const void* w2, const void* b2, double* y, double* logits_out,
                int32_t* idx_out, double* w_out, int64_t* counts_out, double* aux_out,
                int32_t* kept_out, int32_t* offsets_out, int32_t* slot_row_out,
                int32_t* row_token_out, int64_t* dropped_out) {
  std::vector<double> logits(T * E), p(T * E), w(T * k), z(T * k * (int64_t)d, 0.0);
  std::vector<int32_t> idx(T * k), kept(E), offsets(E + 1), slot_row(T * k), row_token(T * k);
  std::vector<int64_t> counts(E);
  int64_t dropped = 0;
  orc_logits(T, d, E, dtype, x, wg, logit_bias, logits.data());
  orc_softmax(T, E, logits.data(), p.data());
  orc_topk(T, E, k, logits.data(), idx.data());
  orc_gate_weights(T, E, k, mode, logits.data(), idx.data(), w.data());
  double aux = orc_aux_loss(T, E, k, p.data(), idx.data(), counts.data(), nullptr, nullptr);
  int64_t C = orc_capacity(T, E, capacity_factor);
  if (orc_dispatch(T, E, k, C, idx.data(), kept.data(), offsets.data(), slot_row.data(),
                   row_token.data(), &dropped))
    return 1;
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      if (slot_row[t * k + j] < 0) continue;
      int e = idx[t * k + j];
      int64_t sz = elem_size(dtype);
      const char* xr = static_cast<const char*>(x) + t * d * sz;
      const char* w1e = static_cast<const char*>(w1) + (int64_t)e * h * d * sz;
      const char* w2e = static_cast<const char*>(w2) + (int64_t)e * d * h * sz;
      const char* b1e = b1 ? static_cast<const char*>(b1) + (int64_t)e * h * sz : nullptr;
      const char* b2e = b2 ? static_cast<const char*>(b2) + (int64_t)e * d * sz : nullptr;
      orc_expert_rows(d, h, dtype, 1, xr, w1e, b1e, w2e, b2e, z.data() + (t * k + j) * (int64_t)d);
    }
  orc_combine(T, d, k, slot_row.data(), w.data(), z.data(), y);
  if (logits_out) std::memcpy(logits_out, logits.data(), sizeof(double) * T * E);
  if (idx_out) std::memcpy(idx_out, idx.data(), sizeof(int32_t) * T * k);
  if (w_out) std::memcpy(w_out, w.data(), sizeof(double) * T * k);
  if (counts_out) std::memcpy(counts_out, counts.data(), sizeof(int64_t) * E);
  if (aux_out) *aux_out = aux;
  if (kept_out) std::memcpy(kept_out, kept.data(), sizeof(int32_t) * E);
  if (offsets_out) std::memcpy(offsets_out, offsets.data(), sizeof(int32_t) * (E + 1));
  if (slot_row_out) std::memcpy(slot_row_out, slot_row.data(), sizeof(int32_t) * T * k);
  if (row_token_out) std::memcpy(row_token_out, row_token.data(), sizeof(int32_t) * T * k);
  if (dropped_out) *dropped_out = dropped;
  return 0;
}

// B. Backward of the whole layer (the gradients that training through the pages'
// MoELayer would take; the pages print no backward, so this is the chain rule
// applied to O1..O7 in reverse).  Given dy = dL/dy [T,d] (dtype) and d_aux = dL/d aux:
//   forward recomputed: l, p, TopK set S_t, w, capacity and kept slots, and for each
//   kept slot (t,j) of expert e: a = W1[e] x_t + b1[e], s = SiLU(a), z = W2[e] s + b2[e];
//   B7  dz = w_tj dy_t;  dw_tj = <dy_t, z>  (a dropped slot has z = 0, so dw = 0);
//   B6  dW2[e] += dz s^T;  db2[e] += dz;  ds = W2[e]^T dz;  da = ds * SiLU'(a);
//       dW1[e] += da x_t^T;  db1[e] += da;  dx_t += W1[e]^T da;
//   B3  gate: both gate forms give w_j = e^{l_j} / sum_{i in S} e^{l_i} on S, so
//       dl_j = w_j (dw_j - sum_{i in S} w_i dw_i) for j in S, 0 elsewhere;
//   B4  balance loss E sum_e f_e P_e with f_e = mean_t p[t,e] and P_e = counts_e / T
//       (counts do not depend on l): dl[t,c] += d_aux (E/T) p[t,c] (P_c - sum_e P_e p[t,e]);
//   B1  dlogit_bias = sum_t dl[t,:];  dWg = dl^T x;  dx_t += Wg^T dl_t.
// Outputs are double; dlb, db1, db2 may be NULL.  logits_in (may be NULL) replaces the
// recomputed router logits l for everything downstream of O1 (routing, gate weights,
// p), so the backward can be evaluated on another implementation's routing decisions.
// Returns 0, or 1 if routing failed.
int orc_backward(int64_t T, int d, int h, int E, int k, int mode, int dtype,
                 double capacity_factor, const void* x, const void* wg, const float* logit_bias,
                 const void* w1, const void* b1, const void* w2, const void* b2, const void* dy,
                 double d_aux, const double* logits_in, double* dx, double* dwg, double* dlb,
                 double* dw1, double* db1, double* dw2, double* db2) {
  std::vector<double> logits(T * E), p(T * E), w(T * k), dw(T * k, 0.0), dl(T * E, 0.0);
  std::vector<int32_t> idx(T * k), kept(E), offsets(E + 1), slot_row(T * k), row_token(T * k);
  std::vector<int64_t> counts(E);
  int64_t dropped = 0;
  if (logits_in)
    std::memcpy(logits.data(), logits_in, sizeof(double) * T * E);
  else
    orc_logits(T, d, E, dtype, x, wg, logit_bias, logits.data());
  orc_softmax(T, E, logits.data(), p.data());
  orc_topk(T, E, k, logits.data(), idx.data());
  orc_gate_weights(T, E, k, mode, logits.data(), idx.data(), w.data());
  orc_aux_loss(T, E, k, p.data(), idx.data(), counts.data(), nullptr, nullptr);
  const int64_t C = orc_capacity(T, E, capacity_factor);
  if (orc_dispatch(T, E, k, C, idx.data(), kept.data(), offsets.data(), slot_row.data(),
                   row_token.data(), &dropped))
    return 1;
  for (int64_t i = 0; i < T * d; ++i) dx[i] = 0.0;
  for (int64_t i = 0; i < (int64_t)E * d; ++i) dwg[i] = 0.0;
  for (int64_t i = 0; i < (int64_t)E * h * d; ++i) dw1[i] = dw2[i] = 0.0;
  if (db1) for (int64_t i = 0; i < (int64_t)E * h; ++i) db1[i] = 0.0;
  if (db2) for (int64_t i = 0; i < (int64_t)E * d; ++i) db2[i] = 0.0;

  // B7, B6: expert path, slot by slot.
  std::vector<double> a(h), sv(h), z(d), dz(d), ds(h), da(h);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      if (slot_row[t * k + j] < 0) continue;
      const int e = idx[t * k + j];
      const int64_t w1o = (int64_t)e * h * d, w2o = (int64_t)e * d * h;
      for (int i = 0; i < h; ++i) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += elem(w1, dtype, w1o + (int64_t)i * d + c) * elem(x, dtype, t * d + c);
        if (b1) acc += elem(b1, dtype, (int64_t)e * h + i);
        a[i] = acc;
        sv[i] = silu(acc);
      }
      double dwt = 0.0;
      for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int i = 0; i < h; ++i) acc += elem(w2, dtype, w2o + (int64_t)o * h + i) * sv[i];
        if (b2) acc += elem(b2, dtype, (int64_t)e * d + o);
        z[o] = acc;
        const double g = elem(dy, dtype, t * d + o);
        dz[o] = w[t * k + j] * g;
        dwt += g * acc;
      }
      dw[t * k + j] = dwt;
      for (int o = 0; o < d; ++o) {
        for (int i = 0; i < h; ++i) dw2[w2o + (int64_t)o * h + i] += dz[o] * sv[i];
        if (db2) db2[(int64_t)e * d + o] += dz[o];
      }
      for (int i = 0; i < h; ++i) {
        double acc = 0.0;
        for (int o = 0; o < d; ++o) acc += elem(w2, dtype, w2o + (int64_t)o * h + i) * dz[o];
        ds[i] = acc;
        da[i] = acc * silu_grad(a[i]);
      }
      for (int i = 0; i < h; ++i) {
        for (int c = 0; c < d; ++c) dw1[w1o + (int64_t)i * d + c] += da[i] * elem(x, dtype, t * d + c);
        if (db1) db1[(int64_t)e * h + i] += da[i];
      }
      for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int i = 0; i < h; ++i) acc += elem(w1, dtype, w1o + (int64_t)i * d + c) * da[i];
        dx[t * d + c] += acc;
      }
    }

  // B3: gate weights -> logits (softmax over the TopK set).
  for (int64_t t = 0; t < T; ++t) {
    double inner = 0.0;
    for (int j = 0; j < k; ++j) inner += w[t * k + j] * dw[t * k + j];
    for (int j = 0; j < k; ++j)
      dl[t * E + idx[t * k + j]] += w[t * k + j] * (dw[t * k + j] - inner);
  }
  // B4: balance loss -> logits.
  if (d_aux != 0.0 && T > 0) {
    for (int64_t t = 0; t < T; ++t) {
      double pp = 0.0;
      for (int e = 0; e < E; ++e) pp += ((double)counts[e] / (double)T) * p[t * E + e];
      for (int c = 0; c < E; ++c)
        dl[t * E + c] += d_aux * ((double)E / (double)T) * p[t * E + c] *
                         ((double)counts[c] / (double)T - pp);
    }
  }
  // B1: router.
  if (dlb)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += dl[t * E + e];
      dlb[e] = acc;
    }
  for (int e = 0; e < E; ++e)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += dl[t * E + e] * elem(x, dtype, t * d + c);
      dwg[(int64_t)e * d + c] = acc;
    }
  for (int64_t t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += dl[t * E + e] * elem(wg, dtype, (int64_t)e * d + c);
      dx[t * d + c] += acc;
    }
  return 0;
}

// O-BF. Dense brute force of the same layer, for tiny inputs only.  It follows
// the formulas literally and shares no intermediate with orc_forward:
//  * TopK(t) is a set: e is in it iff fewer than k experts rank above e, where e'
//    ranks above e when l_e' > l_e, or l_e' == l_e and e' < e.
//  * mode 0: G = softmax over all E of the logits with non-TopK entries at -inf.
//    mode 1: G_e = p_e / sum_{e' in TopK} p_e' on TopK, 0 elsewhere.
//  * kept(t,e): the number of earlier tokens t' < t with e in TopK(t') is below C.
//  * every expert is evaluated on every token; y_t = sum_e [kept] G_e E_e(x_t).
void orc_forward_dense(int64_t T, int d, int h, int E, int k, int mode, int dtype,
                       double capacity_factor, const void* x, const void* wg,
                       const float* logit_bias, const void* w1, const void* b1, const void* w2,
                       const void* b2, double* y) {
  int64_t sz = elem_size(dtype);
  std::vector<double> l(T * E), z(d), a(h);
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += elem(x, dtype, t * (int64_t)d + i) * elem(wg, dtype, (int64_t)e * d + i);
      l[t * E + e] = acc + (logit_bias ? (double)logit_bias[e] : 0.0);
    }
  std::vector<char> in_topk(T * E);
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      int above = 0;
      for (int q = 0; q < E; ++q)
        if (l[t * E + q] > l[t * E + e] || (l[t * E + q] == l[t * E + e] && q < e)) ++above;
      in_topk[t * E + e] = above < k;
    }
  bool cap = capacity_factor > 0.0;
  double C = cap ? std::ceil((double)T * capacity_factor / (double)E) : 0.0;
  for (int64_t t = 0; t < T; ++t) {
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) mx = l[t * E + e] > mx ? l[t * E + e] : mx;
    std::vector<double> G(E, 0.0);
    if (mode == 0) {
      double den = 0.0;
      for (int e = 0; e < E; ++e)
        den += in_topk[t * E + e] ? std::exp(l[t * E + e] - mx) : 0.0;  // exp(-inf) = 0
      for (int e = 0; e < E; ++e)
        G[e] = in_topk[t * E + e] ? std::exp(l[t * E + e] - mx) / den : 0.0;
    } else {
      double s = 0.0;
      for (int e = 0; e < E; ++e) s += std::exp(l[t * E + e] - mx);
      double kept_sum = 0.0;
      for (int e = 0; e < E; ++e)
        if (in_topk[t * E + e]) kept_sum += std::exp(l[t * E + e] - mx) / s;
      for (int e = 0; e < E; ++e)
        G[e] = in_topk[t * E + e] ? (std::exp(l[t * E + e] - mx) / s) / kept_sum : 0.0;
    }
    for (int o = 0; o < d; ++o) y[t * d + o] = 0.0;
    for (int e = 0; e < E; ++e) {
      // Evaluate expert e on token t whether or not it is selected (dense).
      const char* w1e = static_cast<const char*>(w1) + (int64_t)e * h * d * sz;
      const char* w2e = static_cast<const char*>(w2) + (int64_t)e * d * h * sz;
      for (int i = 0; i < h; ++i) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
          acc += elem(w1e, dtype, (int64_t)i * d + c) * elem(x, dtype, t * (int64_t)d + c);
        if (b1) acc += elem(b1, dtype, (int64_t)e * h + i);
        a[i] = acc * (1.0 / (1.0 + std::exp(-acc)));
      }
      for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int i = 0; i < h; ++i) acc += elem(w2e, dtype, (int64_t)o * h + i) * a[i];
        if (b2) acc += elem(b2, dtype, (int64_t)e * d + o);
        z[o] = acc;
      }
      bool kept = in_topk[t * E + e];
      if (kept && cap) {
        int64_t earlier = 0;
        for (int64_t q = 0; q < t; ++q) earlier += in_topk[q * E + e];
        kept = (double)earlier < C;
      }
      if (!kept) continue;
      for (int o = 0; o < d; ++o) y[t * d + o] += G[e] * z[o];
    }
  }
}

}  // extern "C"
