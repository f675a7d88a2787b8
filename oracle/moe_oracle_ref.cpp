// Plain, slow C++ CPU oracle of the MoE layer forward pass.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / --impl reference legs of bench.py load this library (through
// oracle/moe_oracle_c.py).  It shares no code, header or constant with the
// CUDA path; it is built with g++ on its own (oracle/build_oracle.py).
//
// What it computes, from the pages ("Scalable Training of Mixture-of-Experts
// Models with Megatron Core", review page: §1.1 p(x) = Softmax(W_r x) and
// MoE(x) = sum_{i in TopK} p_i(x) E_i(x); §2.1 Route -> Dispatch -> Expert
// computation -> Combine; §2.2 gating l = W_r^T x, softmax and sigmoid
// scoring, force-balanced routing; §5.1 the router in FP32.  Skill page
// "emerging-techniques-moe-training", "Basic MoE Architecture": softmax,
// top-k, division by the top-k sum, per-expert accumulation of
// score * expert(x)):
//
//   route:    l[t,e] = sum_j x[t,j] W_r[e,j] (+ b_r[e]), summed in double over
//             the exact inputs and rounded once to fp32;
//             key = l (+ sel_bias) in fp32 for softmax, fp32(sigma(l)) + b in
//             fp32 for sigmoid; the K largest keys, ties to the lower expert
//             index, listed in descending key order; force-balanced routing
//             puts slot k of token t on expert (t*K + k) mod E;
//             p = exp(l_k - m) / sum_sel exp(l_j - m) (softmax, renormalised),
//             the full softmax at the selected experts (not renormalised),
//             sigma(l_k) / sum_sel sigma (sigmoid, renormalised) or over all E;
//   dispatch: counts, offsets (exclusive prefix sum), dst_row[t,k] =
//             offsets[e] + (number of earlier tokens that selected e), and the
//             inverse maps, built expert by expert with tokens ascending;
//   layer:    E_e(x) = W2_e phi(W1_e x + b1_e) + b2_e, phi = GELU (exact erf)
//             or silu(gate) * up (gate = the first F rows of W1_e);
//             y[t] = sum_k p[t,k] E_{idx[t,k]}(x_t) + S(x_t) (shared expert,
//             weight 1), everything in double, nothing rounded in between.
//
// Loops only: no blocking, no fusion, no reordering beyond the definitions
// above.  The one concession to time is an OpenMP loop over tokens (each
// token's output depends on that token alone).
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }
double silu(double z) { return z * sigmoid(z); }
double gelu(double z) { return 0.5 * z * (1.0 + std::erf(z / std::sqrt(2.0))); }

// One expert's output for one token row: out[h] = W2 phi(W1 x + b1) + b2.
// w1 [R1][h] (R1 = 2F for SwiGLU, F for GELU), w2 [h][F], biases or NULL.
void expert_forward(int h, int F, int act, const float* x, const float* w1, const float* w2,
                    const float* b1, const float* b2, std::vector<double>& hidden,
                    std::vector<double>& z, double* out) {
  const int R1 = act == 1 ? 2 * F : F;
  hidden.assign(R1, 0.0);
  for (int i = 0; i < R1; ++i) {
    double acc = 0.0;
    for (int j = 0; j < h; ++j) acc += (double)x[j] * (double)w1[(size_t)i * h + j];
    if (b1) acc += (double)b1[i];
    hidden[i] = acc;
  }
  z.assign(F, 0.0);
  for (int i = 0; i < F; ++i)
    z[i] = act == 1 ? silu(hidden[i]) * hidden[F + i] : gelu(hidden[i]);
  for (int o = 0; o < h; ++o) {
    double acc = 0.0;
    for (int i = 0; i < F; ++i) acc += z[i] * (double)w2[(size_t)o * F + i];
    if (b2) acc += (double)b2[o];
    out[o] = acc;
  }
}

}  // namespace

extern "C" {

// Route every token.  x [T,h], w_r [E,h], gate_bias [E] or NULL (added to the
// logits), sel_bias [E] or NULL (selection only).  Outputs: logits [T,E] fp32,
// idx [T,K] int32, probs [T,K] double.  score: 0 softmax, 1 sigmoid.
// Returns 0, or -1 on a bad size.
int moe_oracle_route(int T, int h, int E, int K, int score, int renorm, int force_balance,
                     const float* x, const float* w_r, const float* gate_bias,
                     const float* sel_bias, float* logits, int32_t* idx, double* probs) {
  if (T < 0 || h < 1 || E < 1 || K < 1 || K > E) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* xt = x + (size_t)t * h;
    float* lt = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int j = 0; j < h; ++j) acc += (double)xt[j] * (double)w_r[(size_t)e * h + j];
      if (gate_bias) acc += (double)gate_bias[e];
      lt[e] = (float)acc;
    }
    int32_t* it = idx + (size_t)t * K;
    if (force_balance) {
      for (int k = 0; k < K; ++k) it[k] = (int32_t)(((int64_t)t * K + k) % E);
    } else {
      std::vector<float> key(E);
      for (int e = 0; e < E; ++e) {
        if (score == 0) {
          key[e] = lt[e];
          if (sel_bias) key[e] = key[e] + sel_bias[e];
        } else {
          key[e] = (float)sigmoid((double)lt[e]);
          if (sel_bias) key[e] = key[e] + sel_bias[e];
        }
      }
      // K rounds: the largest key not yet taken; scanning experts upwards
      // and replacing only on a strictly larger key gives ties to the lower
      // index.
      std::vector<char> taken(E, 0);
      for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!taken[e] && (best < 0 || key[e] > key[best])) best = e;
        taken[best] = 1;
        it[k] = best;
      }
    }
    double* pt = probs + (size_t)t * K;
    if (score == 0) {
      double m = -INFINITY;
      if (renorm) {
        for (int k = 0; k < K; ++k) m = std::fmax(m, (double)lt[it[k]]);
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += std::exp((double)lt[it[k]] - m);
        for (int k = 0; k < K; ++k) pt[k] = std::exp((double)lt[it[k]] - m) / s;
      } else {
        for (int e = 0; e < E; ++e) m = std::fmax(m, (double)lt[e]);
        double s = 0.0;
        for (int e = 0; e < E; ++e) s += std::exp((double)lt[e] - m);
        for (int k = 0; k < K; ++k) pt[k] = std::exp((double)lt[it[k]] - m) / s;
      }
    } else {
      double s = 0.0;
      if (renorm)
        for (int k = 0; k < K; ++k) s += sigmoid((double)lt[it[k]]);
      else
        for (int e = 0; e < E; ++e) s += sigmoid((double)lt[e]);
      for (int k = 0; k < K; ++k) pt[k] = sigmoid((double)lt[it[k]]) / s;
    }
  }
  return 0;
}

// Dispatch maps of idx [T,K]: counts [E], offsets [E+1], dst_row [T,K],
// src_token [T*K], src_slot [T*K] (all int64).  Returns 0, or -1 when an
// expert id lies outside [0, E).
int moe_oracle_dispatch(int T, int E, int K, const int32_t* idx, int64_t* counts,
                        int64_t* offsets, int64_t* dst_row, int64_t* src_token,
                        int64_t* src_slot) {
  for (int64_t i = 0; i < (int64_t)T * K; ++i)
    if (idx[i] < 0 || idx[i] >= E) return -1;
  for (int e = 0; e < E; ++e) {
    counts[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * K; ++i) counts[e] += idx[i] == e;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; ++e) {
    int64_t r = offsets[e];
    for (int t = 0; t < T; ++t)
      for (int k = 0; k < K; ++k)
        if (idx[(size_t)t * K + k] == e) {
          dst_row[(size_t)t * K + k] = r;
          src_token[r] = t;
          src_slot[r] = k;
          ++r;
        }
  }
  return 0;
}

// Layer output for n_tokens tokens (tokens[i] in [0,T)) from a given routing:
// y[i] = sum_k probs[t,k] E_{idx[t,k]}(x_t) + S(x_t), double [n_tokens, h].
// w1[e] / w2[e]: pointers to expert e's [R1][h] / [h][F] weights (NULL for
// experts no listed token selects); b1 [E][R1], b2 [E][h] or NULL; w1s / w2s:
// the shared expert's weights or NULL.  act: 0 GELU, 1 SwiGLU.
// Returns 0, or -1 when a needed expert's weights are missing.
int moe_oracle_layer_fwd(int T, int h, int E, int K, int F, int act, const float* x,
                         const int32_t* idx, const double* probs, const float* const* w1,
                         const float* const* w2, const float* b1, const float* b2,
                         const float* w1s, const float* w2s, int n_tokens,
                         const int64_t* tokens, double* y) {
  const int R1 = act == 1 ? 2 * F : F;
  for (int i = 0; i < n_tokens; ++i) {
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
    for (int k = 0; k < K; ++k) {
      const int e = idx[(size_t)tokens[i] * K + k];
      if (e < 0 || e >= E || !w1[e] || !w2[e]) return -1;
    }
  }
#pragma omp parallel
  {
    std::vector<double> hidden, z, out(h);
#pragma omp for schedule(dynamic, 1)
    for (int i = 0; i < n_tokens; ++i) {
      const int64_t t = tokens[i];
      const float* xt = x + (size_t)t * h;
      double* yt = y + (size_t)i * h;
      for (int o = 0; o < h; ++o) yt[o] = 0.0;
      for (int k = 0; k < K; ++k) {
        const int e = idx[(size_t)t * K + k];
        expert_forward(h, F, act, xt, w1[e], w2[e], b1 ? b1 + (size_t)e * R1 : nullptr,
                       b2 ? b2 + (size_t)e * h : nullptr, hidden, z, out.data());
        const double p = probs[(size_t)t * K + k];
        for (int o = 0; o < h; ++o) yt[o] += p * out[o];
      }
      if (w1s && w2s) {
        expert_forward(h, F, act, xt, w1s, w2s, nullptr, nullptr, hidden, z, out.data());
        for (int o = 0; o < h; ++o) yt[o] += out[o];
      }
    }
  }
  return 0;
}

// Threads the OpenMP loops use (0 if built without OpenMP).
int moe_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 0;
#endif
}

}  // extern "C"
