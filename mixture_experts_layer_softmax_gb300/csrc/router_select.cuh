// Top-k selection of the route, shared by the router kernels.
//
// "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review),
// §2.2 "Router architecture": softmax or sigmoid scores, top-k selection (the
// lower expert index wins a tie), a selection-only bias (aux-loss-free
// balancing), force-balanced routing; the skill page
// "emerging-techniques-moe-training" ("Top-2 Routing (Mixtral)") divides the
// selected scores by their sum (MOE_FLAG_RENORM).
//
//  * select_and_write: one warp per token (any E; slot j of lane l is expert
//    l + 32 j).
//  * select_row8: one thread per token, E <= 8, the logits in registers.  It
//    makes the same choices and computes the probabilities with the same
//    operations in the same order (sums in the order of the warp version's
//    butterfly), so both give identical results on identical logits.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {

struct RouterArgs {
  int T, E, K, h;
  int score;
  bool renorm, force_balance;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_prob;
  uint8_t* routing_map;
};

// fp32(sigma(l)) with sigma evaluated in double.  Kept out of line: the
// double-precision path must stay behind a real branch (GB300's FP64 rate is
// low), never be computed speculatively for every key.
static __device__ __noinline__ float sigmoid_exact_f32(float l) {
  return (float)(1.0 / (1.0 + exp(-(double)l)));
}

// Selection key of one (token, expert): softmax uses the logit, sigmoid uses
// fp32(sigma(l)) with sigma evaluated in double; then + sel_bias in fp32.
MOE_D float selection_key(float l, int e, const RouterArgs& a) {
  float key = l;
  if (a.score == MOE_SCORE_SIGMOID) key = sigmoid_exact_f32(l);
  if (a.sel_bias) key = __fadd_rn(key, __ldg(a.sel_bias + e));
  return key;
}

// The same key with sigma in fp32 (CUDA's expf, within 2 ulp, then a rounded
// add and a rounded divide): it differs from selection_key by at most
// 4.2e-7 * sigma + ulp(key) <= 5.4e-7 + 1.2e-7 |b|.
MOE_D float selection_key_fast(float l, int e, const RouterArgs& a) {
  float key = l;
  if (a.score == MOE_SCORE_SIGMOID) key = sigmoid_f(l);
  if (a.sel_bias) key = __fadd_rn(key, __ldg(a.sel_bias + e));
  return key;
}

// Order-preserving map of fp32 keys onto uint32 (larger key, larger code;
// -0 is folded onto +0 so the two compare equal, as floats do).  Every finite
// key maps above 0.
MOE_D uint32_t sortable_key(float k) {
  const uint32_t b = __float_as_uint(k == 0.f ? 0.f : k);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
MOE_D float from_sortable_key(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Selects K experts for one token whose logits are spread over the warp
// (slot j of lane l is expert l + 32 j) and writes idx/prob/routing_map.
//
// Sigmoid keys are first ranked with the fp32 sigma.  That ranking equals
// the one of the exact keys whenever the K + 1 best fast keys are separated
// by more than twice their error bound (the selected set and its order cannot
// change); otherwise, for that token only, the keys are recomputed with the
// double-precision sigma and ranked again.  The exact pass evaluates only the
// experts whose fast key is within twice the error bound of the (K+1)-th fast
// key: any other expert has K + 1 experts whose exact keys are strictly above
// its own, so it cannot be selected (GB300's FP64 rate makes the full
// re-evaluation a long tail for the warps that need it).
template <int J>
MOE_D void select_and_write(const float (&logit)[J], int t, const RouterArgs& a, int lane) {
  const unsigned FULL = 0xffffffffu;
  uint32_t taken = 0u;  // bit j: slot j of this lane is selected (a register, not an array)
  float key[J];
  int my_idx = -1;      // lane k < K ends up holding the k-th selected expert
  float my_logit = 0.f; // and its logit
  if (a.force_balance) {
    if (lane < a.K) my_idx = (int)(((int64_t)t * a.K + lane) % a.E);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      // expert e is selected iff (e - t*K) mod E < K
      const int64_t d = (((int64_t)e - (int64_t)t * a.K) % a.E + a.E) % a.E;
      if (e < a.E && d < a.K) taken |= 1u << j;
    }
  } else {
    bool exact = a.score != MOE_SCORE_SIGMOID;  // logits are the exact softmax keys
    float cutoff = -INFINITY;  // exact pass after a fast one: keys that may reach the top K + 1
    float last = 0.f;          // the last key the fast pass ranked
    for (int pass = 0; pass < 2; ++pass) {
      taken = 0u;
      if (exact) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int e = lane + 32 * j;
          const bool cand = e < a.E && (pass == 0 || key[j] >= cutoff);  // key[]: fast keys
          key[j] = cand ? selection_key(logit[j], e, a) : -FLT_MAX;
        }
      } else {
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int e = lane + 32 * j;
          key[j] = -FLT_MAX;
          if (e < a.E) key[j] = selection_key_fast(logit[j], e, a);
        }
      }
      // the fast pass also ranks the (K+1)-th key, to check the K-th gap
      const int rounds = exact ? a.K : min(a.K + 1, a.E);
      // This lane's candidates sorted once, best first (larger key; equal
      // keys: lower expert), so each round offers just the head of the list
      // and the winning lane shifts its list by one.  Codes are 0 past E
      // (below every key).
      uint32_t sc[J];
      int se[J];
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int e = lane + 32 * j;
        sc[j] = e < a.E ? sortable_key(key[j]) : 0u;
        se[j] = e;
      }
#pragma unroll
      for (int pass = 0; pass < J; ++pass)  // odd-even transposition sort
#pragma unroll
        for (int j = pass & 1; j + 1 < J; j += 2) {
          const bool swap = sc[j + 1] > sc[j] || (sc[j + 1] == sc[j] && se[j + 1] < se[j]);
          const uint32_t c0 = sc[j], c1 = sc[j + 1];
          const int e0 = se[j], e1 = se[j + 1];
          sc[j] = swap ? c1 : c0;
          sc[j + 1] = swap ? c0 : c1;
          se[j] = swap ? e1 : e0;
          se[j + 1] = swap ? e0 : e1;
        }
      bool safe = true;
      float prev = 0.f;
      for (int k = 0; k < rounds; ++k) {
        // the warp's largest head key and, among the lanes holding it, the
        // lowest expert index: two warp reductions
        const uint32_t lk = sc[0];
        const uint32_t m = __reduce_max_sync(FULL, lk);
        const int bi = (int)__reduce_min_sync(FULL, lk == m ? (uint32_t)se[0] : 0xffffffffu);
        const float bk = from_sortable_key(m);
        if ((bi & 31) == lane) {
          taken |= 1u << (bi >> 5);
#pragma unroll
          for (int j = 0; j + 1 < J; ++j) {
            sc[j] = sc[j + 1];
            se[j] = se[j + 1];
          }
          sc[J - 1] = 0u;
        }
        if (k < a.K && lane == k) my_idx = bi;
        if (!exact && k > 0 && !(prev - bk > 4e-6f * (1.f + fabsf(prev) + fabsf(bk))))
          safe = false;  // warp-uniform: bk and prev are the same on every lane
        prev = bk;
        last = bk;
      }
      if (exact || safe) break;
      exact = true;
      if (rounds == a.K + 1) cutoff = last - 4e-6f * (1.f + fabsf(last));
    }
    // the (K+1)-th key of the fast pass was marked taken only to rank it
    if (a.routing_map) {
      taken = 0u;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (k >= a.K) break;
        const int e = __shfl_sync(FULL, my_idx, k);
        if ((e & 31) == lane) taken |= 1u << (e >> 5);
      }
    }
  }
  // logit of this lane's selected expert
  {
    float sel_l = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      // fetch logit of expert my_idx from lane my_idx & 31, slot my_idx >> 5
      const int src = my_idx & 31;
      const float v = __shfl_sync(FULL, logit[j], src);
      if (my_idx >= 0 && (my_idx >> 5) == j) sel_l = v;
    }
    my_logit = sel_l;
  }
  const bool active = lane < a.K;
  float p = 0.f;
  if (a.score == MOE_SCORE_SOFTMAX) {
    if (a.renorm) {
      float m = active ? my_logit : -INFINITY;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
      const float ex = active ? expf(my_logit - m) : 0.f;
      float s = ex;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(FULL, s, off);
      p = ex / s;
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (lane + 32 * j < a.E) m = fmaxf(m, logit[j]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (lane + 32 * j < a.E) s += expf(logit[j] - m);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(FULL, s, off);
      p = expf(my_logit - m) / s;
    }
  } else {
    const float sg = active ? sigmoid_f(my_logit) : 0.f;
    float s = 0.f;
    if (a.renorm) {
      s = sg;
    } else {
#pragma unroll
      for (int j = 0; j < J; ++j)
        if (lane + 32 * j < a.E) s += sigmoid_f(logit[j]);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(FULL, s, off);
    p = sg / s;
  }
  if (active) {
    a.topk_idx[(int64_t)t * a.K + lane] = my_idx;
    a.topk_prob[(int64_t)t * a.K + lane] = p;
  }
  if (a.routing_map) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int e = lane + 32 * j;
      if (e < a.E) a.routing_map[(int64_t)t * a.E + e] = (taken >> j) & 1u;
    }
  }
}

// Sum of v[0 .. 7] in the order a warp butterfly (xor 16, 8, .., 1) gives
// lane 0 when lanes 0 .. 7 hold v and the other lanes hold zero.
MOE_D float butterfly_sum8(const float (&v)[8]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[4]), __fadd_rn(v[2], v[6])),
                   __fadd_rn(__fadd_rn(v[1], v[5]), __fadd_rn(v[3], v[7])));
}

// Selects K of E <= 8 experts for token t from its logits l[0 .. E - 1] (one
// thread) and writes idx/prob/routing_map; the same choices and arithmetic as
// select_and_write.  Instead of K rounds of "largest key, lowest index", each
// expert's rank in that order is counted in one parallel pass (experts with a
// larger key, or an equal key and a lower index, come first): the k-th
// selected expert is the one of rank k.  The probabilities are evaluated
// branch-free for all 8 slots and masked.  Returns the selected set as a
// bit mask (bit e: expert e).
MOE_D uint32_t select_row8(const float (&l)[8], int t, const RouterArgs& a) {
  int sel[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) sel[k] = 0;
  if (a.force_balance) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < a.K) sel[k] = (int)(((int64_t)t * a.K + k) % a.E);
  } else {
    bool exact = a.score != MOE_SCORE_SIGMOID;
    float fk[8];                // fast keys (sigmoid, first pass)
    float cutoff = -INFINITY;   // exact pass: only keys that may reach the top K + 1
#pragma unroll
    for (int e = 0; e < 8; ++e) fk[e] = 0.f;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      uint32_t sk[8];  // order-preserving codes; 0 (below every key) past E
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint32_t c = 0u;
        if (e < a.E) {
          if (!exact) {
            fk[e] = selection_key_fast(l[e], e, a);
            c = sortable_key(fk[e]);
          } else if (pass == 0 || fk[e] >= cutoff) {
            c = sortable_key(selection_key(l[e], e, a));
          } else {
            c = sortable_key(-FLT_MAX);
          }
        }
        sk[e] = c;
      }
      int rank[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int r = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j != e) r += (sk[j] > sk[e] || (sk[j] == sk[e] && j < e)) ? 1 : 0;
        rank[e] = r;
      }
      uint32_t code_at[9];  // the code of rank k (k <= 8)
#pragma unroll
      for (int k = 0; k < 9; ++k) code_at[k] = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (rank[e] == k) {
            sel[k] = e;
            code_at[k] = sk[e];
          }
      if (exact) break;
      // the fast keys decide when the K + 1 best are separated by more than
      // twice their error bound (the gaps between ranks 0 .. min(K, E - 1))
      const int rounds = min(a.K + 1, a.E);
      bool safe = true;
#pragma unroll
      for (int k = 1; k < 9; ++k)
        if (k < rounds) {
          const float prev = from_sortable_key(code_at[k - 1]), cur = from_sortable_key(code_at[k]);
          if (!(prev - cur > 4e-6f * (1.f + fabsf(prev) + fabsf(cur)))) safe = false;
        }
      if (safe) break;
      exact = true;
      if (rounds == a.K + 1) {
        uint32_t lc = 0u;  // the code of rank K (a register select: no dynamic index)
#pragma unroll
        for (int k = 0; k < 9; ++k)
          if (k == a.K) lc = code_at[k];
        const float last = from_sortable_key(lc);
        cutoff = last - 4e-6f * (1.f + fabsf(last));
      }
    }
  }
  uint32_t taken = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < a.K) taken |= 1u << sel[k];
  float ls[8];  // logit of the k-th selected expert
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float v = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) v = sel[k] == e ? l[e] : v;
    ls[k] = v;
  }
  float p[8], v[8];
  if (a.score == MOE_SCORE_SOFTMAX) {
    float m = -INFINITY;
    if (a.renorm) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < a.K) m = fmaxf(m, ls[k]);
      float ex[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ex[k] = expf(ls[k] - m);
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = k < a.K ? ex[k] : 0.f;
      const float s = butterfly_sum8(v);
#pragma unroll
      for (int k = 0; k < 8; ++k) p[k] = ex[k] / s;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (e < a.E) m = fmaxf(m, l[e]);
      float ex[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ex[e] = expf(l[e] - m);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = e < a.E ? ex[e] : 0.f;
      const float s = butterfly_sum8(v);
#pragma unroll
      for (int k = 0; k < 8; ++k) p[k] = expf(ls[k] - m) / s;
    }
  } else {
    float sg[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) sg[k] = sigmoid_f(ls[k]);
    float s;
    if (a.renorm) {
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = k < a.K ? sg[k] : 0.f;
      s = butterfly_sum8(v);
    } else {
      float sa[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sa[e] = sigmoid_f(l[e]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = e < a.E ? sa[e] : 0.f;
      s = butterfly_sum8(v);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = sg[k] / s;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < a.K) {
      a.topk_idx[(int64_t)t * a.K + k] = sel[k];
      a.topk_prob[(int64_t)t * a.K + k] = p[k];
    }
  if (a.routing_map)
    for (int e = 0; e < a.E; ++e) a.routing_map[(int64_t)t * a.E + e] = (taken >> e) & 1u;
  return taken;
}

}  // namespace moe
