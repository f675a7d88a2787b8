"""Plain CPU oracle for the single-GPU MoE layer pass (Route, Dispatch, Expert
compute, Combine, and the backward of the training configuration).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA path: it takes plain numpy arrays (the seeded inputs) and computes
everything in float64 with numpy primitives (matmul, exp, a stable sort,
``scipy.special.erf``).  No blocking, fusion or reordering beyond the plain
definitions below.

Sources (page title, then section / equation):

* "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review
  page), §1.1: p(x) = Softmax(W_r x) and MoE(x) = sum_{i in TopK(p(x))}
  p_i(x) E_i(x); §2.1: the Route -> Dispatch -> Expert computation -> Combine
  stages and the router's two outputs (probs, routing_map); §2.2: gating
  l = W_r^T x with W_r in R^{h x E}, softmax scoring p_i = e^{l_i}/sum_j e^{l_j},
  sigmoid scoring p_i = sigma(l_i)/sum_j sigma(l_j), aux-loss-free and
  force-balanced strategies; §4.1.1: memory-efficient permutation
  y = sum_i W2^(i) (p_i phi(W1^(i) x)), valid when the expert has no bias;
  §5.1: the router is kept in FP32.
* "emerging-techniques-moe-training" skill page, "Basic MoE Architecture"
  (MoELayer.forward: softmax -> topk -> divide by the top-k sum -> masked
  per-expert loop with output[mask] += score * expert(x[mask])), "Top-1
  Routing (Switch Transformer)" (argmax), "Mixtral 8x7B Architecture"
  (index_add_ combine), and "Load Balancing" (the auxiliary loss and the
  router z-loss), "Capacity Factor Tuning" (expert capacity and dropping).
* "Mixture-of-Experts from Architecture to Large-Scale Training", "Keep the
  Dense reference baseline" (one expert with top-1 routing is the dense FFN;
  the router weight then gets no gradient; its load-balance loss is exactly
  1) and "Calculation of activated
  parameters and total parameters" (a bias-free SwiGLU expert holds three
  h x F matrices).

Readings where the pages are silent, ambiguous or leave a step open:

* Sigmoid normalisation: with RENORM the denominator runs over the selected
  top-K (DeepSeek-V3 style); without it, over all E experts (the page's
  formula).  Softmax without RENORM is the full softmax at the selected experts.
* Selection key: softmax selects on the fp32 logit (monotone in p); sigmoid
  selects on float32(sigma(l)) + b, sigma evaluated in float64 and rounded to
  fp32, the add done in fp32.  The bias b only selects; it never enters p.
* Ties go to the lower expert index; the K selected experts are listed in
  descending key order.
* Force-balanced routing: expert (t*K + k) mod E for slot k of token t, probs
  from the scoring function at those experts, renormalised.
* Order inside an expert's segment of the permuted buffer: ascending token.
* GELU is the exact erf form; SwiGLU is silu(gate) * up with the gate in the
  first F rows of W1.
* The shared expert has the routed experts' width, weight 1, and is not routed.
* Expert capacity: counted in (token, slot) pairs, floor(cf * T * K / E) (the
  skill page's int(tokens / experts * capacity_factor) with top-K slots); each
  expert keeps its first C slots in ascending token order and drops the rest;
  the kept weights are not renormalised, and a dropped slot still takes part
  in the router's normalisation (its weight gets a gradient through the kept
  ones).
* Auxiliary loss: the slot fractions count the (token, slot) pairs of the
  selection (the page's bincount over all expert indices), the gate
  probabilities are the full softmax of the logits whatever the scoring
  function, and the fractions carry no gradient.

Parity pins for every function here live in tests/test_oracle_*.py.  The
backward has no printed values on the pages: it is pinned by central finite
differences and by the one-expert identity, not by an external implementation.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
ACT_GELU = 0
ACT_SWIGLU = 1


# ---------------------------------------------------------------------------
# Route
# ---------------------------------------------------------------------------

def gating_logits(x, w_r, gate_bias=None, out_dtype=np.float32):
    """Gating projection l = W_r^T x (+ b_r) for every token (Megatron Core
    review, §2.2 "Gating"; §5.1 keeps it in FP32; the skill page's gate is an
    nn.Linear, whose bias b_r is optional here).

    x: [T, h] token rows (any float dtype; bf16 values arrive exactly as fp32).
    w_r: [E, h], the page's W_r in R^{h x E} stored transposed.
    The dot products are taken in float64 over the exact input values and the
    result is rounded once to ``out_dtype`` (fp32 by default: the logit every
    selection decision uses).
    """
    l = np.asarray(x, np.float64) @ np.asarray(w_r, np.float64).T
    if gate_bias is not None:
        l = l + np.asarray(gate_bias, np.float64)[None, :]
    return l.astype(out_dtype)


def sigmoid(z):
    z = np.asarray(z, np.float64)
    return 1.0 / (1.0 + np.exp(-z))


def selection_keys(logits, score, sel_bias=None):
    """The value top-k compares for each (token, expert).

    Softmax: the logit itself (softmax is strictly increasing in it).
    Sigmoid: float32(sigma(l)) + b in fp32, b the selection-only bias of the
    aux-loss-free strategy (Megatron Core review, §2.2 balancing list).
    """
    l = np.asarray(logits)
    if score == SCORE_SOFTMAX:
        keys = l.astype(np.float32) if l.dtype == np.float32 else l.astype(np.float64)
        if sel_bias is not None:
            keys = keys + np.asarray(sel_bias, keys.dtype)[None, :]
        return keys
    s = sigmoid(l)
    if l.dtype == np.float32:
        s = s.astype(np.float32)
        if sel_bias is not None:
            s = s + np.asarray(sel_bias, np.float32)[None, :]
        return s
    if sel_bias is not None:
        s = s + np.asarray(sel_bias, np.float64)[None, :]
    return s


def select_topk(keys, K):
    """Top-K experts per token: a full stable sort on the descending key, so
    equal keys keep ascending expert order (lower index wins a tie).  Returns
    [T, K] int32 in descending-key order."""
    keys = np.asarray(keys)
    order = np.argsort(-keys, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def force_balanced_topk(T, K, E):
    """Force-balanced routing (Megatron Core review, §2.2): slot k of token t
    goes to expert (t*K + k) mod E, so each expert receives exactly T*K/E slots
    when E divides T*K."""
    t = np.arange(T, dtype=np.int64)[:, None]
    k = np.arange(K, dtype=np.int64)[None, :]
    return ((t * K + k) % E).astype(np.int32)


def topk_probs(logits, idx, score, renorm=True):
    """Routing weights of the selected experts, float64 [T, K].

    Softmax, renormalised: exp(l_k - m) / sum_{j selected} exp(l_j - m)
    (skill page, "Basic MoE Architecture": softmax, topk, divide by the top-k
    sum).  Softmax, not renormalised: the full softmax over E at the selected
    experts (review §1.1 p(x)).  Sigmoid, renormalised: sigma(l_k) / sum over
    the selected sigma; not renormalised: over all E (review §2.2).
    """
    l = np.asarray(logits, np.float64)
    idx = np.asarray(idx, np.int64)
    sel = np.take_along_axis(l, idx, axis=1)
    if score == SCORE_SOFTMAX:
        if renorm:
            m = sel.max(axis=1, keepdims=True)
            e = np.exp(sel - m)
            return e / e.sum(axis=1, keepdims=True)
        m = l.max(axis=1, keepdims=True)
        return np.exp(sel - m) / np.exp(l - m).sum(axis=1, keepdims=True)
    s_all = sigmoid(l)
    s_sel = np.take_along_axis(s_all, idx, axis=1)
    if renorm:
        return s_sel / s_sel.sum(axis=1, keepdims=True)
    return s_sel / s_all.sum(axis=1, keepdims=True)


def routing_map(idx, E):
    """Boolean token x expert mask of the assignment (review §2.1, router
    output ``routing_map``)."""
    T = idx.shape[0]
    m = np.zeros((T, E), dtype=bool)
    m[np.arange(T)[:, None], np.asarray(idx, np.int64)] = True
    return m


def route(logits, K, score, renorm=True, sel_bias=None, force_balance=False):
    """Route stage: (idx [T,K] int32, probs [T,K] float64)."""
    T, E = np.asarray(logits).shape
    if force_balance:
        idx = force_balanced_topk(T, K, E)
    else:
        idx = select_topk(selection_keys(logits, score, sel_bias), K)
    return idx, topk_probs(logits, idx, score, renorm)


def selection_margin(logits, K, score, sel_bias=None):
    """Gap between the K-th and (K+1)-th largest selection key per token
    (+inf when K == E).  Tokens with a tiny margin may legitimately route
    differently under a different but valid fp32 rounding of the logits."""
    keys = np.asarray(selection_keys(logits, score, sel_bias), np.float64)
    E = keys.shape[1]
    if K >= E:
        return np.full(keys.shape[0], np.inf)
    s = -np.sort(-keys, axis=1)
    return s[:, K - 1] - s[:, K]


def order_margin(logits, K, score, sel_bias=None):
    """Smallest gap between consecutive keys among the top K+1 (top K when
    K == E): below it, a different valid fp32 rounding of the logits may list
    the selected experts in another order (the selected set is decided by
    selection_margin alone)."""
    keys = np.asarray(selection_keys(logits, score, sel_bias), np.float64)
    s = -np.sort(-keys, axis=1)[:, :min(K + 1, keys.shape[1])]
    if s.shape[1] < 2:
        return np.full(keys.shape[0], np.inf)
    return (s[:, :-1] - s[:, 1:]).min(axis=1)


# ---------------------------------------------------------------------------
# Dispatch
# ---------------------------------------------------------------------------

def dispatch_maps(idx, E, keep=None):
    """Expert-contiguous permutation of the T*K (token, slot) pairs.

    counts[e]  = number of pairs routed to expert e
    offsets    = exclusive prefix sum of counts (E+1 entries)
    dst_row[t,k] = offsets[e] + #{t' < t : e selected by t'}   (e = idx[t,k])
    src_token[r], src_slot[r]: the inverse map.
    With keep (capacity_keep), only the kept pairs are counted and placed;
    dropped pairs get dst_row = -1.
    Built the plainest way: expert by expert, tokens ascending.
    """
    idx = np.asarray(idx, np.int64)
    T, K = idx.shape
    if keep is None:
        keep = np.ones((T, K), bool)
    keep = np.asarray(keep, bool)
    counts = np.array([np.count_nonzero((idx == e) & keep) for e in range(E)], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    dst_row = np.full((T, K), -1, dtype=np.int64)
    src_token = np.full(T * K, -1, dtype=np.int64)
    src_slot = np.full(T * K, -1, dtype=np.int64)
    for e in range(E):
        t_list, k_list = np.nonzero((idx == e) & keep)  # row-major: ascending token
        rows = offsets[e] + np.arange(t_list.size)
        dst_row[t_list, k_list] = rows
        src_token[rows] = t_list
        src_slot[rows] = k_list
    return counts, offsets, dst_row, src_token, src_slot


def expert_capacity(T, K, E, capacity_factor, min_capacity=0):
    """Slots an expert may take: floor(capacity_factor * T * K / E), at least
    min_capacity (skill page, "Capacity Factor Tuning": expert_capacity =
    int(tokens / num_experts * capacity_factor), counted in (token, slot)
    pairs for top-K routing; the DeepSpeed config there also names
    min_capacity)."""
    return max(int(min_capacity), int(math.floor(capacity_factor * T * K / E)))


def capacity_keep(idx, E, capacity):
    """keep[t, k]: whether slot (t, k) is within its expert's capacity -- the
    expert keeps its first `capacity` slots in ascending token order and drops
    the rest ("drop_tokens": tokens exceeding capacity are dropped).  Built the
    plainest way: walk the tokens in order with one counter per expert."""
    idx = np.asarray(idx, np.int64)
    T, K = idx.shape
    seen = np.zeros(E, np.int64)
    keep = np.zeros((T, K), bool)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            keep[t, k] = seen[e] < capacity
            seen[e] += 1
    return keep


def permute_rows(x, src_token):
    """x_perm[r] = x[src_token[r]]: token rows in expert-contiguous order."""
    return np.asarray(x)[np.asarray(src_token, np.int64)]


def unpermute_combine(y_perm, dst_row, weights=None):
    """y[t] = sum_k w[t,k] * y_perm[dst_row[t,k]] (w = 1 when None), in float64
    (review §2.1 "Combine"; skill page's index_add_ accumulation)."""
    y_perm = np.asarray(y_perm, np.float64)
    dst_row = np.asarray(dst_row, np.int64)
    T, K = dst_row.shape
    y = np.zeros((T, y_perm.shape[1]), np.float64)
    for k in range(K):
        g = y_perm[dst_row[:, k]]
        if weights is not None:
            g = g * np.asarray(weights, np.float64)[:, k:k + 1]
        y += g
    return y


# ---------------------------------------------------------------------------
# Expert compute
# ---------------------------------------------------------------------------

def gelu(z):
    """Exact GELU, 0.5 z (1 + erf(z / sqrt 2)) (nn.GELU() default)."""
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def gelu_grad(z):
    z = np.asarray(z, np.float64)
    return 0.5 * (1.0 + _erf(z / math.sqrt(2.0))) + z * np.exp(-0.5 * z * z) / math.sqrt(2.0 * math.pi)


def silu(z):
    z = np.asarray(z, np.float64)
    return z * sigmoid(z)


def silu_grad(z):
    s = sigmoid(z)
    return s * (1.0 + np.asarray(z, np.float64) * (1.0 - s))


def _f64(a):
    return None if a is None else np.asarray(a, np.float64)


def expert_hidden(xr, w1e, b1e, act):
    """Pre-activation H = x W1^T (+ b1) and activation z for one expert.
    SwiGLU: W1 rows [0, F) are the gate, [F, 2F) the up projection,
    z = silu(gate) * up.  GELU: z = GELU(x W1^T + b1)."""
    xr = np.asarray(xr, np.float64)
    w1e = np.asarray(w1e, np.float64)
    H = xr @ w1e.T
    if b1e is not None:
        H = H + np.asarray(b1e, np.float64)[None, :]
    if act == ACT_SWIGLU:
        F = w1e.shape[0] // 2
        z = silu(H[:, :F]) * H[:, F:]
    else:
        z = gelu(H)
    return H, z


def expert_ffn(xr, w1e, w2e, act, b1e=None, b2e=None):
    """E_e(x) = W2 phi(W1 x + b1) + b2 (GELU) or W2 (silu(g) * u) (SwiGLU)."""
    _, z = expert_hidden(xr, w1e, b1e, act)
    out = z @ np.asarray(w2e, np.float64).T
    if b2e is not None:
        out = out + np.asarray(b2e, np.float64)[None, :]
    return out


def _bias_row(b, e):
    return None if b is None else b[e]


# ---------------------------------------------------------------------------
# Layer
# ---------------------------------------------------------------------------

def layer_fwd(x, w_r, w1, w2, K, score, act, *, b1=None, b2=None, sel_bias=None,
              gate_bias=None, renorm=True, force_balance=False, w1_shared=None, w2_shared=None,
              logits_dtype=np.float32, tokens=None, routing=None, capacity=None):
    """The MoE layer output y[t] = sum_k p[t,k] E_{idx[t,k]}(x_t) + S(x_t),
    float64 (review §1.1 MoE(x); §2.1 the four stages).  With a capacity,
    the sum runs over the kept slots only (capacity_keep); the kept weights
    are not renormalised.

    Expert outputs are computed expert by expert over the permuted rows
    (Dispatch, then one FFN per expert, then Combine).  ``tokens`` restricts
    the expert compute and output to a subset of token indices (routing is
    still decided for every token); ``routing`` may pass a precomputed
    (logits, idx, probs).  Returns a dict of the intermediate results.
    """
    x = np.asarray(x)
    T, h = x.shape
    E = np.asarray(w_r).shape[0]
    if routing is None:
        logits = gating_logits(x, w_r, gate_bias, logits_dtype)
        idx, probs = route(logits, K, score, renorm, sel_bias, force_balance)
    else:
        logits, idx, probs = routing
    keep = None if capacity is None else capacity_keep(idx, E, capacity)
    counts, offsets, dst_row, src_token, src_slot = dispatch_maps(idx, E, keep)
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, np.int64)
    want = np.zeros(T, bool)
    want[tokens] = True
    y = np.zeros((T, h), np.float64)
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        rows = rows[want[src_token[rows]]]
        if rows.size == 0:
            continue
        t_r = src_token[rows]
        out = expert_ffn(x[t_r], w1[e], w2[e], act, _bias_row(b1, e), _bias_row(b2, e))
        p = probs[t_r, src_slot[rows]][:, None]
        np.add.at(y, t_r, p * out)
    if w1_shared is not None:
        y[tokens] += expert_ffn(x[tokens], w1_shared, w2_shared, act)
    return dict(logits=logits, idx=idx, probs=probs, counts=counts, offsets=offsets,
                dst_row=dst_row, src_token=src_token, src_slot=src_slot,
                y=y[tokens], tokens=tokens, keep=keep)


def layer_fwd_masked_dense(x, w_r, w1, w2, K, score, act, *, b1=None, b2=None,
                           sel_bias=None, gate_bias=None, renorm=True, force_balance=False,
                           w1_shared=None, w2_shared=None, logits_dtype=np.float32,
                           capacity=None):
    """Second formulation, no permutation: loop over the K slots and over the
    experts with a boolean mask and accumulate score * expert(x[mask]) (the
    skill page's MoELayer.forward loop).  A capacity is applied the other way
    round from capacity_keep: a slot's position inside its expert is the
    running count of the token-major routing mask (a cumulative sum), and the
    slot is kept when that position is below the capacity.  For small cases
    only."""
    x = np.asarray(x)
    T, h = x.shape
    E = np.asarray(w_r).shape[0]
    logits = gating_logits(x, w_r, gate_bias, logits_dtype)
    idx, probs = route(logits, K, score, renorm, sel_bias, force_balance)
    kept = np.ones((T, K), bool)
    if capacity is not None:
        onehot = np.zeros((T * K, E), np.int64)
        onehot[np.arange(T * K), np.asarray(idx, np.int64).reshape(-1)] = 1
        position = (np.cumsum(onehot, axis=0) - onehot)[np.arange(T * K), idx.reshape(-1)]
        kept = (position < capacity).reshape(T, K)
    y = np.zeros((T, h), np.float64)
    for k in range(K):
        for e in range(E):
            mask = (idx[:, k] == e) & kept[:, k]
            if not mask.any():
                continue
            out = expert_ffn(x[mask], w1[e], w2[e], act, _bias_row(b1, e), _bias_row(b2, e))
            y[mask] += probs[mask, k][:, None] * out
    if w1_shared is not None:
        y += expert_ffn(x, w1_shared, w2_shared, act)
    return y


def layer_fwd_prob_before_fc2(x, w1, w2, idx, probs, act):
    """Memory-efficient permutation order (review §4.1.1): the routing weight
    scales the activation before the second linear layer,
    y = sum_i W2^(i) (p_i phi(W1^(i) x)).  Bias-free experts only."""
    x = np.asarray(x, np.float64)
    T, h = x.shape
    y = np.zeros((T, h), np.float64)
    for t in range(T):
        for k in range(idx.shape[1]):
            e = int(idx[t, k])
            _, z = expert_hidden(x[t:t + 1], w1[e], None, act)
            y[t] += ((probs[t, k] * z) @ np.asarray(w2[e], np.float64).T)[0]
    return y


# ---------------------------------------------------------------------------
# Backward (training configuration).  Plain reverse mode of layer_fwd with the
# selection held fixed.
# ---------------------------------------------------------------------------

def router_grad_logits(logits, idx, probs, dprob, score, renorm=True):
    """dL/dl [T, E] from dL/dp [T, K] through the scoring and normalisation.

    Softmax + renorm:  dl_k = p_k (dp_k - sum_j p_j dp_j) on the selected k.
    Softmax, full:     dl_i = [i sel] p_i dp_i - P_i sum_k p_k dp_k, P the full softmax.
    Sigmoid + renorm:  dl_k = s_k (1 - s_k) (dp_k - sum_j p_j dp_j) / S_sel.
    Sigmoid, all-E:    dl_i = s_i (1 - s_i) ([i sel] dp_i - sum_k p_k dp_k) / S_all.
    """
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    idx = np.asarray(idx, np.int64)
    dprob = np.asarray(dprob, np.float64)
    probs = np.asarray(probs, np.float64)
    rows = np.arange(T)[:, None]
    dl = np.zeros((T, E), np.float64)
    pdp = (probs * dprob).sum(axis=1, keepdims=True)
    if score == SCORE_SOFTMAX:
        if renorm:
            dl[rows, idx] = probs * (dprob - pdp)
        else:
            m = l.max(axis=1, keepdims=True)
            P = np.exp(l - m)
            P = P / P.sum(axis=1, keepdims=True)
            dl = -P * pdp
            dl[rows, idx] += probs * dprob
        return dl
    s = sigmoid(l)
    ds = np.zeros((T, E), np.float64)
    if renorm:
        S = np.take_along_axis(s, idx, axis=1).sum(axis=1, keepdims=True)
        ds[rows, idx] = (dprob - pdp) / S
    else:
        S = s.sum(axis=1, keepdims=True)
        ds = -np.broadcast_to(pdp / S, (T, E)).copy()
        ds[rows, idx] += dprob / S
    return ds * s * (1.0 - s)


def layer_bwd(x, w_r, w1, w2, dy, K, score, act, *, b1=None, b2=None, sel_bias=None,
              gate_bias=None, renorm=True, force_balance=False, w1_shared=None, w2_shared=None,
              logits_dtype=np.float32, routing=None, weight_grads=True, aux_coeff=0.0,
              z_coeff=0.0, capacity=None):
    """Gradients of sum(dy * y) + aux_coeff * aux + z_coeff * z (the two
    load-balancing losses below) for the layer: returns a dict with dx [T,h],
    dw_r [E,h], dw1, dw2 (and db1, db2 when biased), dw1_shared, dw2_shared,
    dprob [T,K] and dlogits [T,E].  Experts with no tokens get zero gradient.
    The selection bias gets none (it only selects); the gate bias gets
    db_r = sum_t dl_t.  weight_grads=False skips the expert weight gradients
    (dx, dprob and the router gradients only), for large expert counts."""
    x64 = np.asarray(x, np.float64)
    dy = np.asarray(dy, np.float64)
    T, h = x64.shape
    E = np.asarray(w_r).shape[0]
    if routing is None:
        logits = gating_logits(x, w_r, gate_bias, logits_dtype)
        idx, probs = route(logits, K, score, renorm, sel_bias, force_balance)
    else:
        logits, idx, probs = routing
    keep = None if capacity is None else capacity_keep(idx, E, capacity)
    counts, offsets, dst_row, src_token, src_slot = dispatch_maps(idx, E, keep)
    dx = np.zeros((T, h), np.float64)
    dprob = np.zeros(idx.shape, np.float64)
    dw1 = dw2 = None
    if weight_grads:
        dw1 = np.zeros((E,) + np.asarray(w1[0]).shape, np.float64)
        dw2 = np.zeros((E,) + np.asarray(w2[0]).shape, np.float64)
    db1 = None if b1 is None else np.zeros(np.asarray(b1).shape, np.float64)
    db2 = None if b2 is None else np.zeros(np.asarray(b2).shape, np.float64)
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        t_r = src_token[rows]
        k_r = src_slot[rows]
        xr = x64[t_r]
        w1e = np.asarray(w1[e], np.float64)
        w2e = np.asarray(w2[e], np.float64)
        H, z = expert_hidden(xr, w1e, _bias_row(b1, e), act)
        out = z @ w2e.T
        if b2 is not None:
            out = out + np.asarray(b2[e], np.float64)[None, :]
        p = probs[t_r, k_r][:, None]
        dyr = dy[t_r]
        dprob[t_r, k_r] = (dyr * out).sum(axis=1)
        dout = p * dyr
        if weight_grads:
            dw2[e] = dout.T @ z
        if db2 is not None:
            db2[e] = dout.sum(axis=0)
        dz = dout @ w2e
        if act == ACT_SWIGLU:
            F = w1e.shape[0] // 2
            g, u = H[:, :F], H[:, F:]
            dH = np.concatenate([dz * u * silu_grad(g), dz * silu(g)], axis=1)
        else:
            dH = dz * gelu_grad(H)
        if weight_grads:
            dw1[e] = dH.T @ xr
        if db1 is not None:
            db1[e] = dH.sum(axis=0)
        np.add.at(dx, t_r, dH @ w1e)
    dw1_s = dw2_s = None
    if w1_shared is not None:
        w1s = np.asarray(w1_shared, np.float64)
        w2s = np.asarray(w2_shared, np.float64)
        H, z = expert_hidden(x64, w1s, None, act)
        dw2_s = dy.T @ z if weight_grads else None
        dz = dy @ w2s
        F = w1s.shape[0] // 2
        g, u = H[:, :F], H[:, F:]
        dH = np.concatenate([dz * u * silu_grad(g), dz * silu(g)], axis=1)
        dw1_s = dH.T @ x64 if weight_grads else None
        dx += dH @ w1s
    dl = router_grad_logits(logits, idx, probs, dprob, score, renorm)
    if aux_coeff:
        dl = dl + aux_coeff * aux_loss_grad(logits, idx)
    if z_coeff:
        dl = dl + z_coeff * z_loss_grad(logits)
    dw_r = dl.T @ x64
    dx += dl @ np.asarray(w_r, np.float64)
    return dict(dx=dx, dw_r=dw_r, db_r=dl.sum(axis=0), dw1=dw1, dw2=dw2, db1=db1, db2=db2,
                dw1_shared=dw1_s, dw2_shared=dw2_s, dprob=dprob, dlogits=dl,
                idx=idx, probs=probs, logits=logits)


def grouped_mlp_bwd(x_perm, offsets, prob_perm, w1, w2, dy_perm):
    """Backward of the bias-free SwiGLU expert FFNs over permuted rows (the
    grouped-GEMM part of layer_bwd, written per expert on its own rows):
    returns dx_perm [P,h], dw1 [E,2F,h], dw2 [E,h,F] and dprob_perm [P] with
    dprob_perm[r] = <dy_perm[r], E_e(x_perm[r])>."""
    x_perm = np.asarray(x_perm, np.float64)
    dy_perm = np.asarray(dy_perm, np.float64)
    prob_perm = np.asarray(prob_perm, np.float64)
    E = len(offsets) - 1
    dx = np.zeros_like(x_perm)
    dprob = np.zeros(x_perm.shape[0])
    dw1 = np.zeros((E,) + np.asarray(w1[0]).shape)
    dw2 = np.zeros((E,) + np.asarray(w2[0]).shape)
    for e in range(E):
        r = slice(int(offsets[e]), int(offsets[e + 1]))
        if offsets[e + 1] == offsets[e]:
            continue
        w1e = np.asarray(w1[e], np.float64)
        w2e = np.asarray(w2[e], np.float64)
        H, z = expert_hidden(x_perm[r], w1e, None, ACT_SWIGLU)
        dprob[r] = (dy_perm[r] * (z @ w2e.T)).sum(axis=1)
        dout = prob_perm[r, None] * dy_perm[r]
        dw2[e] = dout.T @ z
        dz = dout @ w2e
        F = w1e.shape[0] // 2
        g, u = H[:, :F], H[:, F:]
        dH = np.concatenate([dz * u * silu_grad(g), dz * silu(g)], axis=1)
        dw1[e] = dH.T @ x_perm[r]
        dx[r] = dH @ w1e
    return dict(dx_perm=dx, dw1=dw1, dw2=dw2, dprob_perm=dprob)


# ---------------------------------------------------------------------------
# Load-balancing losses.  Skill page "emerging-techniques-moe-training",
# "Load Balancing": "Auxiliary Loss" (the fraction of routed slots per expert
# times the expert's mean gate probability, summed and scaled by the number of
# experts) and "Router Z-Loss" (mean squared log-sum-exp of the gate logits);
# the review page's training configuration sets the aux-loss coefficient to
# 1e-3.  The gate probabilities of the auxiliary loss are the full softmax of
# the gate logits whatever the scoring function (the page's code applies
# softmax to the logits).  The slot fractions are counts of a discrete
# selection: they carry no gradient.
# ---------------------------------------------------------------------------

def softmax_full(logits):
    """Row-wise softmax over all E experts, float64."""
    l = np.asarray(logits, np.float64)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def logsumexp_rows(logits):
    """log sum_e exp(l_te) per token, float64 (max-shifted)."""
    l = np.asarray(logits, np.float64)
    m = l.max(axis=1)
    return m + np.log(np.exp(l - m[:, None]).sum(axis=1))


def slot_fractions(idx, E):
    """f_e = (number of (t, k) slots routed to e) / (T * K)."""
    idx = np.asarray(idx, np.int64)
    return np.bincount(idx.ravel(), minlength=E).astype(np.float64) / idx.size


def aux_loss(logits, idx):
    """aux = E * sum_e f_e P_e with f the slot fractions of the selection idx
    and P_e = mean over tokens of softmax(l_t)_e."""
    l = np.asarray(logits, np.float64)
    E = l.shape[1]
    f = slot_fractions(idx, E)
    P = softmax_full(l).mean(axis=0)
    return float(E * (f * P).sum())


def z_loss(logits):
    """z = mean over tokens of (log sum_e exp l_te)^2."""
    return float((logsumexp_rows(logits) ** 2).mean())


def aux_loss_grad(logits, idx):
    """d aux / d l [T, E] with f held fixed: with s_t = softmax(l_t),
    (E / T) s_tj (f_j - sum_e f_e s_te)."""
    l = np.asarray(logits, np.float64)
    T, E = l.shape
    f = slot_fractions(idx, E)
    s = softmax_full(l)
    g = s @ f
    return (E / T) * s * (f[None, :] - g[:, None])


def z_loss_grad(logits):
    """d z / d l [T, E] = (2 / T) lse_t softmax(l_t)_j."""
    l = np.asarray(logits, np.float64)
    T = l.shape[0]
    return (2.0 / T) * logsumexp_rows(l)[:, None] * softmax_full(l)


# ---------------------------------------------------------------------------
# Work accounting (closed forms used by the benchmark's roofline figures)
# ---------------------------------------------------------------------------

def expert_param_count(h, F, act, bias=False):
    """Parameters of one expert: a bias-free SwiGLU expert holds three h x F
    matrices ("Calculation of activated parameters"); a GELU expert two, plus
    F + h biases when biased."""
    if act == ACT_SWIGLU:
        return 3 * h * F
    return 2 * h * F + ((F + h) if bias else 0)


def routed_flops(T, K, h, F, act):
    """Multiply-add FLOPs of the routed expert GEMMs (2 per MAC)."""
    return 2 * T * K * (3 if act == ACT_SWIGLU else 2) * h * F
