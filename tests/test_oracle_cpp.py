"""Pins of the C++ oracle (oracle/moe_oracle_ref.cpp, through
oracle/moe_oracle_c.py): the hand-worked golden router and dispatch cases,
brute-force top-K on tie-heavy keys, the layer invariants (identical experts
give the dense FFN; counts sum to T*K; the permutation is a bijection;
force-balanced counts are exactly T*K/E), and agreement with the numpy
oracle on the same seeded inputs, every configuration kind included."""

import itertools
import os

import numpy as np
import pytest

from mixture_experts_layer_softmax_gb300 import inputs
from oracle import moe_oracle as O
from oracle import moe_oracle_c as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _route_logits(l, K, score, sel_bias=None, renorm=True):
    """Routes given fp32 logits: one input feature equal to 1 and the logits
    as the router weight column, so l = W_r x reproduces them exactly."""
    l = np.asarray(l, np.float32)
    T, E = l.shape
    out = [C.route(np.ones((1, 1), np.float32), l[t][:, None], K, score, renorm, sel_bias)
           for t in range(T)]
    return (np.concatenate([o[0] for o in out]), np.concatenate([o[1] for o in out]),
            np.concatenate([o[2] for o in out]))


def test_router_golden_hand_examples():
    for f in (l.split() for l in open(os.path.join(GOLDEN, "router_4tok.txt"))
              if l.strip() and not l.startswith("#")):
        score = C.SCORE_SOFTMAX if f[0] == "softmax" else C.SCORE_SIGMOID
        K = int(f[1])
        l = np.array([[float(v) for v in f[2:6]]], np.float32)
        b = np.array([float(v) for v in f[6:10]], np.float32)
        lg, idx, p = _route_logits(l, K, score, b if b.any() else None)
        assert (lg == l).all()
        assert list(idx[0]) == [int(v) for v in f[10:12] if v != "-"][:K], f
        np.testing.assert_allclose(p[0], [float(v) for v in f[12:14] if v != "-"][:K],
                                   rtol=0, atol=1e-7)


def test_dispatch_golden_hand_example():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "dispatch_4tok.txt"))
            if l.strip() and not l.startswith("#")]
    get = lambda key: [list(map(int, r[1:])) for r in rows if r[0] == key]
    idx = np.array(get("idx"), np.int32)
    counts, offsets, dst_row, src_token, src_slot = C.dispatch_maps(idx, 3)
    assert counts.tolist() == get("counts")[0]
    assert offsets.tolist() == get("offsets")[0]
    assert dst_row.tolist() == get("dst")
    assert src_token.tolist() == get("src_token")[0]
    assert (idx[src_token, src_slot] == np.repeat(np.arange(3), counts)).all()


@pytest.mark.parametrize("E", [1, 2, 3, 5, 6])
def test_topk_matches_brute_force_with_ties(E):
    rng = np.random.default_rng(100 + E)
    for K in range(1, E + 1):
        l = rng.integers(-2, 3, size=(25, E)).astype(np.float32)  # many ties
        _, idx, _ = _route_logits(l, K, C.SCORE_SOFTMAX)
        for t in range(l.shape[0]):
            row = list(l[t])
            subsets = [S for S in itertools.combinations(range(E), K)
                       if all(row[i] > row[j] or (row[i] == row[j] and i < j)
                              for i in S for j in range(E) if j not in S)]
            assert len(subsets) == 1
            assert list(idx[t]) == sorted(subsets[0], key=lambda i: (-row[i], i))


def _weights(E, h, F, act, seed):
    R1 = 2 * F if act == C.ACT_SWIGLU else F
    w1 = inputs.normal((E, R1, h), h ** -0.5, seed, 5, "bf16")
    w2 = inputs.normal((E, h, F), F ** -0.5, seed, 7, "bf16")
    return w1, w2


CASES = [
    # T, h, E, K, F, act, score, renorm, sel_bias, gate_bias, shared, force, bias
    (256, 128, 8, 2, 512, C.ACT_GELU, C.SCORE_SOFTMAX, True, False, False, False, False, True),
    (97, 64, 16, 4, 48, C.ACT_SWIGLU, C.SCORE_SOFTMAX, False, False, True, False, False, False),
    (120, 96, 32, 8, 40, C.ACT_SWIGLU, C.SCORE_SIGMOID, True, True, False, True, False, False),
    (64, 32, 12, 3, 16, C.ACT_SWIGLU, C.SCORE_SIGMOID, False, False, False, False, False, False),
    (48, 32, 8, 4, 24, C.ACT_SWIGLU, C.SCORE_SOFTMAX, True, False, False, False, True, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}E{c[2]}K{c[3]}")
def test_agrees_with_numpy_oracle(case):
    T, h, E, K, F, act, score, renorm, sb, gb, shared, force, bias = case
    seed = T + E
    x = inputs.normal((T, h), 1.0, seed, 1, "bf16")
    w_r = inputs.normal((E, h), 0.5 * h ** -0.5, seed, 2)
    sel_bias = inputs.normal((E,), 0.1, seed, 4) if sb else None
    gate_bias = inputs.normal((E,), 0.5, seed, 3) if gb else None
    w1, w2 = _weights(E, h, F, act, seed)
    R1 = w1.shape[1]
    b1 = inputs.normal((E, R1), h ** -0.5, seed, 6) if bias else None
    b2 = inputs.normal((E, h), F ** -0.5, seed, 8) if bias else None
    w1s = inputs.normal((2 * F, h), h ** -0.5, seed, 9, "bf16") if shared else None
    w2s = inputs.normal((h, F), F ** -0.5, seed, 10, "bf16") if shared else None
    lg, idx, p = C.route(x, w_r, K, score, renorm, sel_bias, gate_bias, force)
    ref_l = O.gating_logits(x, w_r, gate_bias)
    # both round a double sum to fp32: equal, or one fp32 step apart where the
    # double sums straddle a rounding boundary
    ulp = np.abs(lg.view(np.int32).astype(np.int64) - ref_l.view(np.int32).astype(np.int64))
    assert ulp.max() <= 1
    ref_idx, ref_p = O.route(ref_l, K, score, renorm, sel_bias, force)
    _, idx_on_ref, p_on_ref = _route_logits(ref_l, K, score, sel_bias, renorm) if not force else \
        (None, idx, p)
    if (ulp == 0).all():
        np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_array_equal(idx_on_ref, ref_idx)
    if not force:
        np.testing.assert_allclose(p_on_ref, ref_p, rtol=1e-13, atol=0)
    maps, ref_maps = C.dispatch_maps(ref_idx, E), O.dispatch_maps(ref_idx, E)
    for a, b in zip(maps, ref_maps):
        np.testing.assert_array_equal(a, b)
    y = C.layer_fwd(x, ref_idx, ref_p, w1, w2, act, b1=b1, b2=b2, w1_shared=w1s, w2_shared=w2s)
    y_ref = O.layer_fwd(x, w_r, w1, w2, K, score, act, b1=b1, b2=b2, w1_shared=w1s,
                        w2_shared=w2s, routing=(ref_l, ref_idx, ref_p))["y"]
    assert np.abs(y - y_ref).max() <= 1e-12 * np.abs(y_ref).max()
    toks = np.array([T - 1, 0, T // 2])
    y_sub = C.layer_fwd(x, ref_idx, ref_p, {e: w1[e] for e in np.unique(ref_idx[toks])},
                        {e: w2[e] for e in np.unique(ref_idx[toks])}, act, b1=b1, b2=b2,
                        w1_shared=w1s, w2_shared=w2s, tokens=toks)
    np.testing.assert_array_equal(y_sub, y[toks])


def test_identical_experts_give_the_dense_ffn():
    T, h, E, K, F = 64, 48, 6, 3, 32
    x = inputs.normal((T, h), 1.0, 3, 1, "bf16")
    w_r = inputs.normal((E, h), 0.2, 3, 2)
    one1, one2 = _weights(1, h, F, C.ACT_SWIGLU, 3)
    w1, w2 = np.repeat(one1, E, 0), np.repeat(one2, E, 0)
    _, idx, p = C.route(x, w_r, K, C.SCORE_SOFTMAX)
    y = C.layer_fwd(x, idx, p, w1, w2, C.ACT_SWIGLU)
    H = x.astype(np.float64) @ one1[0].astype(np.float64).T
    g, u = H[:, :F], H[:, F:]
    dense = (g / (1.0 + np.exp(-g)) * u) @ one2[0].astype(np.float64).T
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
    assert np.abs(y - dense).max() <= 1e-12 * np.abs(dense).max()


def test_maps_invariants_and_force_balance():
    T, E, K = 96, 12, 4
    _, idx, _ = C.route(inputs.normal((T, 8), 1.0, 5, 1), inputs.normal((E, 8), 1.0, 5, 2), K,
                        C.SCORE_SIGMOID)
    counts, offsets, dst_row, src_token, src_slot = C.dispatch_maps(idx, E)
    assert counts.sum() == T * K and offsets[-1] == T * K
    assert sorted(dst_row.ravel().tolist()) == list(range(T * K))          # a bijection
    assert (dst_row[src_token, src_slot] == np.arange(T * K)).all()       # inverse maps
    _, fb, _ = C.route(np.zeros((T, 8), np.float32), np.zeros((E, 8), np.float32), K,
                       C.SCORE_SOFTMAX, force_balance=True)
    assert (np.bincount(fb.ravel(), minlength=E) == T * K // E).all()
    with pytest.raises(ValueError):
        C.dispatch_maps(np.array([[E]], np.int32), E)
