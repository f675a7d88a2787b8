"""Pins for the oracle's Route stage (gating, scoring, top-k, renormalisation)
against brute force, hand-worked values, exact sums and library routines."""

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_topk(keys_row, K):
    """The unique K-subset S with every member beating every non-member
    (higher key, or equal key and lower index), listed by (-key, index)."""
    E = len(keys_row)
    found = []
    for S in itertools.combinations(range(E), K):
        inside = set(S)
        ok = all((keys_row[i] > keys_row[j]) or (keys_row[i] == keys_row[j] and i < j)
                 for i in inside for j in range(E) if j not in inside)
        if ok:
            found.append(S)
    assert len(found) == 1
    return sorted(found[0], key=lambda i: (-keys_row[i], i))


@pytest.mark.parametrize("E", [1, 2, 3, 5, 6])
def test_topk_matches_brute_force_with_ties(E):
    rng = np.random.default_rng(E)
    for K in range(1, E + 1):
        keys = rng.integers(-2, 3, size=(40, E)).astype(np.float32)  # many ties
        idx = O.select_topk(keys, K)
        for t in range(keys.shape[0]):
            assert list(idx[t]) == _brute_topk(list(keys[t]), K)


def test_router_golden_hand_examples():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "router_4tok.txt"))
             if l.strip() and not l.startswith("#")]
    for f in lines:
        score = O.SCORE_SOFTMAX if f[0] == "softmax" else O.SCORE_SIGMOID
        K = int(f[1])
        l = np.array([[float(v) for v in f[2:6]]], np.float32)
        b = np.array([float(v) for v in f[6:10]], np.float32)
        idx, p = O.route(l, K, score, renorm=True, sel_bias=b if b.any() else None)
        want_idx = [int(v) for v in f[10:12] if v != "-"][:K]
        want_p = [float(v) for v in f[12:14] if v != "-"][:K]
        assert list(idx[0]) == want_idx, f
        np.testing.assert_allclose(p[0], want_p, rtol=0, atol=1e-7)


def test_renormalised_probs_sum_to_one():
    rng = np.random.default_rng(1)
    l = rng.normal(size=(200, 16)).astype(np.float32)
    for score in (O.SCORE_SOFTMAX, O.SCORE_SIGMOID):
        _, p = O.route(l, 4, score, renorm=True)
        np.testing.assert_allclose(p.sum(1), 1.0, rtol=0, atol=1e-15)
        assert (p > 0).all()


def test_top1_is_argmax():
    # skill page "Top-1 Routing (Switch Transformer)": argmax of the logits;
    # np.argmax returns the first (lowest) index among equal maxima.
    rng = np.random.default_rng(2)
    l = rng.integers(-3, 4, size=(500, 7)).astype(np.float32)
    idx, p = O.route(l, 1, O.SCORE_SOFTMAX)
    assert (idx[:, 0] == np.argmax(l, axis=1)).all()
    assert (p == 1.0).all()


def test_softmax_against_library():
    rng = np.random.default_rng(3)
    l = rng.normal(size=(64, 12)).astype(np.float32)
    idx, p_full = O.route(l, 3, O.SCORE_SOFTMAX, renorm=False)
    ref = np.take_along_axis(sp_softmax(l.astype(np.float64), axis=1), idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(p_full, ref, rtol=1e-13, atol=0)
    # renormalised: the skill page's softmax -> torch.topk -> divide by the sum
    lt = torch.from_numpy(l.astype(np.float64))
    s = torch.softmax(lt, dim=-1)
    ts, ti = torch.topk(s, 3, dim=-1)
    ts = ts / ts.sum(dim=-1, keepdim=True)
    idx_r, p_r = O.route(l, 3, O.SCORE_SOFTMAX, renorm=True)
    assert (ti.numpy() == idx_r).all()  # random normals: no ties
    np.testing.assert_allclose(p_r, ts.numpy(), rtol=1e-13, atol=0)


def test_sigmoid_against_library():
    rng = np.random.default_rng(4)
    l = rng.normal(size=(64, 10)).astype(np.float32)
    b = (0.1 * rng.normal(size=10)).astype(np.float32)
    idx, p = O.route(l, 4, O.SCORE_SIGMOID, renorm=True, sel_bias=b)
    s = torch.sigmoid(torch.from_numpy(l.astype(np.float64)))
    keys = s.float() + torch.from_numpy(b)
    _, ti = torch.topk(keys, 4, dim=-1)
    assert (ti.numpy() == idx).all()
    sel = torch.gather(s, 1, torch.from_numpy(idx.astype(np.int64)))
    np.testing.assert_allclose(p, (sel / sel.sum(-1, keepdim=True)).numpy(), rtol=1e-13)
    # all-E normalisation (the page's formula) when not renormalising
    _, p_all = O.route(l, 4, O.SCORE_SIGMOID, renorm=False, sel_bias=b)
    np.testing.assert_allclose(p_all, (sel / s.sum(-1, keepdim=True)).numpy(), rtol=1e-13)
    # the selection bias never enters p
    _, p_nb = O.route(l, 4, O.SCORE_SIGMOID, renorm=True)
    idx_nb = O.select_topk(O.selection_keys(l, O.SCORE_SIGMOID), 4)
    same = (np.sort(idx_nb, 1) == np.sort(idx, 1)).all(1)
    np.testing.assert_allclose(p_nb[same].sum(1), 1.0)


def test_force_balanced_exact_counts():
    for T, K, E in [(2048, 8, 64), (96, 8, 256), (12, 4, 6)]:
        if (T * K) % E:
            continue
        idx = O.force_balanced_topk(T, K, E)
        counts = np.bincount(idx.ravel(), minlength=E)
        assert (counts == T * K // E).all()
        assert all(len(set(r)) == K for r in idx.tolist())


def test_gating_logits_correctly_rounded():
    # Products of fp32/bf16 values are exact in float64; math.fsum gives the
    # exactly rounded sum.  The oracle's fp32 logit must be that value (up to
    # one ulp in the rare double-rounding case).
    rng = np.random.default_rng(5)
    x = rng.normal(size=(16, 300)).astype(np.float32)
    w = (0.02 * rng.normal(size=(6, 300))).astype(np.float32)
    b = rng.normal(size=6).astype(np.float32)
    l = O.gating_logits(x, w, gate_bias=b)
    exact = np.array([[np.float32(math.fsum([float(a) * float(c) for a, c in zip(x[t], w[e])] + [float(b[e])]))
                       for e in range(6)] for t in range(16)])
    ulp = np.spacing(np.abs(exact))
    assert (np.abs(l - exact) <= ulp).all()
    assert (l == exact).mean() > 0.95


def test_gating_exact_small_integers():
    x = np.array([[1, 2, 3], [-1, 0, 4]], np.float32)
    w = np.array([[1, 1, 1], [0.5, -0.25, 2]], np.float32)
    want = [[Fraction(6), Fraction(1, 2) - Fraction(1, 2) + 6], [Fraction(3), Fraction(-1, 2) + 8]]
    assert O.gating_logits(x, w).tolist() == [[float(v) for v in r] for r in want]


def test_selection_margin():
    l = np.array([[3.0, 1.0, 0.5, 0.25]], np.float32)
    assert O.selection_margin(l, 2, O.SCORE_SOFTMAX)[0] == pytest.approx(0.5)
    assert np.isinf(O.selection_margin(l, 4, O.SCORE_SOFTMAX)[0])


def test_routing_map_rows():
    rng = np.random.default_rng(6)
    l = rng.normal(size=(50, 9)).astype(np.float32)
    idx, _ = O.route(l, 3, O.SCORE_SOFTMAX)
    m = O.routing_map(idx, 9)
    assert (m.sum(1) == 3).all()
    for t in range(50):
        assert set(np.nonzero(m[t])[0]) == set(idx[t])


def test_order_margin():
    l = np.array([[3.0, 1.0, 0.999, 0.25], [5.0, 4.0, 3.0, 2.0]], np.float32)
    om = O.order_margin(l, 2, O.SCORE_SOFTMAX)
    assert om[0] == pytest.approx(0.001, rel=1e-3) and om[1] == pytest.approx(1.0)
    assert np.isinf(O.order_margin(l[:, :1], 1, O.SCORE_SOFTMAX)).all()
