"""Pins for the oracle's load-balancing losses (auxiliary loss and router
z-loss): hand-worked cases from tests/golden/load_balance_losses.txt
(including the single-expert case, whose load-balance loss the pages report as
exactly 1), closed forms for balanced and uniform routing, the zero row sum of
the auxiliary gradient, and central finite differences for both gradients and
for their path into the router weight gradient of the layer backward."""

import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "load_balance_losses.txt")


def _cases():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        head, logits, idx, losses, daux, dz = [p.strip() for p in line.split("|")]
        name, E, K, T = head.split()
        E, K, T = int(E), int(K), int(T)
        l = np.array([float(v) for v in logits.split()]).reshape(T, E)
        i = np.array([int(v) for v in idx.split()]).reshape(T, K)
        aux, z = (float(v) for v in losses.split())
        ga = None if daux == "-" else np.array([float(v) for v in daux.split()]).reshape(T, E)
        gz = None if dz == "-" else np.array([float(v) for v in dz.split()]).reshape(T, E)
        out.append((name, l, i, aux, z, ga, gz))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_hand_worked_losses(case):
    _, l, idx, aux, z, ga, gz = case
    assert O.aux_loss(l, idx) == pytest.approx(aux, rel=1e-14, abs=1e-15)
    assert O.z_loss(l) == pytest.approx(z, rel=1e-14)
    if ga is not None:
        np.testing.assert_allclose(O.aux_loss_grad(l, idx), ga, rtol=1e-14, atol=1e-15)
    if gz is not None:
        np.testing.assert_allclose(O.z_loss_grad(l), gz, rtol=1e-14)


@pytest.mark.parametrize("T,E,K", [(64, 8, 2), (96, 16, 4), (40, 5, 5)])
def test_balanced_uniform_routing_gives_one(T, E, K):
    # force-balanced routing with E | T*K: every f_e = 1/E; equal logits: P_e = 1/E
    idx = O.force_balanced_topk(T, K, E)
    l = np.full((T, E), 0.37)
    assert O.aux_loss(l, idx) == pytest.approx(1.0, rel=1e-14)
    # equal logits c: logsumexp = c + ln E
    assert O.z_loss(l) == pytest.approx((0.37 + np.log(E)) ** 2, rel=1e-14)


def test_single_expert_loss_is_one_for_any_logits():
    rng = np.random.default_rng(3)
    l = rng.normal(size=(50, 1)) * 3
    idx = np.zeros((50, 1), np.int32)
    assert O.aux_loss(l, idx) == 1.0
    np.testing.assert_allclose(O.aux_loss_grad(l, idx), 0.0, atol=0)
    np.testing.assert_allclose(O.z_loss(l), (l[:, 0] ** 2).mean(), rtol=1e-14)


def test_aux_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(4)
    l = rng.normal(size=(30, 7))
    idx = O.select_topk(l, 3)
    np.testing.assert_allclose(O.aux_loss_grad(l, idx).sum(axis=1), 0.0, atol=1e-15)


@pytest.mark.parametrize("seed,T,E,K", [(5, 12, 6, 2), (6, 7, 9, 3)])
def test_gradients_match_central_differences(seed, T, E, K):
    rng = np.random.default_rng(seed)
    l = rng.normal(size=(T, E)) * 1.5
    idx = O.select_topk(l, K)  # held fixed: the slot fractions carry no gradient
    ga, gz = O.aux_loss_grad(l, idx), O.z_loss_grad(l)
    eps = 1e-6
    for t in range(T):
        for j in range(E):
            lp, lm = l.copy(), l.copy()
            lp[t, j] += eps
            lm[t, j] -= eps
            fa = (O.aux_loss(lp, idx) - O.aux_loss(lm, idx)) / (2 * eps)
            fz = (O.z_loss(lp) - O.z_loss(lm)) / (2 * eps)
            assert fa == pytest.approx(ga[t, j], rel=1e-6, abs=1e-9)
            assert fz == pytest.approx(gz[t, j], rel=1e-6, abs=1e-9)


@pytest.mark.parametrize("score", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID])
def test_layer_backward_adds_the_loss_gradients_to_the_router(score):
    # d/dW_r of (a * aux + c * z) with the routing fixed, by central differences,
    # equals the change the two coefficients make to the layer's dW_r and db_r
    rng = np.random.default_rng(11)
    T, h, E, K, F = 10, 6, 5, 2, 4
    x = rng.normal(size=(T, h))
    w_r = rng.normal(size=(E, h)) * 0.6
    w1 = rng.normal(size=(E, 2 * F, h)) / np.sqrt(h)
    w2 = rng.normal(size=(E, h, F)) / np.sqrt(F)
    dy = rng.normal(size=(T, h))
    a, c = 0.3, 0.05
    kw = dict(logits_dtype=np.float64)
    g0 = O.layer_bwd(x, w_r, w1, w2, dy, K, score, O.ACT_SWIGLU, **kw)
    g1 = O.layer_bwd(x, w_r, w1, w2, dy, K, score, O.ACT_SWIGLU, aux_coeff=a, z_coeff=c, **kw)
    idx = g0["idx"]

    def extra(w):
        l = x @ w.T
        return a * O.aux_loss(l, idx) + c * O.z_loss(l)

    eps = 1e-6
    fd = np.zeros_like(w_r)
    for e in range(E):
        for j in range(h):
            wp, wm = w_r.copy(), w_r.copy()
            wp[e, j] += eps
            wm[e, j] -= eps
            fd[e, j] = (extra(wp) - extra(wm)) / (2 * eps)
    np.testing.assert_allclose(g1["dw_r"] - g0["dw_r"], fd, rtol=1e-6, atol=1e-9)
    dl_extra = a * O.aux_loss_grad(g0["logits"], idx) + c * O.z_loss_grad(g0["logits"])
    np.testing.assert_allclose(g1["db_r"] - g0["db_r"], dl_extra.sum(axis=0), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g1["dx"] - g0["dx"], dl_extra @ w_r, rtol=1e-10, atol=1e-13)
