"""Pins for the oracle's backward: central finite differences in float64 on
tiny problems (selection held away from ties), and the one-expert identity
(the router weight gets exactly zero gradient)."""

import numpy as np
import pytest

from oracle import moe_oracle as O


def _problem(seed, score, act, bias, shared, T=9, h=6, E=4, K=2, F=5):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, h))
    w_r = rng.normal(size=(E, h)) * 0.7
    rows = 2 * F if act == O.ACT_SWIGLU else F
    w1 = rng.normal(size=(E, rows, h)) / np.sqrt(h)
    w2 = rng.normal(size=(E, h, F)) / np.sqrt(F)
    kw = {}
    if bias:
        kw["b1"] = rng.normal(size=(E, rows)) * 0.3
        kw["b2"] = rng.normal(size=(E, h)) * 0.3
    if shared:
        kw["w1_shared"] = rng.normal(size=(rows, h)) / np.sqrt(h)
        kw["w2_shared"] = rng.normal(size=(h, F)) / np.sqrt(F)
    kw["gate_bias"] = rng.normal(size=E) * 0.2
    dy = rng.normal(size=(T, h))
    return x, w_r, w1, w2, dy, kw


def _loss(x, w_r, w1, w2, dy, K, score, act, kw, renorm):
    y = O.layer_fwd(x, w_r, w1, w2, K, score, act, renorm=renorm, logits_dtype=np.float64, **kw)
    return float((dy * y["y"]).sum()), y["idx"]


CASES = [
    (O.SCORE_SOFTMAX, O.ACT_GELU, True, False, True),
    (O.SCORE_SOFTMAX, O.ACT_SWIGLU, False, True, False),
    (O.SCORE_SIGMOID, O.ACT_SWIGLU, False, True, True),
    (O.SCORE_SIGMOID, O.ACT_GELU, True, False, False),
]


@pytest.mark.parametrize("score,act,bias,shared,renorm", CASES)
def test_gradients_match_central_differences(score, act, bias, shared, renorm):
    K = 2
    x, w_r, w1, w2, dy, kw = _problem(20 + score * 2 + act, score, act, bias, shared)
    g = O.layer_bwd(x, w_r, w1, w2, dy, K, score, act, renorm=renorm, logits_dtype=np.float64, **kw)
    _, idx0 = _loss(x, w_r, w1, w2, dy, K, score, act, kw, renorm)
    eps = 1e-6

    def check(arr, grad, name, n=12):
        rng = np.random.default_rng(hash(name) % 2**32)
        flat = arr.reshape(-1)
        for j in rng.choice(flat.size, size=min(n, flat.size), replace=False):
            old = flat[j]
            flat[j] = old + eps
            lp, ip = _loss(x, w_r, w1, w2, dy, K, score, act, kw, renorm)
            flat[j] = old - eps
            lm, im = _loss(x, w_r, w1, w2, dy, K, score, act, kw, renorm)
            flat[j] = old
            assert (ip == idx0).all() and (im == idx0).all(), "selection moved: pick another seed"
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad.reshape(-1)[j]) <= 1e-6 * max(1.0, abs(fd)), (name, j, fd, grad.reshape(-1)[j])

    check(x, g["dx"], "x")
    check(w_r, g["dw_r"], "w_r")
    check(w1, g["dw1"], "w1")
    check(w2, g["dw2"], "w2")
    check(kw["gate_bias"], g["db_r"], "gate_bias")
    if bias:
        check(kw["b1"], g["db1"], "b1")
        check(kw["b2"], g["db2"], "b2")
    if shared:
        check(kw["w1_shared"], g["dw1_shared"], "w1s")
        check(kw["w2_shared"], g["dw2_shared"], "w2s")


def test_dprob_is_inner_product_with_expert_output():
    x, w_r, w1, w2, dy, kw = _problem(31, O.SCORE_SOFTMAX, O.ACT_SWIGLU, False, False)
    g = O.layer_bwd(x, w_r, w1, w2, dy, 2, O.SCORE_SOFTMAX, O.ACT_SWIGLU, logits_dtype=np.float64, **kw)
    for t in range(x.shape[0]):
        for k in range(2):
            e = g["idx"][t, k]
            out = O.expert_ffn(x[t:t + 1], w1[e], w2[e], O.ACT_SWIGLU)[0]
            assert g["dprob"][t, k] == pytest.approx(float(dy[t] @ out), rel=1e-12)


def test_single_expert_router_gets_zero_gradient():
    # "Keep the Dense reference baseline": with one expert the router weight
    # cannot receive a gradient (softmax over one logit is constantly 1).
    x, w_r, w1, w2, dy, kw = _problem(32, O.SCORE_SOFTMAX, O.ACT_SWIGLU, False, False, E=1)
    kw.pop("gate_bias")
    g = O.layer_bwd(x, w_r, w1, w2, dy, 1, O.SCORE_SOFTMAX, O.ACT_SWIGLU, **kw)
    assert (g["dw_r"] == 0).all()
    assert (g["dlogits"] == 0).all()


def test_unused_expert_gets_zero_gradient():
    x, w_r, w1, w2, dy, kw = _problem(33, O.SCORE_SOFTMAX, O.ACT_SWIGLU, False, False, E=4, K=1)
    kw["gate_bias"] = np.array([0.0, 0.0, 0.0, -1e9])  # expert 3 never selected
    g = O.layer_bwd(x, w_r, w1, w2, dy, 1, O.SCORE_SOFTMAX, O.ACT_SWIGLU, logits_dtype=np.float64, **kw)
    assert (g["dw1"][3] == 0).all() and (g["dw2"][3] == 0).all()


def test_grouped_mlp_bwd_matches_layer_bwd():
    # the permuted-row expert backward agrees with the layer backward's expert
    # gradients, its dprob and (un-permuted) its dx contribution
    x, w_r, w1, w2, dy, kw = _problem(34, O.SCORE_SIGMOID, O.ACT_SWIGLU, False, False, T=15, E=5, K=3)
    full = O.layer_bwd(x, w_r, w1, w2, dy, 3, O.SCORE_SIGMOID, O.ACT_SWIGLU, logits_dtype=np.float64, **kw)
    idx, probs = full["idx"], full["probs"]
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(idx, 5)
    g = O.grouped_mlp_bwd(x[src_token], offsets, probs[src_token, src_slot], w1, w2, dy[src_token])
    np.testing.assert_allclose(g["dw1"], full["dw1"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dw2"], full["dw2"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["dprob_perm"][dst_row], full["dprob"], rtol=1e-12, atol=1e-13)
    routed_dx = O.unpermute_combine(g["dx_perm"], dst_row)
    np.testing.assert_allclose(routed_dx + full["dlogits"] @ w_r, full["dx"], rtol=1e-11, atol=1e-12)
