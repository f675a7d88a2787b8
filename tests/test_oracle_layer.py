"""Pins for the oracle's layer forward: two independent formulations, the
dense-FFN special cases, the memory-efficient order, library activations and
the closed-form parameter count."""

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import moe_oracle as O


def _weights(rng, E, h, F, act, bias=False, scale=1.0):
    rows = 2 * F if act == O.ACT_SWIGLU else F
    w1 = rng.normal(size=(E, rows, h)) / np.sqrt(h) * scale
    w2 = rng.normal(size=(E, h, F)) / np.sqrt(F) * scale
    b1 = rng.normal(size=(E, rows)) / np.sqrt(h) if bias else None
    b2 = rng.normal(size=(E, h)) / np.sqrt(F) if bias else None
    return w1, w2, b1, b2


def _torch_ffn(x, w1, w2, act, b1=None, b2=None):
    """One expert with library ops in float64 (nn.functional linear/gelu/silu)."""
    xt = torch.from_numpy(np.asarray(x, np.float64))
    w1t, w2t = torch.from_numpy(w1), torch.from_numpy(w2)
    b1t = None if b1 is None else torch.from_numpy(b1)
    b2t = None if b2 is None else torch.from_numpy(b2)
    H = Fnn.linear(xt, w1t, b1t)
    if act == O.ACT_SWIGLU:
        F = w1.shape[0] // 2
        z = Fnn.silu(H[:, :F]) * H[:, F:]
    else:
        z = Fnn.gelu(H, approximate="none")
    return Fnn.linear(z, w2t, b2t).numpy()


@pytest.mark.parametrize("act,bias", [(O.ACT_GELU, True), (O.ACT_GELU, False), (O.ACT_SWIGLU, False)])
def test_expert_ffn_against_library(act, bias):
    rng = np.random.default_rng(10)
    w1, w2, b1, b2 = _weights(rng, 1, 24, 40, act, bias)
    x = rng.normal(size=(9, 24))
    got = O.expert_ffn(x, w1[0], w2[0], act, None if b1 is None else b1[0], None if b2 is None else b2[0])
    want = _torch_ffn(x, w1[0], w2[0], act, None if b1 is None else b1[0], None if b2 is None else b2[0])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("score,act,bias,shared,renorm", [
    (O.SCORE_SOFTMAX, O.ACT_GELU, True, False, True),
    (O.SCORE_SOFTMAX, O.ACT_SWIGLU, False, False, False),
    (O.SCORE_SIGMOID, O.ACT_SWIGLU, False, True, True),
])
def test_masked_dense_equals_permuted(score, act, bias, shared, renorm):
    rng = np.random.default_rng(11)
    T, h, E, K, F = 37, 16, 5, 2, 24
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = (rng.normal(size=(E, h)) / 4).astype(np.float32)
    w1, w2, b1, b2 = _weights(rng, E, h, F, act, bias)
    sh = _weights(rng, 1, h, F, act)[:2] if shared else (None, None)
    kw = dict(b1=b1, b2=b2, renorm=renorm,
              w1_shared=None if sh[0] is None else sh[0][0], w2_shared=None if sh[1] is None else sh[1][0])
    if score == O.SCORE_SIGMOID:
        kw["sel_bias"] = (0.1 * rng.normal(size=E)).astype(np.float32)
    a = O.layer_fwd(x, w_r, w1, w2, K, score, act, **kw)["y"]
    b = O.layer_fwd_masked_dense(x, w_r, w1, w2, K, score, act, **kw)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_skill_page_moe_layer_semantics():
    """The skill page's MoELayer.forward (gate = nn.Linear with bias, softmax,
    topk, renormalise, masked loop) run with torch ops in float64 equals the
    oracle with the gate bias."""
    rng = np.random.default_rng(12)
    T, h, E, K, F = 40, 12, 6, 2, 20
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = (rng.normal(size=(E, h)) / 3).astype(np.float32)
    b_r = rng.normal(size=E).astype(np.float32)
    w1, w2, b1, b2 = _weights(rng, E, h, F, O.ACT_GELU, bias=True)
    xt = torch.from_numpy(x.astype(np.float64))
    logits = Fnn.linear(xt, torch.from_numpy(w_r.astype(np.float64)), torch.from_numpy(b_r.astype(np.float64)))
    logits = logits.float().double()  # the router's fp32 logits
    scores = torch.softmax(logits, dim=-1)
    ts, ti = torch.topk(scores, K, dim=-1)
    ts = ts / ts.sum(dim=-1, keepdim=True)
    out = torch.zeros(T, h, dtype=torch.float64)
    for i in range(K):
        for e in range(E):
            mask = ti[:, i] == e
            if mask.any():
                out[mask] += ts[mask, i:i + 1] * torch.from_numpy(
                    _torch_ffn(xt[mask].numpy(), w1[e], w2[e], O.ACT_GELU, b1[e], b2[e]))
    got = O.layer_fwd(x, w_r, w1, w2, K, O.SCORE_SOFTMAX, O.ACT_GELU, b1=b1, b2=b2, gate_bias=b_r)
    np.testing.assert_allclose(got["y"], out.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("score", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID])
def test_identical_experts_is_dense_ffn(score):
    rng = np.random.default_rng(13)
    T, h, E, K, F = 30, 16, 8, 3, 32
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = rng.normal(size=(E, h)).astype(np.float32)
    w1, w2, _, _ = _weights(rng, 1, h, F, O.ACT_SWIGLU)
    w1 = np.repeat(w1, E, 0)
    w2 = np.repeat(w2, E, 0)
    y = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU)["y"]
    np.testing.assert_allclose(y, _torch_ffn(x, w1[0], w2[0], O.ACT_SWIGLU), rtol=1e-12, atol=1e-12)


def test_one_expert_top1_is_dense_ffn():
    # "Keep the Dense reference baseline": one expert with top-1 routing is
    # the dense FFN it replaces.
    rng = np.random.default_rng(14)
    T, h, F = 21, 8, 16
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = rng.normal(size=(1, h)).astype(np.float32)
    w1, w2, b1, b2 = _weights(rng, 1, h, F, O.ACT_GELU, bias=True)
    y = O.layer_fwd(x, w_r, w1, w2, 1, O.SCORE_SOFTMAX, O.ACT_GELU, b1=b1, b2=b2)["y"]
    # p == 1 exactly; only BLAS summation order separates the two
    np.testing.assert_allclose(y, _torch_ffn(x, w1[0], w2[0], O.ACT_GELU, b1[0], b2[0]), rtol=1e-13, atol=1e-14)


def test_memory_efficient_order_matches_standard():
    # Megatron Core review §4.1.1: for bias-free experts, scaling by p before
    # the second linear layer gives the same output.
    rng = np.random.default_rng(15)
    T, h, E, K, F = 17, 8, 4, 2, 12
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = rng.normal(size=(E, h)).astype(np.float32)
    w1, w2, _, _ = _weights(rng, E, h, F, O.ACT_SWIGLU)
    r = O.layer_fwd(x, w_r, w1, w2, K, O.SCORE_SOFTMAX, O.ACT_SWIGLU)
    y2 = O.layer_fwd_prob_before_fc2(x, w1, w2, r["idx"], r["probs"], O.ACT_SWIGLU)
    np.testing.assert_allclose(r["y"], y2, rtol=1e-12, atol=1e-13)


def test_token_subset_matches_full():
    rng = np.random.default_rng(16)
    T, h, E, K, F = 40, 8, 5, 2, 12
    x = rng.normal(size=(T, h)).astype(np.float32)
    w_r = rng.normal(size=(E, h)).astype(np.float32)
    w1, w2, _, _ = _weights(rng, E, h, F, O.ACT_SWIGLU)
    full = O.layer_fwd(x, w_r, w1, w2, K, O.SCORE_SOFTMAX, O.ACT_SWIGLU)["y"]
    sub = O.layer_fwd(x, w_r, w1, w2, K, O.SCORE_SOFTMAX, O.ACT_SWIGLU, tokens=[3, 17, 39])["y"]
    np.testing.assert_allclose(sub, full[[3, 17, 39]], rtol=1e-13, atol=1e-14)


def test_parameter_count_closed_form():
    # "Calculation of activated parameters": eight bias-free SwiGLU experts of
    # width 1024 at hidden 2048 hold as many parameters as the dense layer of
    # width 8192 they replace: 8 * (3 * 2048 * 1024) = 3 * 2048 * 8192.
    assert 8 * O.expert_param_count(2048, 1024, O.ACT_SWIGLU) == 3 * 2048 * 8192 == 50331648
    assert O.routed_flops(4096, 8, 7168, 2048, O.ACT_SWIGLU) == 6 * 4096 * 8 * 7168 * 2048
