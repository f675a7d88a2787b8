"""GPU parity of the router's load-balancing losses (moe_router_aux_loss)
against the oracle: the auxiliary loss and the z-loss within the fp32
tolerance (1e-4 relative), the weighted logit gradients added in place within
1e-4 of their largest magnitude, bitwise-identical reruns, and out-of-range
expert ids reported without being counted."""

import numpy as np
import pytest
import torch

from gpu_util import lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]

CASES = [
    # T, E, K, logit scale, seed
    (1, 1, 1, 1.0, 1),
    (3, 2, 1, 1.0, 2),
    (300, 8, 2, 2.0, 3),
    (777, 20, 3, 1.0, 4),
    (1000, 33, 5, 3.0, 5),
    (4096, 256, 8, 1.0, 6),     # DeepSeek-V3-sized router
    (16384, 128, 8, 2.0, 7),    # Qwen3-sized router
    (33000, 64, 8, 0.5, 8),     # more tokens than the partial-sum blocks cover at 64 each
]


def _run(M, T, E, K, logits, idx, ca, cz, d0):
    cfg = M.make_config(T, 8, E, K, 8, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    losses = torch.full((2,), float("nan"), device="cuda")
    dl = None if d0 is None else to_dev(d0, "f32")
    M.moe_router_aux_loss(cfg, to_dev(logits, "f32"), torch.from_numpy(idx).cuda(), ca, cz, losses,
                          dl, ws)
    torch.cuda.synchronize()
    return to_np(losses), (None if dl is None else to_np(dl))


@pytest.mark.parametrize("T,E,K,scale,seed", CASES)
def test_losses_and_gradients_match_oracle(T, E, K, scale, seed):
    M = lib()
    logits = inputs.normal((T, E), scale, 200 + seed, 1)
    idx = O.select_topk(logits, K)
    ca, cz = 1e-2, 1e-3
    d0 = inputs.normal((T, E), 1e-4 / max(T, 1), 200 + seed, 2)
    losses, dl = _run(M, T, E, K, logits, idx, ca, cz, d0)
    assert M.moe_get_error() == M.MOE_OK
    aux, z = O.aux_loss(logits, idx), O.z_loss(logits)
    assert abs(losses[0] - aux) <= 1e-4 * abs(aux), (losses[0], aux)
    assert abs(losses[1] - z) <= 1e-4 * abs(z), (losses[1], z)
    inc = ca * O.aux_loss_grad(logits, idx) + cz * O.z_loss_grad(logits)
    ok, err, bound = tol_ok(dl - d0.astype(np.float64), inc, "f32")
    # fp32 rounding of the accumulation into d0 adds at most ulp(|d0| + |inc|)
    slack = 2.0 ** -23 * float(np.max(np.abs(d0) + np.abs(inc)))
    assert err <= bound + slack, (err, bound, slack)


def test_losses_without_gradient_and_zero_coefficients():
    M = lib()
    T, E, K = 500, 16, 4
    logits = inputs.normal((T, E), 1.0, 300, 1)
    idx = O.select_topk(logits, K)
    d0 = inputs.normal((T, E), 1.0, 300, 2)
    losses, dl = _run(M, T, E, K, logits, idx, 0.0, 0.0, d0)
    np.testing.assert_array_equal(dl, d0)  # zero coefficients: dlogits untouched
    losses2, _ = _run(M, T, E, K, logits, idx, 0.5, 0.5, None)  # no gradient buffer
    np.testing.assert_array_equal(losses, losses2)
    assert abs(losses[0] - O.aux_loss(logits, idx)) <= 1e-4 * O.aux_loss(logits, idx)


def test_single_expert_and_balanced_cases_are_one():
    M = lib()
    # the single-expert baseline: load-balance loss exactly 1
    T = 1000
    logits = inputs.normal((T, 1), 2.0, 301, 1)
    losses, _ = _run(M, T, 1, 1, logits, np.zeros((T, 1), np.int32), 1.0, 0.0, None)
    assert losses[0] == pytest.approx(1.0, rel=1e-6)
    # force-balanced routing, equal logits
    T, E, K = 1024, 64, 8
    losses, _ = _run(M, T, E, K, np.full((T, E), 0.25, np.float32), O.force_balanced_topk(T, K, E),
                     1.0, 1.0, None)
    assert losses[0] == pytest.approx(1.0, rel=1e-6)
    assert losses[1] == pytest.approx((0.25 + np.log(E)) ** 2, rel=1e-6)


def test_reruns_are_bitwise_identical():
    M = lib()
    T, E, K = 5000, 128, 8
    logits = inputs.normal((T, E), 1.5, 302, 1)
    idx = O.select_topk(logits, K)
    d0 = np.zeros((T, E), np.float32)
    a = _run(M, T, E, K, logits, idx, 1e-3, 1e-3, d0)
    b = _run(M, T, E, K, logits, idx, 1e-3, 1e-3, d0)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_bad_expert_ids_are_reported_and_not_counted():
    M = lib()
    T, E, K = 64, 8, 2
    logits = inputs.normal((T, E), 1.0, 303, 1)
    idx = O.select_topk(logits, K)
    bad = idx.copy()
    bad[5, 1] = 99
    losses, _ = _run(M, T, E, K, logits, bad, 1.0, 0.0, None)
    assert M.moe_get_error() == M.MOE_ERR_DEVICE_BOUNDS
    assert M.moe_get_error() == M.MOE_OK
    f = np.bincount(np.delete(bad.ravel(), 5 * K + 1), minlength=E) / (T * K)
    P = O.softmax_full(logits).mean(axis=0)
    assert losses[0] == pytest.approx(E * (f * P).sum(), rel=1e-4)
