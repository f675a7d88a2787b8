"""GPU parity of the backward (training configuration: bf16, SwiGLU, renormalised
router) against the oracle: the expert GEMMs' data and weight gradients with
ragged expert sizes and empty experts, the router backward, and the whole
layer backward including the shared expert; plus bitwise determinism."""

import numpy as np
import pytest
import torch

from gpu_util import Layer, lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs, workloads as W
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("T,h,E,K,F,skew", [
    (600, 512, 8, 2, 768, False),
    (300, 200, 5, 2, 136, True),     # M = 200 and 272: ragged weight-gradient tiles
    (400, 256, 64, 8, 128, False),
    (700, 128, 1, 1, 256, False),
    (2000, 128, 8, 1, 64, False),    # a single 64-wide FFN; experts of ~250 rows (two blocks)
    (300, 136, 96, 2, 136, "half"),  # every other expert without rows, over 3 chunks of 32 experts
])
def test_grouped_mlp_backward_matches_oracle(T, h, E, K, F, skew):
    M = lib()
    rng = np.random.default_rng(T + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    if skew == "half":
        logits[:, 1::2] -= 100.0  # the odd experts get no rows
    elif skew:
        logits[:, 0] += 3.0
        logits[:, E - 1] -= 100.0  # expert E-1 gets no rows: its gradients must be 0
    idx, _ = O.route(logits, K, O.SCORE_SOFTMAX)
    counts, offsets, _, _, _ = O.dispatch_maps(idx, E)
    P = T * K
    x_perm = inputs.normal((P, h), 1.0, 1, 1, "bf16")
    dy_perm = inputs.normal((P, h), 1.0, 1, 2, "bf16")
    w1 = inputs.normal((E, 2 * F, h), h ** -0.5, 1, 3, "bf16")
    w2 = inputs.normal((E, h, F), F ** -0.5, 1, 4, "bf16")
    prob = rng.uniform(0.05, 1.0, size=P).astype(np.float32)
    cfg = M.make_config(T, h, E, K, F)
    cfgb = M.make_config(T, h, E, K, F, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_SAVE_FOR_BWD)
    ws = torch.empty(M.moe_workspace_size(cfgb), dtype=torch.uint8, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    d_off = torch.from_numpy(offsets.astype(np.int32)).cuda()
    d_x, d_dy, d_w1, d_w2 = (to_dev(a, "bf16") for a in (x_perm, dy_perm, w1, w2))
    d_p = to_dev(prob, "f32")
    H = torch.empty(P, 2 * F, **bf)
    a = torch.empty(P, F, **bf)
    M.moe_expert_fc1(cfg, d_x, d_off, d_p, d_w1, None, H, a)
    dx = torch.full((P, h), float("nan"), **bf)
    dw1 = torch.full((E, 2 * F, h), float("nan"), **bf)
    dw2 = torch.full((E, h, F), float("nan"), **bf)
    dprob = torch.full((P,), float("nan"), device="cuda")
    M.moe_grouped_mlp_bwd(cfgb, d_dy, d_x, H, a, d_off, d_p, d_w1, d_w2, dx, dw1, dw2, dprob, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    ref = O.grouped_mlp_bwd(x_perm, offsets, prob, w1, w2, dy_perm)
    for name, g in (("dx_perm", dx), ("dw1", dw1), ("dw2", dw2), ("dprob_perm", dprob)):
        ok, err, bound = tol_ok(to_np(g), ref[name], "bf16")
        assert ok, (name, err, bound)
    empty = np.flatnonzero(counts == 0)
    if skew:
        assert len(empty) > 0 and (len(empty) >= E // 2 or skew is True)
    assert (to_np(dw1)[empty] == 0).all() and (to_np(dw2)[empty] == 0).all()


def _bwd_workloads():
    return [
        W.DSV3.replace(name="dsv3_small", T=300, h=256, F=128),
        W.MIXTRAL.replace(name="mixtral_small_bwd", T=400, h=256, F=384, backward=True),
        W.QWEN3.replace(name="qwen3_small_bwd", T=500, h=128, E=32, K=4, F=64, backward=True),
        W.Workload("one_expert_bwd", T=130, h=128, E=1, K=1, F=136, backward=True, seed=7),
    ]


def _run_layer_bwd(M, L, ca=0.0, cz=0.0):
    w = L.w
    cfg = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD, ca, cz)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y, idx, prob, _ = L.run_fwd(M, ws=ws, cfg=cfg)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    g = L.get
    out = dict(dx=torch.full((w.T, w.h), float("nan"), **bf),
               dw_r=torch.full((w.E, w.h), float("nan"), device="cuda"),
               db_r=torch.full((w.E,), float("nan"), device="cuda"),
               dw1=torch.full((w.E, 2 * w.F, w.h), float("nan"), **bf),
               dw2=torch.full((w.E, w.h, w.F), float("nan"), **bf))
    if w.n_shared:
        out["dw1_shared"] = torch.full((2 * w.F, w.h), float("nan"), **bf)
        out["dw2_shared"] = torch.full((w.h, w.F), float("nan"), **bf)
    M.moe_layer_bwd(cfg, g("x"), g("w_r"), g("w1"), g("w2"), g("w1_shared"), g("w2_shared"), g("dy"),
                    out["dx"], out["dw_r"], out["db_r"], out["dw1"], out["dw2"],
                    out.get("dw1_shared"), out.get("dw2_shared"), ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    if ca or cz:
        out["losses"] = torch.full((2,), float("nan"), device="cuda")
        M.moe_layer_losses(cfg, out["losses"], ws)
        torch.cuda.synchronize()
    return idx, out


@pytest.mark.parametrize("w", _bwd_workloads(), ids=lambda w: w.name)
def test_layer_backward_matches_oracle(w):
    M = lib()
    L = Layer(w)
    idx, out = _run_layer_bwd(M, L)
    h = L.h
    ref = O.layer_bwd(h["x"], h["w_r"], h["w1"], h["w2"], h["dy"], w.K, w.score, w.act,
                      sel_bias=h.get("sel_bias"), gate_bias=h.get("gate_bias"), renorm=w.renorm,
                      force_balance=w.force_balance, w1_shared=h.get("w1_shared"),
                      w2_shared=h.get("w2_shared"))
    # the selection must be the oracle's for every token (else pick another seed)
    np.testing.assert_array_equal(to_np(idx), ref["idx"])
    for name in ("dx", "dw_r", "db_r", "dw1", "dw2", "dw1_shared", "dw2_shared"):
        if name not in out:
            continue
        ok, err, bound = tol_ok(to_np(out[name]), ref[name], "bf16")
        assert ok, (name, err, bound)
    if w.E == 1:  # one expert: the router gets exactly no gradient
        assert (to_np(out["dw_r"]) == 0).all() and (to_np(out["db_r"]) == 0).all()


def test_layer_backward_is_deterministic():
    M = lib()
    L = Layer(_bwd_workloads()[0])
    _, a = _run_layer_bwd(M, L)
    _, b = _run_layer_bwd(M, L)
    for k in a:
        assert torch.equal(_bits(a[k]), _bits(b[k])), k


@pytest.mark.parametrize("score", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID])
def test_router_backward_matches_oracle(score):
    M = lib()
    T, h, E, K = 513, 256, 64, 6
    x = inputs.normal((T, h), 1.0, 5, 1, "bf16")
    w_r = inputs.normal((E, h), 0.05, 5, 2)
    logits = O.gating_logits(x, w_r)
    idx, probs = O.route(logits, K, score, True)
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(idx, E)
    dprob = inputs.normal((T, K), 1.0, 5, 3)
    dprob_perm = dprob[src_token, src_slot].astype(np.float32)
    cfg = M.make_config(T, h, E, K, 64, score=score,
                        flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_SAVE_FOR_BWD)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    dl = torch.empty(T, K, device="cuda")
    dw_r = torch.empty(E, h, device="cuda")
    db_r = torch.empty(E, device="cuda")
    dxr = torch.empty(T, h, device="cuda")
    M.moe_router_bwd(cfg, to_dev(x, "bf16"), to_dev(logits, "f32"), i32(idx),
                     to_dev(probs.astype(np.float32), "f32"), i32(offsets), i32(dst_row),
                     i32(src_token), to_dev(dprob_perm, "f32"), to_dev(w_r, "f32"), dl, dw_r, db_r,
                     dxr, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    dl_ref = O.router_grad_logits(logits, idx, probs, dprob, score, True)
    np.testing.assert_allclose(to_np(dl), np.take_along_axis(dl_ref, idx.astype(np.int64), 1),
                               rtol=1e-5, atol=1e-6)
    for got, want in ((dw_r, dl_ref.T @ x.astype(np.float64)), (db_r, dl_ref.sum(0)),
                      (dxr, dl_ref @ w_r.astype(np.float64))):
        ok, err, bound = tol_ok(to_np(got), want, "f32")
        assert ok, (err, bound)


@pytest.mark.parametrize("w", _bwd_workloads()[:3], ids=lambda w: w.name)
def test_layer_backward_with_load_balancing_losses(w):
    """With both loss weights set (scaled with T so their dense logit gradient
    is comparable to the routed one), dx, dW_r and db_r match the oracle's
    gradient of sum(dy * y) + a * aux + c * z, the losses match at 1e-4, and
    the change the weights make to dW_r and db_r matches the oracle's at fp32
    accuracy."""
    M = lib()
    L = Layer(w)
    ca, cz = 10.0 * w.T, 1.0 * w.T
    idx0, out0 = _run_layer_bwd(M, L)
    idx, out = _run_layer_bwd(M, L, ca, cz)
    h = L.h
    kw = dict(sel_bias=h.get("sel_bias"), gate_bias=h.get("gate_bias"), renorm=w.renorm,
              force_balance=w.force_balance, w1_shared=h.get("w1_shared"),
              w2_shared=h.get("w2_shared"))
    ref = O.layer_bwd(h["x"], h["w_r"], h["w1"], h["w2"], h["dy"], w.K, w.score, w.act,
                      aux_coeff=ca, z_coeff=cz, **kw)
    np.testing.assert_array_equal(to_np(idx), ref["idx"])
    for name in ("dx", "dw_r", "db_r"):
        ok, err, bound = tol_ok(to_np(out[name]), ref[name], "bf16")
        assert ok, (name, err, bound)
    losses = to_np(out["losses"])
    aux, z = O.aux_loss(ref["logits"], ref["idx"]), O.z_loss(ref["logits"])
    assert abs(losses[0] - aux) <= 1e-4 * aux and abs(losses[1] - z) <= 1e-4 * z, (losses, aux, z)
    dl = ca * O.aux_loss_grad(ref["logits"], ref["idx"]) + cz * O.z_loss_grad(ref["logits"])
    x64 = h["x"].astype(np.float64)
    for name, want in (("dw_r", dl.T @ x64), ("db_r", dl.sum(axis=0))):
        got = to_np(out[name]).astype(np.float64) - to_np(out0[name]).astype(np.float64)
        slack = 2.0 ** -23 * float(np.abs(to_np(out[name])).max())
        ok, err, bound = tol_ok(got, want, "f32")
        assert err <= bound + slack, (name, err, bound, slack)


def test_stage_events_time_the_layer_stages_without_changing_results():
    """moe_set_stage_events: the layer calls record the registered events at
    their stage boundaries, in order, and the results stay bit-identical to
    a run without them."""
    M = lib()
    L = Layer(_bwd_workloads()[0])
    _, plain = _run_layer_bwd(M, L)
    fwd = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    bwd = [torch.cuda.Event(enable_timing=True) for _ in range(9)]
    for ev in fwd + bwd:
        ev.record()
    torch.cuda.synchronize()
    M.moe_set_stage_events(M.MOE_PASS_FWD, fwd)
    M.moe_set_stage_events(M.MOE_PASS_BWD, bwd)
    try:
        _, timed = _run_layer_bwd(M, L)
    finally:
        M.moe_set_stage_events(M.MOE_PASS_FWD, [])
        M.moe_set_stage_events(M.MOE_PASS_BWD, [])
    for k in plain:
        assert torch.equal(_bits(plain[k]), _bits(timed[k])), k
    for evs in (fwd, bwd):
        gaps = [a.elapsed_time(b) for a, b in zip(evs[:-1], evs[1:])]
        assert all(g >= 0.0 for g in gaps), gaps        # recorded in boundary order
        total = evs[0].elapsed_time(evs[-1])
        assert abs(sum(gaps) - total) <= 1e-3 + 1e-3 * total
    assert bwd[4].elapsed_time(bwd[5]) > 0.0             # the dW1 GEMM ran between 4 and 5
