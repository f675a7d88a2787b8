"""Parity at the full workload sizes, in the launch configuration the
benchmark times (moe_layer_fwd / moe_layer_bwd over device-resident seeded
inputs).  The oracle cannot run the whole layer at these sizes, so it checks:
  * the routing of every token (bit-exact except tokens whose top-K margin is
    below 1e-5) and the dispatch maps of the full batch (bit-exact, from the
    oracle's own routing fed to moe_permute);
  * the output rows of a sample of tokens whose experts lie in a small set, so
    the oracle needs only those experts' weights (regenerated on the host from
    the same seeded streams);
  * for the training configuration, dx of sampled tokens and dW1/dW2 of one
    expert (all of its rows);
  * bitwise determinism of the full-size forward."""

import numpy as np
import pytest
import torch

from gpu_util import check_routing, lib, needs_gpu, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs, workloads as W
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]

FULL = [W.MIXTRAL, W.QWEN3, W.DSV3, W.ALL["sweep_T32768_h2048_E256_K8_F1024_random"],
        W.ALL["sweep_T8192_h2048_E64_K8_F1024_balanced"]]


class Full:
    """Device-generated full-size inputs plus the host pieces the oracle needs."""

    def __init__(self, M, w):
        self.M, self.w = M, w
        dev = torch.device("cuda")
        bf = torch.bfloat16
        self.d = {}
        for role in w.roles():
            if role in ("w_r", "sel_bias"):
                self.d[role] = torch.from_numpy(w.host(role)).to(dev)
            elif role == "gate_bias":
                self.d[role] = torch.from_numpy(w.gate_bias()).to(dev)
            else:
                t = torch.empty(w.shape(role), dtype=bf, device=dev)
                M.synth_normal(t, w.seed, inputs.TAG[role], w.std(role))
                self.d[role] = t
        self.x = w.host("x")
        self.w_r = w.host("w_r")
        self.sel_bias = w.host("sel_bias") if w.sel_bias_std > 0 else None
        self.gate_bias = w.gate_bias()
        self.logits = O.gating_logits(self.x, self.w_r, self.gate_bias)
        self.idx, self.probs = O.route(self.logits, w.K, w.score, w.renorm, self.sel_bias,
                                       w.force_balance)
        self.margin = (np.full(w.T, np.inf) if w.force_balance else
                       O.selection_margin(self.logits, w.K, w.score, self.sel_bias))

    def expert_weights(self, experts):
        w = self.w
        R1, h, F = w.w1_rows, w.h, w.F
        w1 = {e: inputs.normal((R1, h), w.std("w1"), w.seed, inputs.TAG["w1"], "bf16", start=e * R1 * h)
              for e in experts}
        w2 = {e: inputs.normal((h, F), w.std("w2"), w.seed, inputs.TAG["w2"], "bf16", start=e * h * F)
              for e in experts}
        return w1, w2

    def sample(self, want, budget=3.0e8):
        """Tokens whose experts all lie in a set grown (in token order) while
        the host weights stay under `budget` elements; margin-exempt tokens
        are skipped."""
        w = self.w
        per_expert = w.w1_rows * w.h + w.h * w.F
        budget = max(budget, 1.05 * w.K * per_expert)  # room for at least one token
        chosen = set()
        ok = self.margin >= 1e-5
        for t in range(w.T):
            if not ok[t]:
                continue
            new = set(self.idx[t].tolist()) - chosen
            if (len(chosen) + len(new)) * per_expert > budget:
                continue
            chosen |= new
            if (np.isin(self.idx, sorted(chosen)).all(1) & ok).sum() >= want:
                break
        toks = np.nonzero(np.isin(self.idx, sorted(chosen)).all(1) & ok)[0][:want]
        return toks, sorted(set(self.idx[toks].ravel().tolist()))

    def shared(self):
        w = self.w
        if not w.n_shared:
            return None, None
        return w.host("w1_shared"), w.host("w2_shared")


def _fwd(M, F, flags_extra=0, ws=None):
    w, g = F.w, F.d.get
    cfg = M.config_for(w, flags_extra)
    if ws is None:
        ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(w.T, w.h, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    M.moe_layer_fwd(cfg, g("x"), g("w_r"), g("gate_bias"), g("sel_bias"), g("w1"), None, g("w2"),
                    None, g("w1_shared"), g("w2_shared"), y, idx, None, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    return y, idx, ws


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_forward(w):
    M = lib()
    F = Full(M, w)
    y, idx, ws = _fwd(M, F)
    # routing of every token whose selection is unique
    check_routing(to_np(idx), None, F.idx, None, F.logits, w.K, w.score, F.sel_bias,
                  w.force_balance)
    # dispatch maps of the whole batch from the oracle's routing
    counts, offsets, dst_row, src_token, _ = O.dispatch_maps(F.idx, w.E)
    cfg = M.config_for(w)
    P = w.T * w.K
    i32 = dict(dtype=torch.int32, device="cuda")
    g_counts, g_off = torch.empty(w.E, **i32), torch.empty(w.E + 1, **i32)
    g_dst, g_src = torch.empty(w.T, w.K, **i32), torch.empty(P, **i32)
    M.moe_permute(cfg, None, torch.from_numpy(F.idx).cuda(), None, None, g_counts, g_off, g_dst,
                  g_src, None, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(g_counts), counts)
    np.testing.assert_array_equal(to_np(g_off), offsets)
    np.testing.assert_array_equal(to_np(g_dst), dst_row)
    np.testing.assert_array_equal(to_np(g_src), src_token)
    # sampled output rows
    toks, experts = F.sample(64)
    assert toks.size >= 1
    w1, w2 = F.expert_weights(experts)
    w1s, w2s = F.shared()
    ref = O.layer_fwd(F.x, F.w_r, w1, w2, w.K, w.score, w.act, w1_shared=w1s, w2_shared=w2s,
                      tokens=toks, routing=(F.logits, F.idx, F.probs))["y"]
    got = y[torch.from_numpy(toks).cuda()].float().cpu().numpy()
    good, err, bound = tol_ok(got, ref, "bf16")
    assert good, (toks.size, experts, err, bound)
    # bitwise determinism at full size
    y2, _, _ = _fwd(M, F, ws=ws)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_full_size_training_backward():
    M = lib()
    w = W.DSV3
    F = Full(M, w)
    ok = F.margin >= 1e-5
    cfg = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD)
    y, idx, ws = _fwd(M, F, M.MOE_FLAG_SAVE_FOR_BWD)
    # every token, near ties included, must select the oracle's experts, or the
    # oracle's gradients would not be those of the GPU's forward (the listing
    # order of the K experts does not enter any gradient)
    np.testing.assert_array_equal(np.sort(to_np(idx), 1), np.sort(F.idx, 1))
    g = F.d.get
    bf = dict(dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(w.T, w.h, **bf)
    dw_r = torch.empty(w.E, w.h, device="cuda")
    dw1, dw2 = torch.empty_like(g("w1")), torch.empty_like(g("w2"))
    dw1s, dw2s = torch.empty_like(g("w1_shared")), torch.empty_like(g("w2_shared"))
    M.moe_layer_bwd(cfg, g("x"), g("w_r"), g("w1"), g("w2"), g("w1_shared"), g("w2_shared"),
                    g("dy"), dx, dw_r, None, dw1, dw2, dw1s, dw2s, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    dy = w.host("dy")
    w1s, w2s = F.shared()
    # dx of sampled tokens (token-local: its experts, the shared expert, the router)
    toks, experts = F.sample(2)
    w1, w2 = F.expert_weights(experts)
    ref = O.layer_bwd(F.x[toks], F.w_r, w1, w2, dy[toks], w.K, w.score, w.act, w1_shared=w1s,
                      w2_shared=w2s, routing=(F.logits[toks], F.idx[toks], F.probs[toks]),
                      weight_grads=False)
    got = dx[torch.from_numpy(toks).cuda()].float().cpu().numpy()
    good, err, bound = tol_ok(got, ref["dx"], "bf16")
    assert good, ("dx", toks, err, bound)
    # dW1, dW2 of one expert over all of its rows
    counts = np.bincount(F.idx.ravel(), minlength=w.E)
    e = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    t_e, k_e = np.nonzero(F.idx == e)
    w1e, w2e = F.expert_weights([e])
    gr = O.grouped_mlp_bwd(F.x[t_e], np.array([0, t_e.size]), F.probs[t_e, k_e], [w1e[e]], [w2e[e]],
                           dy[t_e])
    for name, t in (("dw1", dw1), ("dw2", dw2)):
        good, err, bound = tol_ok(t[e].float().cpu().numpy(), gr[name][0], "bf16")
        assert good, (name, e, err, bound)
    # the shared expert's weight gradients see every token: check a slice of rows
    H, z = O.expert_hidden(F.x, w1s, None, w.act)
    dW2s_ref = dy.astype(np.float64)[:, :64].T @ z  # rows 0..63 of dW2_shared
    good, err, bound = tol_ok(dw2s[:64].float().cpu().numpy(), dW2s_ref, "bf16")
    assert good, ("dw2_shared", err, bound)
