"""Parity at the full workload sizes, in the launch configuration the
benchmark times (moe_layer_fwd / moe_layer_bwd over device-resident seeded
inputs).  The oracle cannot run the whole layer at these sizes, so it checks:
  * the routing of every token (bit-exact except tokens whose top-K margin is
    below 1e-5) and the dispatch maps of the full batch (bit-exact, from the
    oracle's own routing fed to moe_permute);
  * the output rows of a sample of tokens whose experts lie in a small set, so
    the oracle needs only those experts' weights (regenerated on the host from
    the same seeded streams);
  * rows of every expert class through the staged expert GEMMs
    (moe_permute -> moe_expert_fc1 -> moe_expert_fc2 on the oracle's routing,
    with the same tilings the benchmark's workloads select): rows in the first,
    a middle and the last tile of every Mixtral expert and of the heaviest,
    median and lightest expert elsewhere, so the multi-tile CTA-pair schedules
    that only full sizes reach are compared with the oracle, one expert's
    weights at a time;
  * for the training configuration: dx of 16 tokens, dW1/dW2 of the lightest,
    median and heaviest expert (all of their rows), dprob of sampled slots, and
    the whole dW_r against dl^T x computed in float64 from the GPU's dprob
    (dl needs every expert's output for every token, which the host cannot
    regenerate; dprob itself is pinned on the sampled slots);
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

    def expert_classes(self, counts, every=False):
        """Experts to compare row by row: all of them (`every`), else the
        lightest non-empty, the median and the heaviest."""
        nz = np.nonzero(counts > 0)[0]
        if every:
            return [int(e) for e in nz]
        order = nz[np.argsort(counts[nz], kind="stable")]
        return sorted({int(order[0]), int(order[order.size // 2]), int(order[-1])})

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


def _tile_rows(n):
    """Rows of an expert segment of n rows at tile edges: the first rows, both
    sides of the 128-row boundary (the two CTAs of a pair tile), a middle
    pair, and the last rows (the ragged tail)."""
    cand = [0, 1, 127, 128, 255, 256, n // 2, n // 2 + 1, n - 2, n - 1]
    return sorted({r for r in cand if 0 <= r < n})


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_expert_rows(w):
    M = lib()
    F = Full(M, w)
    g = F.d.get
    cfg = M.config_for(w)
    T, h, E, K, Fd = w.T, w.h, w.E, w.K, w.F
    P = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.from_numpy(F.idx.astype(np.int32)).cuda()
    prob = torch.from_numpy(F.probs.astype(np.float32)).cuda()
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device="cuda")
    x_perm, a, y_perm = torch.empty(P, h, **bf), torch.empty(P, Fd, **bf), torch.empty(P, h, **bf)
    M.moe_permute(cfg, g("x"), idx, prob, x_perm, counts, offsets, dst_row, src_token, perm_prob, ws)
    M.moe_expert_fc1(cfg, x_perm, offsets, perm_prob, g("w1"), None, None, a)
    M.moe_expert_fc2(cfg, a, offsets, perm_prob, g("w2"), None, y_perm)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    o_counts, o_off, _, o_src, o_slot = O.dispatch_maps(F.idx, E)
    np.testing.assert_array_equal(to_np(offsets), o_off)
    experts = F.expert_classes(o_counts, every=(E <= 8))
    for e in experts:
        n = int(o_counts[e])
        rows = np.array(_tile_rows(n)) + int(o_off[e])
        t_r, k_r = o_src[rows], o_slot[rows]
        w1, w2 = F.expert_weights([e])
        p = F.probs[t_r, k_r][:, None]
        _, z = O.expert_hidden(F.x[t_r], w1[e], None, w.act)
        a_ref = p * z
        y_ref = p * O.expert_ffn(F.x[t_r], w1[e], w2[e], w.act)
        r_d = torch.from_numpy(rows).cuda()
        for name, got, ref in (("a", a[r_d], a_ref), ("y_perm", y_perm[r_d], y_ref)):
            good, err, bound = tol_ok(got.float().cpu().numpy(), ref, "bf16")
            assert good, (name, e, n, rows.tolist(), err, bound)


def _greedy_cover(idx, margin_ok, want):
    """`want` tokens chosen one by one, each time the one that adds the fewest
    experts not yet chosen (ties to the lower token), so the oracle needs few
    experts' weights."""
    chosen, toks = set(), []
    sel = [set(r.tolist()) for r in idx]
    free = np.nonzero(margin_ok)[0].tolist()
    while len(toks) < want and free:
        best = min(free, key=lambda t: (len(sel[t] - chosen), t))
        toks.append(best)
        chosen |= sel[best]
        free.remove(best)
    return np.array(sorted(toks)), sorted(chosen)


def test_full_size_training_backward_wide():
    """The DS-V3 training step at full size, wider than one expert: dx of 16
    tokens, the weight gradients of the lightest, median and heaviest expert,
    dprob of sampled slots, and all of dW_r."""
    M = lib()
    w = W.DSV3
    F = Full(M, w)
    cfg = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD)
    y, idx_g, ws = _fwd(M, F, M.MOE_FLAG_SAVE_FOR_BWD)
    idx_np = to_np(idx_g)
    np.testing.assert_array_equal(np.sort(idx_np, 1), np.sort(F.idx, 1))
    g = F.d.get
    T, h, E, K, Fd = w.T, w.h, w.E, w.K, w.F
    P = T * K
    bf = dict(dtype=torch.bfloat16, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    dx = torch.empty(T, h, **bf)
    dw_r = torch.empty(E, h, device="cuda")
    dw1, dw2 = torch.empty_like(g("w1")), torch.empty_like(g("w2"))
    dw1s, dw2s = torch.empty_like(g("w1_shared")), torch.empty_like(g("w2_shared"))
    M.moe_layer_bwd(cfg, g("x"), g("w_r"), g("w1"), g("w2"), g("w1_shared"), g("w2_shared"),
                    g("dy"), dx, dw_r, None, dw1, dw2, dw1s, dw2s, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    dy = w.host("dy")
    w1s, w2s = F.shared()
    counts = np.bincount(F.idx.ravel(), minlength=E)

    # dW1, dW2 of three expert classes over all of their rows
    for e in F.expert_classes(counts):
        t_e, k_e = np.nonzero(F.idx == e)
        w1e, w2e = F.expert_weights([e])
        gr = O.grouped_mlp_bwd(F.x[t_e], np.array([0, t_e.size]), F.probs[t_e, k_e], [w1e[e]],
                               [w2e[e]], dy[t_e])
        for name, t in (("dw1", dw1), ("dw2", dw2)):
            good, err, bound = tol_ok(t[e].float().cpu().numpy(), gr[name][0], "bf16")
            assert good, (name, e, int(counts[e]), err, bound)

    # dx of 16 tokens: per expert (one expert's weights at a time) the routed
    # rows' dx and dprob, then the shared expert and the router's part
    toks, experts = _greedy_cover(F.idx, F.margin >= 1e-5, 16)
    n = toks.size
    dx_ref = np.zeros((n, h))
    dprob_ref = np.zeros((n, K))
    for e in experts:
        tt, kk = np.nonzero(F.idx[toks] == e)
        w1e, w2e = F.expert_weights([e])
        gr = O.grouped_mlp_bwd(F.x[toks[tt]], np.array([0, tt.size]), F.probs[toks[tt], kk],
                               [w1e[e]], [w2e[e]], dy[toks[tt]])
        np.add.at(dx_ref, tt, gr["dx_perm"])
        dprob_ref[tt, kk] = gr["dprob_perm"]
    sh = O.grouped_mlp_bwd(F.x[toks], np.array([0, n]), np.ones(n), [w1s], [w2s], dy[toks])
    dx_ref += sh["dx_perm"]
    dl = O.router_grad_logits(F.logits[toks], F.idx[toks], F.probs[toks], dprob_ref, w.score,
                              w.renorm)
    dx_ref += dl @ F.w_r.astype(np.float64)
    good, err, bound = tol_ok(dx[torch.from_numpy(toks).cuda()].float().cpu().numpy(), dx_ref,
                              "bf16")
    assert good, ("dx", toks.tolist(), err, bound)

    # dprob of every slot from the staged backward (the same kernels), pinned
    # against the oracle on the 16 tokens' slots; then the whole dW_r of the
    # layer backward against dl^T x in float64 from that dprob
    cfg_s = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD)
    ws_s = torch.empty(M.moe_workspace_size(cfg_s), dtype=torch.uint8, device="cuda")
    prob_g = torch.from_numpy(O.topk_probs(F.logits, idx_np, w.score, w.renorm).astype(np.float32)).cuda()
    counts_g, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device="cuda")
    x_perm, dy_perm = torch.empty(P, h, **bf), torch.empty(P, h, **bf)
    H, a = torch.empty(P, 2 * Fd, **bf), torch.empty(P, Fd, **bf)
    M.moe_permute(cfg_s, g("x"), idx_g, prob_g, x_perm, counts_g, offsets, dst_row, src_token,
                  perm_prob, ws_s)
    M.moe_expert_fc1(cfg_s, x_perm, offsets, perm_prob, g("w1"), None, H, a)
    M.moe_permute(cfg_s, g("dy"), idx_g, prob_g, dy_perm, counts_g, offsets, dst_row, src_token,
                  perm_prob, ws_s)
    dprob_perm = torch.empty(P, dtype=torch.float32, device="cuda")
    dx_perm = torch.empty(P, h, **bf)
    # (dW1, dW2 of the layer backward were checked above; their buffers are reused)
    M.moe_grouped_mlp_bwd(cfg_s, dy_perm, x_perm, H, a, offsets, perm_prob, g("w1"), g("w2"),
                          dx_perm, dw1, dw2, dprob_perm, ws_s)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    dprob_g = to_np(dprob_perm)[to_np(dst_row)]               # [T, K] in the GPU's slot order
    for i, t in enumerate(toks):
        order = [int(np.nonzero(F.idx[t] == e)[0][0]) for e in idx_np[t]]
        got, ref = dprob_g[t], dprob_ref[i, order]
        assert np.abs(got - ref).max() <= 2e-2 * np.abs(ref).max() + 1e-3, ("dprob", int(t))
    dl_all = O.router_grad_logits(F.logits, idx_np, O.topk_probs(F.logits, idx_np, w.score,
                                                                  w.renorm),
                                  dprob_g.astype(np.float64), w.score, w.renorm)
    dw_r_ref = dl_all.T @ F.x.astype(np.float64)
    good, err, bound = tol_ok(to_np(dw_r), dw_r_ref, "f32")
    assert good, ("dw_r", err, bound)
