"""GPU parity of the expert capacity (token dropping) against the oracle:
dispatch maps and permuted rows bit-exact with dropped slots, the layer
forward and the training backward within the bf16 tolerance, the capacity
formula, and a capacity at least the largest load reproducing the dropless
run bit for bit."""

import numpy as np
import pytest
import torch

from gpu_util import Layer, lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs
from mixture_experts_layer_softmax_gb300 import workloads as W
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]


@pytest.mark.parametrize("T,E,K,C,skew", [
    (1000, 8, 2, 200, False), (1000, 128, 8, 50, True), (33, 4, 4, 1, False),
    (5000, 64, 8, 600, False), (4096, 256, 8, 160, False), (300, 16, 2, 10 ** 6, False),
])
def test_permute_with_capacity_bit_exact(T, E, K, C, skew):
    M = lib()
    h = 64
    rng = np.random.default_rng(T + E + C % 1000)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    if skew:
        logits[:, :3] += 3.0
    oi, op = O.route(logits, K, O.SCORE_SOFTMAX)
    keep = O.capacity_keep(oi, E, C)
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(oi, E, keep)
    n = int(offsets[-1])
    x = inputs.normal((T, h), 1.0, 5, 1, "bf16")
    cfg = M.make_config(T, h, E, K, 8, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM,
                        capacity=C)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    P = T * K
    d = dict(x_perm=torch.zeros(P, h, dtype=torch.bfloat16, device="cuda"),
             counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             dst_row=torch.empty(T, K, dtype=torch.int32, device="cuda"),
             src_token=torch.full((P,), -7, dtype=torch.int32, device="cuda"),
             perm_prob=torch.zeros(P, dtype=torch.float32, device="cuda"))
    M.moe_permute(cfg, to_dev(x, "bf16"), torch.from_numpy(oi).cuda(), to_dev(op, "f32"),
                  d["x_perm"], d["counts"], d["offsets"], d["dst_row"], d["src_token"],
                  d["perm_prob"], ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    np.testing.assert_array_equal(to_np(d["counts"]), counts)
    np.testing.assert_array_equal(to_np(d["offsets"]), offsets)
    np.testing.assert_array_equal(to_np(d["dst_row"]), dst_row)
    np.testing.assert_array_equal(to_np(d["src_token"])[:n], src_token[:n])
    np.testing.assert_array_equal(to_np(d["perm_prob"])[:n],
                                  op.astype(np.float32)[src_token[:n], src_slot[:n]])
    np.testing.assert_array_equal(to_np(d["x_perm"])[:n], O.permute_rows(x, src_token[:n]))
    if C >= np.bincount(oi.ravel(), minlength=E).max():
        assert keep.all()


def test_capacity_formula_matches_oracle():
    M = lib()
    for T, K, E, cf, mn in [(4096, 8, 256, 1.25, 0), (8192, 2, 8, 1.0, 0), (100, 1, 64, 0.1, 4),
                            (1000, 2, 3, 1.0, 0), (16384, 8, 128, 2.0, 4)]:
        assert M.moe_expert_capacity(T, K, E, cf, mn) == O.expert_capacity(T, K, E, cf, mn)
    assert M.moe_expert_capacity(10, 0, 4, 1.0, 0) == -1
    assert M.moe_expert_capacity(10, 2, 4, float("nan"), 0) == -1


def _workloads():
    return [
        W.MIXTRAL.replace(name="mixtral_small_cap", T=400, h=256, F=384, backward=True),
        W.DSV3.replace(name="dsv3_small_cap", T=300, h=256, F=128),
        W.QWEN3.replace(name="qwen3_small_cap", T=500, h=128, E=32, K=4, F=64, backward=True),
    ]


def _capacity(w, cf):
    return O.expert_capacity(w.T, w.K, w.E, cf)


@pytest.mark.parametrize("w", _workloads(), ids=lambda w: w.name)
def test_layer_forward_with_capacity_matches_oracle(w):
    M = lib()
    L = Layer(w)
    C = _capacity(w, 0.9)  # below the mean load: every workload drops slots
    cfg = M.config_for(w, 0, capacity=C)
    y, idx, prob, _ = L.run_fwd(M, cfg=cfg)
    h = L.h
    ref = O.layer_fwd(h["x"], h["w_r"], h["w1"], h["w2"], w.K, w.score, w.act,
                      sel_bias=h.get("sel_bias"), gate_bias=h.get("gate_bias"), renorm=w.renorm,
                      force_balance=w.force_balance, w1_shared=h.get("w1_shared"),
                      w2_shared=h.get("w2_shared"), capacity=C)
    np.testing.assert_array_equal(to_np(idx), ref["idx"])
    assert (~ref["keep"]).any()
    ok, err, bound = tol_ok(to_np(y), ref["y"], "bf16")
    assert ok, (err, bound)


@pytest.mark.parametrize("w", _workloads(), ids=lambda w: w.name)
def test_layer_backward_with_capacity_matches_oracle(w):
    M = lib()
    L = Layer(w)
    C = _capacity(w, 0.9)
    cfg = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD, capacity=C)
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
    h = L.h
    ref = O.layer_bwd(h["x"], h["w_r"], h["w1"], h["w2"], h["dy"], w.K, w.score, w.act,
                      sel_bias=h.get("sel_bias"), gate_bias=h.get("gate_bias"), renorm=w.renorm,
                      force_balance=w.force_balance, w1_shared=h.get("w1_shared"),
                      w2_shared=h.get("w2_shared"), capacity=C)
    np.testing.assert_array_equal(to_np(idx), ref["idx"])
    for name in ("dx", "dw_r", "db_r", "dw1", "dw2", "dw1_shared", "dw2_shared"):
        if name not in out:
            continue
        ok, err, bound = tol_ok(to_np(out[name]), ref[name], "bf16")
        assert ok, (name, err, bound)


def test_capacity_at_least_the_largest_load_is_the_dropless_layer():
    M = lib()
    w = _workloads()[0]
    L = Layer(w)
    y0, idx0, _, _ = L.run_fwd(M)
    y1, idx1, _, _ = L.run_fwd(M, cfg=M.config_for(w, 0, capacity=w.T * w.K))
    np.testing.assert_array_equal(to_np(idx0), to_np(idx1))
    assert torch.equal(y0, y1)


def test_router_bwd_entry_rejects_capacity():
    M = lib()
    cfg = M.make_config(64, 128, 8, 2, 128, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM, capacity=10)
    f = M.raw("moe_router_bwd")
    assert f(cfg, *([None] * 14), 0, None) == M.MOE_ERR_UNSUPPORTED
