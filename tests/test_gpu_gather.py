"""GPU checks of the gather-fused FC1 (moe_expert_fc1_gather): it must give
bit for bit the output of moe_expert_fc1 on the permuted rows (the same MMAs
see the same operands), on CTA pairs and single CTAs, SwiGLU and GELU with
biases, skewed loads with empty experts, ragged hidden sizes and capacity
drops; and a forward pass built from it (maps-only dispatch, gathered FC1)
must equal the layer forward bit for bit and the oracle within the bf16
tolerance."""

import numpy as np
import pytest
import torch

from gpu_util import Layer, lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs
from mixture_experts_layer_softmax_gb300 import workloads as W
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]


@pytest.mark.parametrize("T,h,E,K,F,act,bias,tiling,skew,cap", [
    (2048, 512, 4, 2, 256, "swiglu", False, "2cta", False, 0),
    (1500, 136, 8, 2, 200, "swiglu", False, "2cta", True, 0),
    (1000, 256, 16, 4, 128, "swiglu", False, "1cta", True, 0),
    (777, 200, 8, 2, 96, "gelu", True, "1cta", False, 0),
    (1200, 128, 4, 2, 64, "gelu", True, "2cta", False, 0),
    (600, 256, 1, 1, 128, "swiglu", False, "1cta", False, 0),
    (900, 128, 8, 2, 128, "swiglu", False, "1cta", True, 150),
])
def test_gather_fc1_equals_fc1_on_permuted_rows(T, h, E, K, F, act, bias, tiling, skew, cap):
    M = lib()
    rng = np.random.default_rng(T + h + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    if skew:
        logits[:, 0] += 3.0
        logits[:, E - 1] -= 50.0  # expert E-1 gets nothing
    idx, prob = O.route(logits, K, O.SCORE_SOFTMAX)
    x = inputs.normal((T, h), 1.0, 40, 1, "bf16")
    R1 = 2 * F if act == "swiglu" else F
    w1 = inputs.normal((E, R1, h), h ** -0.5, 40, 2, "bf16")
    b1 = inputs.normal((E, F), 0.1, 40, 3, "bf16") if bias else None
    flags = M.MOE_FLAG_RENORM | {"1cta": M.MOE_FLAG_GEMM_1CTA, "2cta": M.MOE_FLAG_GEMM_2CTA}[tiling]
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16, M.MOE_SCORE_SOFTMAX,
                        M.MOE_ACT_SWIGLU if act == "swiglu" else M.MOE_ACT_GELU, int(bias), 0,
                        flags, capacity=cap)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    P = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    xd = to_dev(x, "bf16")
    x_perm = torch.zeros(P, h, dtype=torch.bfloat16, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device="cuda")
    M.moe_permute(cfg, xd, torch.from_numpy(idx).cuda(), to_dev(prob, "f32"), x_perm, counts, offsets,
                  dst_row, src_token, perm_prob, ws)
    w1d = to_dev(w1, "bf16")
    b1d = None if b1 is None else to_dev(b1, "bf16")
    n = int(to_np(offsets)[-1])
    outs = []
    for gather in (False, True):
        a = torch.full((P, F), float("nan"), dtype=torch.bfloat16, device="cuda")
        save = torch.full((P, R1), float("nan"), dtype=torch.bfloat16, device="cuda")
        if gather:
            M.moe_expert_fc1_gather(cfg, xd, src_token, offsets, perm_prob, w1d, b1d, save, a)
        else:
            M.moe_expert_fc1(cfg, x_perm, offsets, perm_prob, w1d, b1d, save, a)
        torch.cuda.synchronize()
        assert M.moe_get_error() == M.MOE_OK
        outs.append((a[:n].clone(), save[:n].clone()))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    if skew:
        assert int(to_np(counts)[E - 1]) == 0


def test_gather_rejects_fp32_configs():
    M = lib()
    cfg = M.make_config(64, 128, 8, 2, 128, M.MOE_F32)
    f = M.raw("moe_expert_fc1_gather")
    assert f(cfg, *([None] * 8), None) == M.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("w", [
    W.MIXTRAL.replace(name="mixtral_gather", T=1024, h=512, F=512),
    W.QWEN3.replace(name="qwen3_gather", T=600, h=256, E=32, K=4, F=128),
    W.DSV3.replace(name="dsv3_gather_fwd", T=300, h=256, F=128, backward=False),
], ids=lambda w: w.name)
def test_forward_with_gathered_fc1_equals_layer_forward(w):
    M = lib()
    L = Layer(w)
    y_layer, idx_l, prob_l, _ = L.run_fwd(M)
    cfg = M.config_for(w)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    g = L.get
    T, h, E, K, F = w.T, w.h, w.E, w.K, w.F
    P = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    idx, prob = torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device="cuda")
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device="cuda")
    a, y_perm, y = torch.empty(P, F, **bf), torch.empty(P, h, **bf), torch.empty(T, h, **bf)
    M.moe_router_topk(cfg, g("x"), g("w_r"), g("gate_bias"), g("sel_bias"), None, idx, prob, None, ws)
    M.moe_permute(cfg, None, idx, prob, None, counts, offsets, dst_row, src_token, perm_prob, ws)
    M.moe_expert_fc1_gather(cfg, g("x"), src_token, offsets, perm_prob, g("w1"), None, None, a)
    M.moe_expert_fc2(cfg, a, offsets, perm_prob, g("w2"), None, y_perm)
    shared = None
    if w.n_shared:
        cs = M.make_config(T, h, 1, 1, F, cfg.dtype, cfg.score, cfg.act, 0, 0, cfg.flags)
        soff = torch.tensor([0, T], **i32)
        a_s, shared = torch.empty(T, F, **bf), torch.empty(T, h, **bf)
        M.moe_expert_fc1(cs, g("x"), soff, None, g("w1_shared"), None, None, a_s)
        M.moe_expert_fc2(cs, a_s, soff, None, g("w2_shared"), None, shared)
    M.moe_unpermute_combine(cfg, y_perm, dst_row, None, shared, y)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    assert torch.equal(idx, idx_l)
    assert torch.equal(y, y_layer)
    ref = L.oracle_fwd()
    ok_tok = L.margins(ref["logits"]) >= 1e-5
    ok, err, bound = tol_ok(to_np(y)[ok_tok], ref["y"][ok_tok], "bf16")
    assert ok, (err, bound)
