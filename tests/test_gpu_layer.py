"""GPU parity of the expert GEMMs and of the whole forward layer against the
oracle, at sizes the oracle finishes in seconds that still span several
tiles and ragged tails, plus determinism."""

import numpy as np
import pytest
import torch

from gpu_util import Layer, check_routing, lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs, workloads as W
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]


def _grouped_case(P_tokens, h, E, K, F, act, bias, dtype, skew=False, seed=0):
    rng = np.random.default_rng(seed)
    logits = rng.normal(size=(P_tokens, E)).astype(np.float32)
    if skew:
        logits[:, 0] += 3.0
        logits[:, E - 1] -= 100.0  # the last expert gets nothing
    idx, _ = O.route(logits, K, O.SCORE_SOFTMAX)
    counts, offsets, _, src_token, _ = O.dispatch_maps(idx, E)
    P = P_tokens * K
    R1 = 2 * F if act == O.ACT_SWIGLU else F
    x_perm = inputs.normal((P, h), 1.0, seed, 1, dtype)
    w1 = inputs.normal((E, R1, h), h ** -0.5, seed, 2, dtype)
    w2 = inputs.normal((E, h, F), F ** -0.5, seed, 3, dtype)
    b1 = inputs.normal((E, F), h ** -0.5, seed, 4, dtype) if bias else None
    b2 = inputs.normal((E, h), F ** -0.5, seed, 5, dtype) if bias else None
    prob = rng.uniform(0.05, 1.0, size=P).astype(np.float32)
    return dict(x_perm=x_perm, w1=w1, w2=w2, b1=b1, b2=b2, prob=prob, offsets=offsets,
                counts=counts, P=P, R1=R1)


GROUPED = [
    # tokens, h, E, K, F, act, bias, dtype, skew, path
    (600, 512, 8, 2, 768, O.ACT_SWIGLU, False, "bf16", False, "1cta"),
    (600, 512, 8, 2, 768, O.ACT_SWIGLU, False, "bf16", False, "2cta"),
    (300, 200, 5, 2, 136, O.ACT_SWIGLU, False, "bf16", True, "1cta"),
    (300, 200, 5, 2, 136, O.ACT_SWIGLU, False, "bf16", True, "2cta"),
    (700, 256, 1, 1, 384, O.ACT_SWIGLU, False, "bf16", False, "2cta"),
    (2100, 256, 4, 2, 384, O.ACT_SWIGLU, False, "bf16", False, "default"),
    (150, 128, 16, 4, 264, O.ACT_GELU, False, "bf16", True, "1cta"),
    (150, 128, 16, 4, 264, O.ACT_GELU, True, "bf16", False, "1cta"),
    (150, 128, 16, 4, 264, O.ACT_GELU, True, "bf16", False, "2cta"),
    (600, 512, 8, 2, 768, O.ACT_SWIGLU, False, "bf16", False, "simt"),
    (256, 128, 8, 2, 512, O.ACT_GELU, True, "f32", False, "default"),
    (100, 96, 3, 2, 52, O.ACT_SWIGLU, False, "f32", True, "default"),
]


@pytest.mark.parametrize("T,h,E,K,F,act,bias,dtype,skew,path", GROUPED)
def test_grouped_mlp_matches_oracle(T, h, E, K, F, act, bias, dtype, skew, path):
    M = lib()
    c = _grouped_case(T, h, E, K, F, act, bias, dtype, skew, seed=T + F)
    flags = M.MOE_FLAG_RENORM | {"simt": M.MOE_FLAG_GEMM_SIMT, "1cta": M.MOE_FLAG_GEMM_1CTA,
                                 "2cta": M.MOE_FLAG_GEMM_2CTA, "default": 0}[path]
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16 if dtype == "bf16" else M.MOE_F32,
                        M.MOE_SCORE_SOFTMAX, act, int(bias), 0, flags)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    P = c["P"]
    y_perm = torch.full((P, h), float("nan"), dtype=tdt, device="cuda")
    act_save = torch.full((P, c["R1"]), float("nan"), dtype=tdt, device="cuda")
    dv = lambda a: None if a is None else to_dev(a, dtype)
    M.moe_grouped_mlp_fwd(cfg, dv(c["x_perm"]), torch.from_numpy(c["offsets"].astype(np.int32)).cuda(),
                          to_dev(c["prob"], "f32"), dv(c["w1"]), dv(c["b1"]), dv(c["w2"]), dv(c["b2"]),
                          act_save, y_perm, ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    ref = np.zeros((P, h))
    ref_h = np.zeros((P, c["R1"]))
    off = c["offsets"]
    for e in range(E):
        r = slice(off[e], off[e + 1])
        if off[e + 1] == off[e]:
            continue
        b1e = None if c["b1"] is None else c["b1"][e]
        b2e = None if c["b2"] is None else c["b2"][e]
        ref[r] = c["prob"][r, None] * O.expert_ffn(c["x_perm"][r], c["w1"][e], c["w2"][e], act, b1e, b2e)
        ref_h[r] = O.expert_hidden(c["x_perm"][r], c["w1"][e], b1e, act)[0]
    ok, err, bound = tol_ok(to_np(y_perm), ref, dtype)
    assert ok, (err, bound)
    ok, err, bound = tol_ok(to_np(act_save), ref_h, dtype)
    assert ok, ("act_save", err, bound)



# Per-expert row counts around the pair kernel's 256-row tiles and its
# 128-row tail tiles: tails of 1, 64, 65, 127, 128 rows (half tiles), of 129,
# 255 rows (full tiles), whole blocks, an empty expert and a 5-block expert.
PAIR_TAIL_COUNTS = [1, 64, 65, 127, 128, 129, 192, 255, 256, 257, 300, 384, 385, 0, 640]


@pytest.mark.parametrize("act,bias,F", [(O.ACT_SWIGLU, False, 384), (O.ACT_SWIGLU, False, 200),
                                        (O.ACT_GELU, True, 264)])
def test_pair_tiles_with_tail_tiles_match_oracle(act, bias, F):
    """Every tail kind of the CTA-pair GEMMs (half and full tail tiles, ragged
    hidden sizes) within the bf16 tolerance of the oracle; the gathering FC1
    equals FC1 on the permuted rows bit for bit."""
    M = lib()
    counts = np.array(PAIR_TAIL_COUNTS, dtype=np.int64)
    E, h, seed = len(counts), 256, 71 + F
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    P = int(offsets[-1])
    R1 = 2 * F if act == O.ACT_SWIGLU else F
    T = 4000  # token rows the permuted rows are gathered from (T >= P)
    rng = np.random.default_rng(seed)
    src_token = rng.integers(0, T, size=P).astype(np.int32)
    x = inputs.normal((T, h), 1.0, seed, 1, "bf16")
    x_perm = x[src_token]
    w1 = inputs.normal((E, R1, h), h ** -0.5, seed, 2, "bf16")
    w2 = inputs.normal((E, h, F), F ** -0.5, seed, 3, "bf16")
    b1 = inputs.normal((E, F), h ** -0.5, seed, 4, "bf16") if bias else None
    b2 = inputs.normal((E, h), F ** -0.5, seed, 5, "bf16") if bias else None
    prob = rng.uniform(0.05, 1.0, size=P).astype(np.float32)
    # K = 1 and T = P: the permuted-row entry points see exactly P rows (the
    # routing is not used; the offsets are given)
    cfg = M.make_config(P, h, E, 1, F, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, act, int(bias), 0,
                        M.MOE_FLAG_RENORM | M.MOE_FLAG_GEMM_2CTA)
    dv = lambda a: None if a is None else to_dev(a, "bf16")
    offs = torch.from_numpy(offsets).cuda()
    probd = to_dev(prob, "f32")
    a = torch.full((P, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    save = torch.full((P, R1), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_perm = torch.full((P, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.moe_expert_fc1(cfg, dv(x_perm), offs, probd, dv(w1), dv(b1), save, a)
    M.moe_expert_fc2(cfg, a, offs, probd, dv(w2), dv(b2), y_perm)
    a_g = torch.full((P, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    save_g = torch.full((P, R1), float("nan"), dtype=torch.bfloat16, device="cuda")
    cfg_g = M.make_config(T, h, E, 1, F, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, act, int(bias), 0,
                          M.MOE_FLAG_RENORM | M.MOE_FLAG_GEMM_2CTA)
    assert P <= T
    M.moe_expert_fc1_gather(cfg_g, dv(x), torch.from_numpy(src_token).cuda(), offs, probd,
                            dv(w1), dv(b1), save_g, a_g)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    assert torch.equal(a, a_g) and torch.equal(save, save_g)
    ref = np.zeros((P, h))
    ref_h = np.zeros((P, R1))
    for e in range(E):
        r = slice(offsets[e], offsets[e + 1])
        if counts[e] == 0:
            continue
        b1e = None if b1 is None else b1[e]
        b2e = None if b2 is None else b2[e]
        ref[r] = prob[r, None] * O.expert_ffn(x_perm[r], w1[e], w2[e], act, b1e, b2e)
        ref_h[r] = O.expert_hidden(x_perm[r], w1[e], b1e, act)[0]
    ok, err, bound = tol_ok(to_np(y_perm), ref, "bf16")
    assert ok, (err, bound)
    ok, err, bound = tol_ok(to_np(save), ref_h, "bf16")
    assert ok, ("act_save", err, bound)


def small_workloads():
    return [
        W.TINY,
        W.MIXTRAL.replace(name="mixtral_small", T=600, h=512, F=768),
        W.QWEN3.replace(name="qwen3_small", T=1000, h=256, F=192),
        W.DSV3.replace(name="dsv3_small", T=300, h=256, F=128),
        W.Workload("sweep_small_random", T=512, h=256, E=64, K=8, F=128, seed=5),
        W.Workload("sweep_small_balanced", T=512, h=256, E=64, K=8, F=128, force_balance=True, seed=5),
        W.Workload("edge_one_token", T=1, h=64, E=4, K=2, F=64, seed=9),
        W.Workload("edge_three_tokens_K_eq_E", T=3, h=64, E=3, K=3, F=40, seed=9),
        W.Workload("edge_single_expert", T=130, h=128, E=1, K=1, F=136, seed=9),
        W.Workload("edge_gelu_bf16_bias", T=200, h=128, E=8, K=2, F=256, act=W.GELU, has_bias=True,
                   seed=9),
        # the one-launch router inside the layer: sigmoid keys with a selection
        # bias and a shared expert, and force-balanced routing
        W.DSV3.replace(name="dsv3_like_E8_small", T=400, h=256, E=8, K=2, F=128),
        W.Workload("mixtral_like_balanced_small", T=512, h=256, E=8, K=2, F=128,
                   force_balance=True, seed=9),
    ]


@pytest.mark.parametrize("w", small_workloads(), ids=lambda w: w.name)
def test_layer_forward_matches_oracle(w):
    M = lib()
    L = Layer(w)
    y, idx, prob, _ = L.run_fwd(M)
    ref = L.oracle_fwd()
    ok_tok = check_routing(to_np(idx), to_np(prob), ref["idx"], ref["probs"], ref["logits"], w.K,
                           w.score, L.h.get("sel_bias"), w.force_balance)
    good, err, bound = tol_ok(to_np(y)[ok_tok], ref["y"][ok_tok], w.dtype)
    assert good, (err, bound)


@pytest.mark.parametrize("w", small_workloads()[1:4], ids=lambda w: w.name)
def test_layer_forward_is_deterministic(w):
    M = lib()
    L = Layer(w)
    y1, i1, p1, ws = L.run_fwd(M)
    y2, i2, p2, _ = L.run_fwd(M, ws=ws)
    assert torch.equal(y1.view(torch.int16) if y1.dtype == torch.bfloat16 else y1,
                       y2.view(torch.int16) if y2.dtype == torch.bfloat16 else y2)
    assert torch.equal(i1, i2) and torch.equal(p1, p2)


@pytest.mark.parametrize("w", small_workloads()[1:6], ids=lambda w: w.name)
def test_layer_forward_on_cta_pairs_matches_oracle(w):
    M = lib()
    L = Layer(w)
    y, idx, prob, _ = L.run_fwd(M, flags_extra=M.MOE_FLAG_GEMM_2CTA)
    ref = L.oracle_fwd()
    ok_tok = check_routing(to_np(idx), to_np(prob), ref["idx"], ref["probs"], ref["logits"], w.K,
                           w.score, L.h.get("sel_bias"), w.force_balance)
    good, err, bound = tol_ok(to_np(y)[ok_tok], ref["y"][ok_tok], w.dtype)
    assert good, (err, bound)


def test_layer_simt_and_tensor_core_paths_agree():
    M = lib()
    w = W.MIXTRAL.replace(name="mixtral_small", T=300, h=256, F=384)
    L = Layer(w)
    y_tc, *_ = L.run_fwd(M)
    y_simt, *_ = L.run_fwd(M, flags_extra=M.MOE_FLAG_GEMM_SIMT)
    ok, err, bound = tol_ok(to_np(y_tc), to_np(y_simt), "bf16")
    assert ok, (err, bound)


def test_empty_batch_is_a_no_op():
    M = lib()
    cfg = M.make_config(0, 64, 4, 2, 64)
    ws = torch.empty(max(M.moe_workspace_size(cfg), 256), dtype=torch.uint8, device="cuda")
    e = torch.empty(0, device="cuda")
    z = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    M.moe_layer_fwd(cfg, z, torch.zeros(4, 64, device="cuda"), None, None, z, None, z, None, None,
                    None, z, None, None, ws)
    assert M.moe_get_error() == M.MOE_OK
