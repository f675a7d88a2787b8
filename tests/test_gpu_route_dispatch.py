"""GPU parity of Route, Dispatch and Combine against the oracle: routing,
counts, offsets and the permutation are bit-exact given the same fp32 logits;
permuted rows are exact copies; the combine matches to fp32 rounding."""

import numpy as np
import pytest
import torch

from gpu_util import check_routing, lib, needs_gpu, to_dev, to_np, tol_ok
from mixture_experts_layer_softmax_gb300 import inputs
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]

ROUTER_CASES = [
    # T, E, K, score, renorm, bias, force
    (1, 1, 1, 0, True, False, False),
    (3, 2, 2, 0, True, False, False),
    (127, 8, 2, 0, True, False, False),
    (1000, 8, 2, 0, False, False, False),
    (513, 3, 3, 0, True, False, False),
    (700, 64, 8, 0, True, False, False),
    (700, 128, 8, 0, True, True, False),
    (300, 256, 8, 1, True, True, False),
    (300, 256, 8, 1, False, True, False),
    (256, 256, 16, 1, True, False, False),
    (512, 64, 8, 0, True, False, True),
    (96, 256, 8, 1, True, True, True),
    (200, 33, 5, 1, True, False, False),
]


@pytest.mark.parametrize("T,E,K,score,renorm,bias,force", ROUTER_CASES)
def test_router_from_logits_bit_exact(T, E, K, score, renorm, bias, force):
    M = lib()
    logits = inputs.normal((T, E), 1.0, 100 + E, 1)
    if E > 4:  # plant exact ties: the lower index must win
        logits[::7, 1] = logits[::7, 0]
        logits[::11, E - 1] = logits[::11, 2]
    b = inputs.normal((E,), 0.1, 101, 2) if bias else None
    flags = (M.MOE_FLAG_RENORM if renorm else 0) | (M.MOE_FLAG_FORCE_BALANCE if force else 0)
    cfg = M.make_config(T, 8, E, K, 8, M.MOE_F32, score, M.MOE_ACT_SWIGLU, 0, 0, flags)
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    prob = torch.empty(T, K, dtype=torch.float32, device="cuda")
    rmap = torch.empty(T, E, dtype=torch.uint8, device="cuda")
    M.moe_router_topk_from_logits(cfg, to_dev(logits, "f32"), None if b is None else to_dev(b, "f32"),
                                  idx, prob, rmap)
    torch.cuda.synchronize()
    oi, op = O.route(logits, K, score, renorm, b, force)
    np.testing.assert_array_equal(to_np(idx), oi)
    np.testing.assert_allclose(to_np(prob), op, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(to_np(rmap).astype(bool), O.routing_map(oi, E))


@pytest.mark.parametrize("bias", [False, True])
def test_router_sigmoid_near_ties_bit_exact(bias):
    """Sigmoid keys a few ulps apart (and exact ties): the fp32 first pass
    must hand such tokens to the double-precision ranking, so the selection
    and its order still equal the oracle's."""
    M = lib()
    T, E, K = 256, 64, 8
    rng = np.random.default_rng(7)
    base = rng.normal(size=(T, 1))
    steps = np.stack([rng.permutation(E) for _ in range(T)])
    logits = (base + steps * 1.5e-7).astype(np.float32)  # neighbours 1-2 ulps apart or equal
    b = (rng.integers(-3, 4, size=E) * 6e-8).astype(np.float32) if bias else None
    cfg = M.make_config(T, 8, E, K, 8, M.MOE_F32, M.MOE_SCORE_SIGMOID, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    prob = torch.empty(T, K, dtype=torch.float32, device="cuda")
    rmap = torch.empty(T, E, dtype=torch.uint8, device="cuda")
    M.moe_router_topk_from_logits(cfg, to_dev(logits, "f32"), None if b is None else to_dev(b, "f32"),
                                  idx, prob, rmap)
    torch.cuda.synchronize()
    oi, op = O.route(logits, K, M.MOE_SCORE_SIGMOID, True, b)
    np.testing.assert_array_equal(to_np(idx), oi)
    np.testing.assert_allclose(to_np(prob), op, rtol=2e-6, atol=1e-7)
    np.testing.assert_array_equal(to_np(rmap).astype(bool), O.routing_map(oi, E))


@pytest.mark.parametrize("T,h,E,K,score,dtype,gate_bias", [
    (300, 128, 8, 2, 0, "bf16", False), (257, 4096, 8, 2, 0, "bf16", False),
    (256, 128, 8, 2, 0, "f32", False), (100, 256, 16, 4, 0, "bf16", True),
    (100, 64, 32, 8, 1, "f32", False), (300, 512, 128, 8, 0, "bf16", True),
    (200, 7168, 256, 8, 1, "bf16", False), (64, 200, 5, 2, 0, "bf16", False),
    # 16, 20 and 32 experts (tensor cores, one tile of experts), a large batch of
    # the one-launch router (more clusters than fit at once), and a 32-expert
    # weight with a long h
    (130, 1024, 32, 4, 0, "bf16", True), (90, 512, 20, 3, 1, "bf16", False),
    (20000, 256, 8, 2, 0, "bf16", True), (77, 2048, 32, 8, 1, "bf16", False),
    # the one-launch router (bf16, E <= 8): a ragged last tile, a long h, and
    # h <= 64 (a single K block: three of the cluster's four CTAs have none)
    (8193, 4096, 8, 2, 1, "bf16", True), (300, 4608, 8, 2, 0, "bf16", False),
    (100, 64, 8, 2, 0, "bf16", True), (129, 8, 3, 1, 1, "bf16", False),
    (1, 512, 8, 2, 0, "bf16", True), (1, 512, 8, 8, 1, "bf16", False),
    # the tiled gating GEMM at larger sizes: 96 and 200 experts (ragged expert
    # tiles), more token tiles than SMs, and the full Qwen3 and DeepSeek-V3
    # shapes (one slice of h; h cut into slices)
    (10000, 4096, 96, 8, 0, "bf16", True), (10000, 2048, 200, 6, 1, "bf16", True),
    (33000, 512, 64, 8, 0, "bf16", False), (16384, 4096, 128, 8, 0, "bf16", True),
    (4096, 7168, 256, 8, 1, "bf16", False),
])
def test_router_gating_matches_oracle(T, h, E, K, score, dtype, gate_bias):
    M = lib()
    x = inputs.normal((T, h), 1.0, 7, 1, dtype)
    w_r = inputs.normal((E, h), 0.02 if h > 256 else 0.1, 7, 2)
    gb = inputs.normal((E,), 0.5, 7, 3) if gate_bias else None
    cfg = M.make_config(T, h, E, K, 16, M.MOE_BF16 if dtype == "bf16" else M.MOE_F32, score,
                        M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    prob = torch.empty(T, K, dtype=torch.float32, device="cuda")
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    M.moe_router_topk(cfg, to_dev(x, dtype), to_dev(w_r, "f32"), None if gb is None else to_dev(gb, "f32"),
                      None, logits, idx, prob, None, ws)
    torch.cuda.synchronize()
    ol = O.gating_logits(x, w_r, gb)
    gl = to_np(logits)
    scale = np.abs(x).astype(np.float64) @ np.abs(w_r).astype(np.float64).T
    assert np.all(np.abs(gl - ol) <= 1e-6 * scale + 1e-30)
    # selection: the set wherever the K-th / (K+1)-th gap is >= 1e-5, the
    # listing order wherever every gap in the top K + 1 is
    oi, _ = O.route(ol, K, score, True)
    check_routing(to_np(idx), None, oi, None, ol, K, score)


@pytest.mark.parametrize("E,K,score,renorm,bias,force", [
    (8, 2, 0, True, False, False), (8, 2, 0, False, False, False), (8, 8, 0, True, False, False),
    (8, 3, 1, True, True, False), (8, 4, 1, False, False, False), (5, 2, 1, True, True, False),
    (8, 2, 0, True, False, True), (6, 3, 1, True, False, True), (1, 1, 0, True, False, False),
])
def test_router_small_e_selection_matches_warp_selection(E, K, score, renorm, bias, force):
    """The one-launch router for E <= 8 selects with one thread per token; on
    the logits it wrote, the warp-per-token selection must give the same
    experts and bit-identical probabilities."""
    M = lib()
    T, h = 1000, 512
    x = inputs.normal((T, h), 1.0, 31, 1, "bf16")
    w_r = inputs.normal((E, h), 0.05, 31, 2)
    if score == M.MOE_SCORE_SIGMOID:  # many near ties among the sigmoid keys
        w_r[:, :] *= 0.02
    b = inputs.normal((E,), 0.01, 31, 3) if bias else None
    flags = (M.MOE_FLAG_RENORM if renorm else 0) | (M.MOE_FLAG_FORCE_BALANCE if force else 0)
    cfg = M.make_config(T, h, E, K, 16, M.MOE_BF16, score, M.MOE_ACT_SWIGLU, 0, 0, flags)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    prob = torch.empty(T, K, dtype=torch.float32, device="cuda")
    rmap = torch.empty(T, E, dtype=torch.uint8, device="cuda")
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    bd = None if b is None else to_dev(b, "f32")
    M.moe_router_topk(cfg, to_dev(x, "bf16"), to_dev(w_r, "f32"), None, bd, logits, idx, prob,
                      rmap, ws)
    idx2 = torch.empty_like(idx)
    prob2 = torch.empty_like(prob)
    rmap2 = torch.empty_like(rmap)
    M.moe_router_topk_from_logits(cfg, logits, bd, idx2, prob2, rmap2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(idx), to_np(idx2))
    np.testing.assert_array_equal(to_np(prob).view(np.uint32), to_np(prob2).view(np.uint32))
    np.testing.assert_array_equal(to_np(rmap), to_np(rmap2))


@pytest.mark.parametrize("T,E,K,skew", [
    (1, 1, 1, False), (3, 2, 2, False), (127, 8, 2, False), (1000, 8, 2, True),
    (1000, 128, 8, True), (2049, 256, 8, False), (4096, 64, 8, False), (33, 4, 4, False),
    # more tokens than the one-launch dispatch has warps (several tokens per
    # warp in the row scatter), and more chunks than warps
    (40000, 16, 4, True), (320000, 8, 2, False),
])
def test_permute_maps_bit_exact(T, E, K, skew):
    M = lib()
    h = 64
    rng = np.random.default_rng(T + E)
    logits = rng.normal(size=(T, E)).astype(np.float32)
    if skew:
        logits[:, 0] += 100.0  # everyone picks expert 0; several experts get nothing
    oi, op = O.route(logits, K, O.SCORE_SOFTMAX)
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(oi, E)
    x = inputs.normal((T, h), 1.0, 3, 1, "bf16")
    cfg = M.make_config(T, h, E, K, 8, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    P = T * K
    d = dict(x_perm=torch.empty(P, h, dtype=torch.bfloat16, device="cuda"),
             counts=torch.empty(E, dtype=torch.int32, device="cuda"),
             offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
             dst_row=torch.empty(T, K, dtype=torch.int32, device="cuda"),
             src_token=torch.empty(P, dtype=torch.int32, device="cuda"),
             perm_prob=torch.empty(P, dtype=torch.float32, device="cuda"))
    M.moe_permute(cfg, to_dev(x, "bf16"), torch.from_numpy(oi).cuda(), to_dev(op, "f32"),
                  d["x_perm"], d["counts"], d["offsets"], d["dst_row"], d["src_token"],
                  d["perm_prob"], ws)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    np.testing.assert_array_equal(to_np(d["counts"]), counts)
    np.testing.assert_array_equal(to_np(d["offsets"]), offsets)
    np.testing.assert_array_equal(to_np(d["dst_row"]), dst_row)
    np.testing.assert_array_equal(to_np(d["src_token"]), src_token)
    np.testing.assert_array_equal(to_np(d["perm_prob"]), op.astype(np.float32)[src_token, src_slot])
    np.testing.assert_array_equal(to_np(d["x_perm"]), O.permute_rows(x, src_token))


def test_permute_rejects_bad_expert_ids_without_faulting():
    M = lib()
    T, E, K, h = 64, 8, 2, 32
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[5, 1] = 99  # out of range: reported, row skipped
    cfg = M.make_config(T, h, E, K, 8, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    P = T * K
    x_perm = torch.zeros(P, h, dtype=torch.bfloat16, device="cuda")
    out = [torch.zeros(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, P, P)]
    M.moe_permute(cfg, torch.zeros(T, h, dtype=torch.bfloat16, device="cuda"),
                  torch.from_numpy(idx).cuda(), None, x_perm, out[0], out[1], out[2], out[3],
                  None, ws)
    assert M.moe_get_error() == M.MOE_ERR_DEVICE_BOUNDS
    assert M.moe_get_error() == M.MOE_OK  # cleared
    assert int(out[1][-1]) == P - 1


@pytest.mark.parametrize("T,E,K,h,dtype,weighted,shared", [
    (1, 1, 1, 8, "bf16", False, False), (300, 8, 2, 4096, "bf16", False, True),
    (257, 16, 4, 136, "bf16", True, False), (100, 8, 2, 128, "f32", True, True),
    (2000, 64, 8, 512, "bf16", False, False),
])
def test_combine_matches_oracle(T, E, K, h, dtype, weighted, shared):
    M = lib()
    rng = np.random.default_rng(T)
    oi, op = O.route(rng.normal(size=(T, E)).astype(np.float32), K, O.SCORE_SOFTMAX)
    _, _, dst_row, _, _ = O.dispatch_maps(oi, E)
    y_perm = inputs.normal((T * K, h), 1.0, 9, 1, dtype)
    sy = inputs.normal((T, h), 1.0, 9, 2, dtype) if shared else None
    cfg = M.make_config(T, h, E, K, 8, M.MOE_BF16 if dtype == "bf16" else M.MOE_F32, 0,
                        M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)
    y = torch.empty(T, h, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    M.moe_unpermute_combine(cfg, to_dev(y_perm, dtype), torch.from_numpy(dst_row.astype(np.int32)).cuda(),
                            to_dev(op, "f32") if weighted else None,
                            None if sy is None else to_dev(sy, dtype), y)
    torch.cuda.synchronize()
    ref = O.unpermute_combine(y_perm, dst_row, op.astype(np.float32) if weighted else None)
    if shared:
        ref = ref + sy
    g = to_np(y)
    if dtype == "bf16":  # one rounding of the fp32 sum
        assert np.all(np.abs(g - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6 * K)
    else:
        np.testing.assert_allclose(g, ref, rtol=1e-6, atol=1e-5)


def test_bounded_wait_times_out_and_context_survives():
    M = lib()
    M.moe_test_bounded_wait(2000)
    assert M.moe_get_error() == M.MOE_ERR_TIMEOUT
    assert M.moe_get_error() == M.MOE_OK
    t = torch.ones(8, device="cuda")
    assert float(t.sum()) == 8.0


@pytest.mark.parametrize("T,h,E,K,dtype", [
    (1000, 256, 8, 2, "bf16"),    # one-launch router: histograms from its epilogue
    (257, 128, 6, 3, "bf16"),     # ragged last chunk, E < 8
    (1, 64, 8, 1, "bf16"),
    (777, 128, 64, 8, "bf16"),    # tensor-core gating GEMM + selection, then the histogram step
    (10000, 256, 64, 8, "bf16"), (12000, 512, 256, 8, "bf16"),
    (300, 64, 16, 4, "f32"),
])
def test_router_histogram_hand_off_gives_the_same_dispatch(T, h, E, K, dtype):
    """MOE_FLAG_HIST_FROM_ROUTER: the router leaves the per-chunk histograms in
    the workspace and moe_permute starts from them; maps and rows are bit-for-
    bit those of moe_permute counting on its own."""
    M = lib()
    x = to_dev(inputs.normal((T, h), 1.0, T + E, 1, dtype), dtype)
    w_r = to_dev(inputs.normal((E, h), 0.05, T + E, 2), "f32")
    dt = M.MOE_BF16 if dtype == "bf16" else M.MOE_F32
    base = M.MOE_FLAG_RENORM
    cfg_h = M.make_config(T, h, E, K, 8, dt, 0, M.MOE_ACT_SWIGLU, 0, 0, base | M.MOE_FLAG_HIST_FROM_ROUTER)
    cfg = M.make_config(T, h, E, K, 8, dt, 0, M.MOE_ACT_SWIGLU, 0, 0, base)
    ws = torch.full((M.moe_workspace_size(cfg_h),), 0x7f, dtype=torch.uint8, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    P = T * K
    idx, prob = torch.empty(T, K, **i32), torch.empty(T, K, device="cuda")
    M.moe_router_topk(cfg_h, x, w_r, None, None, None, idx, prob, None, ws)

    def dispatch(c, w):
        out = dict(x_perm=torch.empty(P, h, dtype=x.dtype, device="cuda"),
                   counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
                   dst_row=torch.empty(T, K, **i32), src_token=torch.empty(P, **i32),
                   perm_prob=torch.empty(P, device="cuda"))
        M.moe_permute(c, x, idx, prob, out["x_perm"], out["counts"], out["offsets"],
                      out["dst_row"], out["src_token"], out["perm_prob"], w)
        return out

    got = dispatch(cfg_h, ws)
    ws_plain = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    want = dispatch(cfg, ws_plain)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    for k in want:
        a, b = want[k], got[k]
        if a.dtype in (torch.bfloat16, torch.float32) and k == "x_perm":
            a, b = a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32), \
                b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
        assert torch.equal(a, b), k
    assert int(got["offsets"][-1]) == P
    if dtype == "bf16" and h % 128 == 0:  # the MXFP8 dispatch takes the same hand-off
        sfb = M.moe_mxfp8_scale_bytes(P, h, E)
        res = []
        for c, w in ((cfg_h, ws), (cfg, ws_plain)):
            q = torch.zeros(P, h, dtype=torch.uint8, device="cuda")
            sf = torch.zeros(max(sfb, 16), dtype=torch.uint8, device="cuda")
            m = [torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T, K, **i32),
                 torch.empty(P, **i32), torch.empty(P, device="cuda")]
            M.moe_permute_mxfp8(c, x, idx, prob, q, sf, *m, w)
            res.append([q, sf] + m)
        torch.cuda.synchronize()
        assert M.moe_get_error() == M.MOE_OK
        for a, b in zip(*res):
            assert torch.equal(a, b)
