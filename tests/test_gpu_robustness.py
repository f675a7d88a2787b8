"""Robustness of the C ABI on the GPU without faulting it:

* host-side failure injection (moe_test_inject_cuda_failure): the injected
  calls return MOE_ERR_CUDA before enqueuing anything (their outputs stay
  untouched), and the next calls work and match the uninjected results;
* canary guard words: every output buffer of every entry point, and the
  workspace, sit between guard regions filled with a byte pattern; after
  calls on ragged shapes (row, column and expert counts that leave partial
  tiles) the guards are unchanged, so no kernel writes outside its
  buffers."""

import numpy as np
import pytest
import torch

from gpu_util import lib, needs_gpu, to_dev
from mixture_experts_layer_softmax_gb300 import inputs
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]

GUARD = 8192  # bytes before and after each buffer
PATTERN = 0xA5


class Guarded:
    """Device buffers carved from larger byte buffers whose borders hold PATTERN."""

    def __init__(self):
        self.bufs = []

    def new(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        t = raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            t.copy_(fill if torch.is_tensor(fill) else torch.full(shape, fill, dtype=dtype))
        self.bufs.append((raw, n))
        return t

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.bufs):
            head = raw[:GUARD].cpu().numpy()
            tail = raw[GUARD + n:].cpu().numpy()
            assert (head == PATTERN).all() and (tail == PATTERN).all(), f"buffer {i}: guard overwritten"


def _layer_inputs(g, T, h, E, K, F, seed):
    x = g.new((T, h), torch.bfloat16, to_dev(inputs.normal((T, h), 1.0, seed, 1, "bf16"), "bf16"))
    w_r = g.new((E, h), torch.float32, to_dev(inputs.normal((E, h), 0.02, seed, 2), "f32"))
    w1 = g.new((E, 2 * F, h), torch.bfloat16,
               to_dev(inputs.normal((E, 2 * F, h), h ** -0.5, seed, 3, "bf16"), "bf16"))
    w2 = g.new((E, h, F), torch.bfloat16,
               to_dev(inputs.normal((E, h, F), F ** -0.5, seed, 4, "bf16"), "bf16"))
    return x, w_r, w1, w2


@pytest.mark.parametrize("T,h,E,K,F,flags_extra", [
    (333, 136, 13, 3, 200, 0),                # ragged rows, columns, experts
    (1030, 256, 8, 2, 384, "2cta"),           # CTA-pair tiles
    (77, 128, 64, 8, 64, 0),                  # many experts below one tile
])
def test_layer_forward_and_backward_write_only_their_buffers(T, h, E, K, F, flags_extra):
    M = lib()
    g = Guarded()
    x, w_r, w1, w2 = _layer_inputs(g, T, h, E, K, F, 7 + T)
    flags = M.MOE_FLAG_RENORM | M.MOE_FLAG_SAVE_FOR_BWD | (M.MOE_FLAG_GEMM_2CTA if flags_extra == "2cta" else 0)
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, M.MOE_ACT_SWIGLU, 0, 0, flags)
    ws = g.new((M.moe_workspace_size(cfg),), torch.uint8, 0)
    y = g.new((T, h), torch.bfloat16, float("nan"))
    idx = g.new((T, K), torch.int32, -5)
    prob = g.new((T, K), torch.float32, float("nan"))
    M.moe_layer_fwd(cfg, x, w_r, None, None, w1, None, w2, None, None, None, y, idx, prob, ws)
    dy = g.new((T, h), torch.bfloat16, to_dev(inputs.normal((T, h), 1.0, 9, 5, "bf16"), "bf16"))
    dx = g.new((T, h), torch.bfloat16, float("nan"))
    dw_r = g.new((E, h), torch.float32, float("nan"))
    db_r = g.new((E,), torch.float32, float("nan"))
    dw1 = g.new((E, 2 * F, h), torch.bfloat16, float("nan"))
    dw2 = g.new((E, h, F), torch.bfloat16, float("nan"))
    M.moe_layer_bwd(cfg, x, w_r, w1, w2, None, None, dy, dx, dw_r, db_r, dw1, dw2, None, None, ws)
    assert M.moe_get_error() == M.MOE_OK
    g.check()
    for t in (y, dx, dw_r, db_r, dw1, dw2):
        assert torch.isfinite(t.float()).all()


def test_step_entry_points_write_only_their_buffers():
    M = lib()
    g = Guarded()
    T, h, E, K, F = 501, 264, 7, 3, 136
    x, w_r, w1, w2 = _layer_inputs(g, T, h, E, K, F, 11)
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16, M.MOE_SCORE_SIGMOID, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    ws = g.new((M.moe_workspace_size(cfg),), torch.uint8, 0)
    P = T * K
    i32 = torch.int32
    logits = g.new((T, E), torch.float32, float("nan"))
    idx = g.new((T, K), i32, -1)
    prob = g.new((T, K), torch.float32, float("nan"))
    rmap = g.new((T, E), torch.uint8, 7)
    M.moe_router_topk(cfg, x, w_r, None, None, logits, idx, prob, rmap, ws)
    x_perm = g.new((P, h), torch.bfloat16, float("nan"))
    counts, offsets = g.new((E,), i32, -1), g.new((E + 1,), i32, -1)
    dst_row, src_token = g.new((T, K), i32, -1), g.new((P,), i32, -1)
    perm_prob = g.new((P,), torch.float32, float("nan"))
    M.moe_permute(cfg, x, idx, prob, x_perm, counts, offsets, dst_row, src_token, perm_prob, ws)
    # the allocation-free dispatch writes the same buffers (and only them)
    x_perm2 = g.new((P, h), torch.bfloat16, float("nan"))
    counts2, offsets2 = g.new((E,), i32, -1), g.new((E + 1,), i32, -1)
    dst_row2, src_token2 = g.new((T, K), i32, -1), g.new((P,), i32, -1)
    perm_prob2 = g.new((P,), torch.float32, float("nan"))
    M.moe_permute_noalloc(cfg, x, idx, prob, x_perm2, counts2, offsets2, dst_row2, src_token2,
                          perm_prob2)
    H = g.new((P, 2 * F), torch.bfloat16, float("nan"))
    a = g.new((P, F), torch.bfloat16, float("nan"))
    M.moe_expert_fc1(cfg, x_perm, offsets, perm_prob, w1, None, H, a)
    y_perm = g.new((P, h), torch.bfloat16, float("nan"))
    M.moe_expert_fc2(cfg, a, offsets, perm_prob, w2, None, y_perm)
    y = g.new((T, h), torch.bfloat16, float("nan"))
    M.moe_unpermute_combine(cfg, y_perm, dst_row, None, None, y)
    losses = g.new((2,), torch.float32, float("nan"))
    dlog = g.new((T, E), torch.float32, 0.0)
    M.moe_router_aux_loss(cfg, logits, idx, 1e-2, 1e-3, losses, dlog, ws)
    assert M.moe_get_error() == M.MOE_OK
    g.check()
    assert torch.isfinite(y.float()).all()
    for a_, b_ in ((counts, counts2), (offsets, offsets2), (dst_row, dst_row2),
                   (src_token, src_token2), (perm_prob, perm_prob2),
                   (x_perm.view(torch.int16), x_perm2.view(torch.int16))):
        assert torch.equal(a_, b_)


def test_mxfp8_entry_points_write_only_their_buffers():
    M = lib()
    g = Guarded()
    T, h, E, K, F = 300, 384, 6, 2, 256
    x, w_r, w1, w2 = _layer_inputs(g, T, h, E, K, F, 13)
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    ws = g.new((M.moe_workspace_size(cfg),), torch.uint8, 0)
    P = T * K
    i32 = torch.int32
    idx = g.new((T, K), i32, -1)
    prob = g.new((T, K), torch.float32, float("nan"))
    M.moe_router_topk(cfg, x, w_r, None, None, None, idx, prob, None, ws)
    u8 = torch.uint8
    xq = g.new((P, h), u8, 0)
    xsf = g.new((M.moe_mxfp8_scale_bytes(P, h, E),), u8, 0)
    counts, offsets = g.new((E,), i32, -1), g.new((E + 1,), i32, -1)
    dst_row, src_token = g.new((T, K), i32, -1), g.new((P,), i32, -1)
    perm_prob = g.new((P,), torch.float32, float("nan"))
    M.moe_permute_mxfp8(cfg, x, idx, prob, xq, xsf, counts, offsets, dst_row, src_token, perm_prob, ws)
    w1q = g.new((E * 2 * F, h), u8, 0)
    w1sf = g.new((M.moe_mxfp8_scale_bytes(E * 2 * F, h, E),), u8, 0)
    w2q = g.new((E * h, F), u8, 0)
    w2sf = g.new((M.moe_mxfp8_scale_bytes(E * h, F, E),), u8, 0)
    M.moe_mxfp8_quantize(E * 2 * F, h, E, None, w1, w1q, w1sf)
    M.moe_mxfp8_quantize(E * h, F, E, None, w2, w2q, w2sf)
    a = g.new((P, F), torch.bfloat16, float("nan"))
    aq = g.new((P, F), u8, 0)
    asf = g.new((M.moe_mxfp8_scale_bytes(P, F, E),), u8, 0)
    M.moe_expert_fc1_mxfp8(cfg, xq, xsf, offsets, perm_prob, w1q, w1sf, a, aq, asf)
    y_perm = g.new((P, h), torch.bfloat16, float("nan"))
    M.moe_expert_fc2_mxfp8(cfg, aq, asf, offsets, w2q, w2sf, y_perm)
    assert M.moe_get_error() == M.MOE_OK
    g.check()
    assert torch.isfinite(y_perm.float()).all()


def test_injected_cuda_failures_enqueue_nothing_and_the_library_recovers():
    M = lib()
    T, h, E, K = 200, 128, 8, 2
    x = to_dev(inputs.normal((T, h), 1.0, 21, 1, "bf16"), "bf16")
    w_r = to_dev(inputs.normal((E, h), 0.02, 21, 2), "f32")
    cfg = M.make_config(T, h, E, K, 64, M.MOE_BF16, M.MOE_SCORE_SOFTMAX, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    ref_prob = torch.empty(T, K, device="cuda")
    M.moe_router_topk(cfg, x, w_r, None, None, None, ref_idx, ref_prob, None, ws)
    torch.cuda.synchronize()
    assert M.moe_test_inject_cuda_failure(2) == 0
    for _ in range(2):
        idx = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
        prob = torch.full((T, K), float("nan"), device="cuda")
        with pytest.raises(M.MoeError) as ei:
            M.moe_router_topk(cfg, x, w_r, None, None, None, idx, prob, None, ws)
        assert ei.value.status == M.MOE_ERR_CUDA
        torch.cuda.synchronize()
        assert (idx == -9).all() and torch.isnan(prob).all()  # nothing was enqueued
    assert M.moe_get_error() == M.MOE_OK                        # not consumed by the status read
    M.moe_router_topk(cfg, x, w_r, None, None, None, idx, prob, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(idx, ref_idx) and torch.equal(prob, ref_prob)
    assert M.moe_test_inject_cuda_failure(0) == 0
