"""Helpers for the GPU parity tests: seeded host inputs -> device tensors,
the tolerance of the layer's outputs, and oracle calls on the same inputs."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from mixture_experts_layer_softmax_gb300 import inputs, workloads
from oracle import moe_oracle as O

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def lib():
    from mixture_experts_layer_softmax_gb300 import _build
    _build.build()
    from mixture_experts_layer_softmax_gb300 import moe
    return moe


def to_dev(a: np.ndarray, dtype: str):
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def to_np(t):
    return t.float().cpu().numpy() if t.dtype in (torch.bfloat16, torch.float16) else t.cpu().numpy()


def tol_ok(gpu, ref, dtype):
    """The output tolerance: bf16 max|g - o| <= 2e-2 max|o| + 1e-3,
    fp32 max|g - o| <= 1e-4 max|o|.  Returns (ok, err, bound)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    bound = 2e-2 * scale + 1e-3 if dtype == "bf16" else 1e-4 * scale
    return err <= bound, err, bound


def check_routing(gpu_idx, gpu_prob, ref_idx, ref_prob, logits, K, score, sel_bias=None,
                  force_balance=False, prob_rtol=1e-5):
    """Routing parity: the selected set of every token whose K-th/(K+1)-th key
    gap is >= 1e-5, the listing order where every gap inside the top K+1 is
    >= 1e-5 (near-equal keys may be listed either way), probabilities per
    (token, expert).  Returns the mask of tokens whose selection is unique."""
    T = ref_idx.shape[0]
    if force_balance:
        sel_ok = ord_ok = np.ones(T, bool)
    else:
        sel_ok = O.selection_margin(logits, K, score, sel_bias) >= 1e-5
        ord_ok = sel_ok & (O.order_margin(logits, K, score, sel_bias) >= 1e-5)
    assert sel_ok.mean() > 0.98
    np.testing.assert_array_equal(gpu_idx[ord_ok], ref_idx[ord_ok])
    gs, rs = np.argsort(gpu_idx, 1), np.argsort(ref_idx, 1)
    g_sorted = np.take_along_axis(gpu_idx, gs, 1)
    r_sorted = np.take_along_axis(ref_idx, rs, 1)
    np.testing.assert_array_equal(g_sorted[sel_ok], r_sorted[sel_ok])
    if gpu_prob is not None:
        np.testing.assert_allclose(np.take_along_axis(gpu_prob, gs, 1)[sel_ok],
                                   np.take_along_axis(ref_prob, rs, 1)[sel_ok],
                                   rtol=prob_rtol, atol=1e-6)
    return sel_ok


class Layer:
    """A workload's seeded host inputs and their device copies."""

    def __init__(self, w: workloads.Workload):
        self.w = w
        self.h = {r: w.host(r) for r in w.roles()}
        self.d = {r: to_dev(a, w.tensor_dtype(r)) for r, a in self.h.items()}

    def get(self, role):
        return self.d.get(role)

    def oracle_fwd(self, tokens=None):
        w, h = self.w, self.h
        return O.layer_fwd(h["x"], h["w_r"], h["w1"], h["w2"], w.K, w.score, w.act,
                           b1=h.get("b1"), b2=h.get("b2"), sel_bias=h.get("sel_bias"),
                           gate_bias=h.get("gate_bias"), renorm=w.renorm,
                           force_balance=w.force_balance, w1_shared=h.get("w1_shared"),
                           w2_shared=h.get("w2_shared"), tokens=tokens)

    def margins(self, logits):
        w = self.w
        if w.force_balance:
            return np.full(w.T, np.inf)
        return O.selection_margin(logits, w.K, w.score, self.h.get("sel_bias"))

    def run_fwd(self, M, flags_extra=0, ws=None, cfg=None):
        w = self.w
        cfg = cfg if cfg is not None else M.config_for(w, flags_extra)
        if ws is None:
            ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        y = torch.empty(w.T, w.h, dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float32,
                        device="cuda")
        idx = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
        prob = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
        g = self.get
        M.moe_layer_fwd(cfg, g("x"), g("w_r"), g("gate_bias"), g("sel_bias"), g("w1"), g("b1"),
                        g("w2"), g("b2"), g("w1_shared"), g("w2_shared"), y, idx, prob, ws)
        torch.cuda.synchronize()
        assert M.moe_get_error() == M.MOE_OK
        return y, idx, prob, ws
