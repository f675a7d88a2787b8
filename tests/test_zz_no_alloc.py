"""moe_permute_noalloc: dispatch for callers that cannot allocate device
memory (plugins of a framework that owns all device memory, serving loops
that must not allocate after start-up).  It must give exactly what
moe_permute gives, call after call, although every call reuses the same
fixed scratch array inside the library.  This file is collected last."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import lib, needs_gpu, to_dev
from mixture_experts_layer_softmax_gb300 import inputs
from oracle import moe_oracle as O

pytestmark = [pytest.mark.gpu, needs_gpu]


def _buffers(T, E, K, h):
    P = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(x_perm=torch.full((P, h), -1.0, dtype=torch.bfloat16, device="cuda"),
                counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
                dst_row=torch.full((T, K), -1, **i32), src_token=torch.full((P,), -1, **i32),
                perm_prob=torch.full((P,), -1.0, device="cuda"))


def _routing(T, E, K, seed):
    logits = inputs.normal((T, E), 1.0, seed, 1)
    return O.route(logits, K, O.SCORE_SOFTMAX)


@pytest.mark.parametrize("shapes", [[(4096, 128, 8, 256), (300, 8, 2, 64)],
                                    [(32768, 256, 8, 64), (33, 3, 3, 128)]])
def test_noalloc_matches_permute_on_consecutive_calls(shapes):
    M = lib()
    for call, (T, E, K, h) in enumerate(shapes):
        idx, prob = _routing(T, E, K, seed=40 + call)
        x = to_dev(inputs.normal((T, h), 1.0, 41 + call, 1, "bf16"), "bf16")
        idx_d, prob_d = torch.from_numpy(idx).cuda(), to_dev(prob, "f32")
        cfg = M.make_config(T, h, E, K, 8)
        ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        want = _buffers(T, E, K, h)
        M.moe_permute(cfg, x, idx_d, prob_d, want["x_perm"], want["counts"], want["offsets"],
                      want["dst_row"], want["src_token"], want["perm_prob"], ws)
        got = _buffers(T, E, K, h)
        st = M.raw("moe_permute_noalloc")(
            ctypes.byref(cfg), x.data_ptr(), idx_d.data_ptr(), prob_d.data_ptr(),
            got["x_perm"].data_ptr(), got["counts"].data_ptr(), got["offsets"].data_ptr(),
            got["dst_row"].data_ptr(), got["src_token"].data_ptr(), got["perm_prob"].data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert st == M.MOE_OK
        torch.cuda.synchronize()
        assert M.moe_get_error() == M.MOE_OK
        for k in want:  # integer maps and copied rows: bit-exact
            a, b = want[k], got[k]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), (call, k)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    M = lib()
    cfg = M.make_config(32800, 64, 256, 8, 8)  # ceil(32800/32) * 256 > 262144
    st = M.raw("moe_permute_noalloc")(ctypes.byref(cfg), None, 1 << 20, None, None, 1 << 20,
                                       1 << 20, 1 << 20, 1 << 20, None, None)
    assert st == M.MOE_ERR_UNSUPPORTED


def test_noalloc_reports_bad_expert_ids_without_faulting():
    """An out-of-range expert id is skipped and reported through the status
    word, as moe_permute does; the next call on the shared scratch is clean."""
    M = lib()
    T, E, K, h = 64, 8, 2, 32
    P = T * K
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[5, 1] = 99
    cfg = M.make_config(T, h, E, K, 8, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)
    x = torch.zeros(T, h, dtype=torch.bfloat16, device="cuda")
    x_perm = torch.zeros(P, h, dtype=torch.bfloat16, device="cuda")
    out = [torch.zeros(n, dtype=torch.int32, device="cuda") for n in (E, E + 1, P, P)]
    M.moe_permute_noalloc(cfg, x, torch.from_numpy(idx).cuda(), None, x_perm, out[0], out[1],
                          out[2], out[3], None)
    assert M.moe_get_error() == M.MOE_ERR_DEVICE_BOUNDS
    assert M.moe_get_error() == M.MOE_OK
    assert int(out[1][-1]) == P - 1
    idx[5, 1] = 2
    M.moe_permute_noalloc(cfg, x, torch.from_numpy(idx).cuda(), None, x_perm, out[0], out[1],
                          out[2], out[3], None)
    assert M.moe_get_error() == M.MOE_OK
    assert int(out[1][-1]) == P


def test_noalloc_injected_failure_enqueues_nothing():
    M = lib()
    T, E, K, h = 100, 8, 2, 64
    P = T * K
    idx, prob = _routing(T, E, K, seed=7)
    cfg = M.make_config(T, h, E, K, 8)
    x = to_dev(inputs.normal((T, h), 1.0, 8, 1, "bf16"), "bf16")
    bufs = _buffers(T, E, K, h)
    assert M.moe_test_inject_cuda_failure(1) == 0
    with pytest.raises(M.MoeError) as ei:
        M.moe_permute_noalloc(cfg, x, torch.from_numpy(idx).cuda(), to_dev(prob, "f32"),
                              bufs["x_perm"], bufs["counts"], bufs["offsets"], bufs["dst_row"],
                              bufs["src_token"], bufs["perm_prob"])
    assert ei.value.status == M.MOE_ERR_CUDA
    torch.cuda.synchronize()
    assert (bufs["counts"] == -1).all() and (bufs["dst_row"] == -1).all()
    assert M.moe_test_inject_cuda_failure(0) == 0
    M.moe_permute_noalloc(cfg, x, torch.from_numpy(idx).cuda(), to_dev(prob, "f32"),
                          bufs["x_perm"], bufs["counts"], bufs["offsets"], bufs["dst_row"],
                          bufs["src_token"], bufs["perm_prob"])
    torch.cuda.synchronize()
    assert int(bufs["offsets"][-1]) == P
