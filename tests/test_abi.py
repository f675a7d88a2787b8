"""The C-ABI library loads on a CPU-only host, exports every symbol
include/moe.h declares, and rejects bad arguments before touching CUDA
(these calls return before any CUDA runtime call, so they run without a GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def M():
    from mixture_experts_layer_softmax_gb300 import _build
    _build.build()
    from mixture_experts_layer_softmax_gb300 import moe
    return moe


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(M):
    names = declared_functions()
    assert "moe_layer_fwd" in names and "moe_router_topk" in names
    lib = ctypes.CDLL(M.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(M.exported_symbols())


def test_version_and_status_strings(M):
    assert M.moe_version().count(".") == 2
    assert M.moe_status_string(M.MOE_ERR_WORKSPACE) == "workspace missing or too small"
    assert M.moe_status_string(99) == "unknown status"


def _cfg(M, **kw):
    base = dict(T=64, h=128, E=8, K=2, F=256, dtype=M.MOE_BF16, score=M.MOE_SCORE_SOFTMAX,
                act=M.MOE_ACT_SWIGLU, has_bias=0, n_shared=0, flags=M.MOE_FLAG_RENORM)
    base.update(kw)
    return M.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(K=9), 1), (dict(T=-1), 1), (dict(h=0), 1), (dict(dtype=7), 1), (dict(flags=1 << 20), 1),
    (dict(E=300, K=2), 2), (dict(K=17, E=64), 2), (dict(h=100), 2), (dict(F=20), 2),
    (dict(act=1, has_bias=1), 2), (dict(n_shared=2), 1),
    (dict(aux_loss_coeff=float("nan")), 1), (dict(z_loss_coeff=float("inf")), 1),
])
def test_config_rejections(M, kw, status):
    cfg = _cfg(M, **kw)
    assert M.moe_workspace_size(cfg) == 0
    f = M.raw("moe_layer_fwd")
    fake = 1 << 20  # never dereferenced: validation fails first
    st = f(ctypes.byref(cfg), fake, fake, None, None, fake, None, fake, None, None, None, fake,
           None, None, fake, 1 << 40, None)
    assert st == status


def test_workspace_size_monotone_and_aligned(M):
    a = M.moe_workspace_size(_cfg(M))
    b = M.moe_workspace_size(_cfg(M, T=128))
    c = M.moe_workspace_size(_cfg(M, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_SAVE_FOR_BWD))
    assert 0 < a < b and c > a and a % 256 == 0


def test_validate_only_and_workspace_errors(M):
    cfg = _cfg(M, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_VALIDATE_ONLY)
    need = M.moe_workspace_size(cfg)
    f = M.raw("moe_layer_fwd")
    P = 1 << 20  # fake aligned addresses, never touched under VALIDATE_ONLY
    args = [P, P, None, None, P, None, P, None, None, None, P, None, None]
    assert f(ctypes.byref(cfg), *args, P, need, None) == M.MOE_OK
    assert f(ctypes.byref(cfg), *args, P, need - 1, None) == M.MOE_ERR_WORKSPACE
    assert f(ctypes.byref(cfg), *args, None, need, None) == M.MOE_ERR_WORKSPACE
    assert f(ctypes.byref(cfg), *args, P + 128, need, None) == M.MOE_ERR_INVALID_ARG  # ws alignment
    bad = list(args)
    bad[0] = P + 4  # x misaligned
    assert f(ctypes.byref(cfg), *bad, P, need, None) == M.MOE_ERR_INVALID_ARG
    bad = list(args)
    bad[1] = None  # w_r missing
    assert f(ctypes.byref(cfg), *bad, P, need, None) == M.MOE_ERR_INVALID_ARG
    shared = _cfg(M, n_shared=1, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_VALIDATE_ONLY)
    assert f(ctypes.byref(shared), *args, P, 1 << 40, None) == M.MOE_ERR_INVALID_ARG


def test_other_entry_points_validate(M):
    cfg = _cfg(M, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_VALIDATE_ONLY)
    P = 1 << 20
    big = 1 << 40
    assert M.raw("moe_router_topk_from_logits")(ctypes.byref(cfg), P, None, P, P, None, None) == 0
    assert M.raw("moe_router_topk_from_logits")(ctypes.byref(cfg), None, None, P, P, None, None) == 1
    assert M.raw("moe_permute")(ctypes.byref(cfg), P, P, P, None, P, P, P, P, P, P, big, None) == 1
    assert M.raw("moe_permute")(ctypes.byref(cfg), P, P, P, P, P, P, P, P, P, P, big, None) == 0
    assert M.raw("moe_permute")(ctypes.byref(cfg), P, P, P, P, P, P, P, P, P, None, 0, None) == 3
    assert M.raw("moe_unpermute_combine")(ctypes.byref(cfg), P, P, None, None, P, None) == 0
    assert M.raw("moe_unpermute_combine")(ctypes.byref(cfg), P + 8, P, None, None, P, None) == 1
    assert M.raw("moe_grouped_mlp_fwd")(ctypes.byref(cfg), P, P, P, P, None, P, None, None, P, P,
                                        big, None) == 0
    gelu_b = _cfg(M, act=M.MOE_ACT_GELU, has_bias=1, flags=M.MOE_FLAG_VALIDATE_ONLY)
    assert M.raw("moe_grouped_mlp_fwd")(ctypes.byref(gelu_b), P, P, P, P, None, P, None, None, P,
                                        P, big, None) == 1
    assert M.raw("moe_test_bounded_wait")(0, None) == 1
    nal = M.raw("moe_permute_noalloc")
    assert nal(ctypes.byref(cfg), P, P, P, P, P, P, P, P, P, None) == M.MOE_OK
    assert nal(ctypes.byref(cfg), None, P, P, None, P, P, P, P, P, None) == M.MOE_OK  # maps only
    assert nal(ctypes.byref(cfg), P, P, P, None, P, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert nal(ctypes.byref(cfg), P + 8, P, P, P, P, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert nal(ctypes.byref(cfg), P, P, P, P, None, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert nal(ctypes.byref(cfg), P, None, P, P, P, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert nal(None, P, P, P, P, P, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG


def test_mxfp8_argument_checks(M):
    assert M.moe_mxfp8_scale_bytes(1000, 256, 4) == (8 + 4) * 2 * 512
    assert M.moe_mxfp8_scale_bytes(4096 * 4, 7168, 256 // 256) == (128 + 1) * 56 * 512
    assert M.moe_mxfp8_scale_bytes(10, 100, 1) == 0      # K not a multiple of 128
    assert M.moe_mxfp8_scale_bytes(10, 128, 0) == 0
    q = M.raw("moe_mxfp8_quantize")
    P = 1 << 20  # fake aligned addresses: validation fails (or returns) first
    assert q(10, 96, 1, None, P, P, P, None) == M.MOE_ERR_UNSUPPORTED
    assert q(10, 128, 3, None, P, P, P, None) == M.MOE_ERR_INVALID_ARG  # 10 % 3 != 0
    assert q(10, 128, 1, None, None, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert q(10, 128, 1, None, P + 8, P, P, None) == M.MOE_ERR_INVALID_ARG
    assert q(0, 128, 1, None, None, None, None, None) == M.MOE_OK
    assert q(10, 128, 300, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG   # > 256 groups
    f1 = M.raw("moe_expert_fc1_mxfp8")
    f2 = M.raw("moe_expert_fc2_mxfp8")
    ok = _cfg(M, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_VALIDATE_ONLY)
    assert f1(ctypes.byref(ok), P, P, P, None, P, P, P, None, None, None) == M.MOE_OK
    assert f1(ctypes.byref(ok), P, P, P, None, P, P, None, P, P, None) == M.MOE_OK
    assert f1(ctypes.byref(ok), P, P, P, None, P, P, None, None, None, None) == M.MOE_ERR_INVALID_ARG
    assert f1(ctypes.byref(ok), P, P, P, None, P, P, None, P, None, None) == M.MOE_ERR_INVALID_ARG
    assert f2(ctypes.byref(ok), P, P, P, P, P, P, None) == M.MOE_OK
    assert f2(ctypes.byref(ok), P, None, P, P, P, P, None) == M.MOE_ERR_INVALID_ARG
    for kw in (dict(act=M.MOE_ACT_GELU), dict(F=192), dict(h=200), dict(dtype=M.MOE_F32, h=128)):
        bad = _cfg(M, flags=M.MOE_FLAG_RENORM | M.MOE_FLAG_VALIDATE_ONLY, **kw)
        assert f1(ctypes.byref(bad), P, P, P, None, P, P, P, None, None, None) == M.MOE_ERR_UNSUPPORTED
        assert f2(ctypes.byref(bad), P, P, P, P, P, P, None) == M.MOE_ERR_UNSUPPORTED


def test_failure_injection_counter(M):
    assert M.moe_test_inject_cuda_failure(3) == 0
    assert M.moe_test_inject_cuda_failure(0) == 3   # cleared, the pending count returned
    assert M.moe_test_inject_cuda_failure(-1) == -1
    assert M.moe_test_inject_cuda_failure(0) == 0


def test_stage_event_registration_checks(M):
    f = M.raw("moe_set_stage_events")
    arr = (ctypes.c_void_p * 17)()
    assert f(0, arr, 0) == M.MOE_OK and f(1, None, 0) == M.MOE_OK   # clear
    assert f(2, arr, 1) == M.MOE_ERR_INVALID_ARG                    # unknown pass
    assert f(0, arr, 17) == M.MOE_ERR_INVALID_ARG                   # more than 16
    assert f(0, None, 3) == M.MOE_ERR_INVALID_ARG
    assert f(1, arr, 16) == M.MOE_OK and f(1, arr, 0) == M.MOE_OK   # NULL entries are skipped
