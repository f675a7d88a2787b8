"""Python binding of the C ABI in include/moe.h (ctypes; argument marshalling
only).  Every function here has the C entry point's name and forwards torch
tensors' device pointers and the current CUDA stream; all computation runs in
the library's CUDA kernels.  There is no fallback: if the library has not been
built (``mixture_experts_layer_softmax_gb300._build.build()``) importing this
module raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libmoe_gb300.so")
SYNTH_PATH = os.path.join(PKG, "_build", "libmoe_synth.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

# ---- enums (moe.h) ----------------------------------------------------------
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID = 0, 1
MOE_ACT_GELU, MOE_ACT_SWIGLU = 0, 1
MOE_FLAG_RENORM, MOE_FLAG_FORCE_BALANCE = 1, 2
MOE_FLAG_VALIDATE_ONLY, MOE_FLAG_SAVE_FOR_BWD, MOE_FLAG_GEMM_SIMT = 8, 16, 32
MOE_FLAG_GEMM_1CTA, MOE_FLAG_GEMM_2CTA = 64, 128
MOE_FLAG_HIST_FROM_ROUTER = 256


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("h", ctypes.c_int32), ("E", ctypes.c_int32),
                ("K", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("score", ctypes.c_int32), ("act", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("aux_loss_coeff", ctypes.c_float), ("z_loss_coeff", ctypes.c_float),
                ("capacity", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {moe_status_string(status)} ({status})")


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config_t)
_SIG = {
    "moe_workspace_size": (ctypes.c_size_t, [_CFG]),
    "moe_router_topk": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_router_topk_from_logits": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_permute": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "moe_permute_noalloc": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_mlp_fwd": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_size_t, _P]),
    "moe_expert_fc1": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_fc2": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P]),
    "moe_expert_fc1_gather": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_mxfp8_scale_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    "moe_mxfp8_quantize": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                          _P, _P, _P]),
    "moe_permute_mxfp8": (ctypes.c_int, [_CFG] + [_P] * 11 + [ctypes.c_size_t, _P]),
    "moe_expert_fc1_mxfp8": (ctypes.c_int, [_CFG] + [_P] * 10),
    "moe_expert_fc2_mxfp8": (ctypes.c_int, [_CFG] + [_P] * 7),
    "moe_unpermute_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_layer_fwd": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                     ctypes.c_size_t, _P]),
    "moe_grouped_mlp_bwd": (ctypes.c_int, [_CFG] + [_P] * 13 + [ctypes.c_size_t, _P]),
    "moe_router_bwd": (ctypes.c_int, [_CFG] + [_P] * 14 + [ctypes.c_size_t, _P]),
    "moe_layer_bwd": (ctypes.c_int, [_CFG] + [_P] * 15 + [ctypes.c_size_t, _P]),
    "moe_layer_losses": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_size_t, _P]),
    "moe_expert_capacity": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_float, ctypes.c_int32]),
    "moe_router_aux_loss": (ctypes.c_int, [_CFG, _P, _P, ctypes.c_float, ctypes.c_float, _P, _P,
                                           _P, ctypes.c_size_t, _P]),
    "moe_get_error": (ctypes.c_int, [_P]),
    "moe_set_stage_events": (ctypes.c_int, [ctypes.c_int32, ctypes.POINTER(ctypes.c_void_p),
                                            ctypes.c_int32]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_test_bounded_wait": (ctypes.c_int, [ctypes.c_int64, _P]),
    "moe_test_inject_cuda_failure": (ctypes.c_int32, [ctypes.c_int32]),
}
for _name, (_res, _args) in _SIG.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def exported_symbols():
    return list(_SIG)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st)


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws), ws.numel() * ws.element_size()


def make_config(T, h, E, K, F, dtype=MOE_BF16, score=MOE_SCORE_SOFTMAX, act=MOE_ACT_SWIGLU,
                has_bias=0, n_shared=0, flags=MOE_FLAG_RENORM, aux_loss_coeff=0.0,
                z_loss_coeff=0.0, capacity=0) -> moe_config_t:
    return moe_config_t(int(T), int(h), int(E), int(K), int(F), int(dtype), int(score), int(act),
                        int(has_bias), int(n_shared), int(flags), float(aux_loss_coeff),
                        float(z_loss_coeff), int(capacity))


def config_for(w, flags_extra=0, aux_loss_coeff=0.0, z_loss_coeff=0.0, capacity=0) -> moe_config_t:
    """moe_config_t of a workloads.Workload."""
    flags = (MOE_FLAG_RENORM if w.renorm else 0) | (MOE_FLAG_FORCE_BALANCE if w.force_balance else 0)
    return make_config(w.T, w.h, w.E, w.K, w.F, MOE_BF16 if w.dtype == "bf16" else MOE_F32,
                       w.score, w.act, int(w.has_bias), w.n_shared, flags | flags_extra,
                       aux_loss_coeff, z_loss_coeff, capacity)


# ---- entry points -------------------------------------------------------------
def moe_status_string(status) -> str:
    return _lib.moe_status_string(int(status)).decode()


def moe_version() -> str:
    return _lib.moe_version().decode()


def moe_expert_capacity(T, K, E, capacity_factor, min_capacity=0) -> int:
    return int(_lib.moe_expert_capacity(int(T), int(K), int(E), float(capacity_factor),
                                        int(min_capacity)))


def moe_workspace_size(cfg) -> int:
    return int(_lib.moe_workspace_size(ctypes.byref(cfg)))


def moe_router_topk(cfg, x, w_r, gate_bias, sel_bias, logits, topk_idx, topk_prob,
                    routing_map=None, ws=None, stream=None):
    wp, wb = _ws(ws)
    _check("moe_router_topk", _lib.moe_router_topk(
        ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(gate_bias), _ptr(sel_bias), _ptr(logits),
        _ptr(topk_idx), _ptr(topk_prob), _ptr(routing_map), wp, wb, _stream(stream)))


def moe_router_topk_from_logits(cfg, logits, sel_bias, topk_idx, topk_prob, routing_map=None,
                                stream=None):
    _check("moe_router_topk_from_logits", _lib.moe_router_topk_from_logits(
        ctypes.byref(cfg), _ptr(logits), _ptr(sel_bias), _ptr(topk_idx), _ptr(topk_prob),
        _ptr(routing_map), _stream(stream)))


def moe_permute(cfg, x, topk_idx, topk_prob, x_perm, counts, offsets, dst_row, src_token,
                perm_prob, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_permute", _lib.moe_permute(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_prob), _ptr(x_perm), _ptr(counts),
        _ptr(offsets), _ptr(dst_row), _ptr(src_token), _ptr(perm_prob), wp, wb, _stream(stream)))


def moe_permute_noalloc(cfg, x, topk_idx, topk_prob, x_perm, counts, offsets, dst_row, src_token,
                        perm_prob, stream=None):
    """moe_permute for callers that cannot allocate device memory: no
    workspace; the library's fixed scratch array is used (see moe.h)."""
    _check("moe_permute_noalloc", _lib.moe_permute_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_prob), _ptr(x_perm), _ptr(counts),
        _ptr(offsets), _ptr(dst_row), _ptr(src_token), _ptr(perm_prob), _stream(stream)))


def moe_grouped_mlp_fwd(cfg, x_perm, offsets, perm_prob, w1, b1, w2, b2, act_save, y_perm, ws,
                        stream=None):
    wp, wb = _ws(ws)
    _check("moe_grouped_mlp_fwd", _lib.moe_grouped_mlp_fwd(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(perm_prob), _ptr(w1), _ptr(b1),
        _ptr(w2), _ptr(b2), _ptr(act_save), _ptr(y_perm), wp, wb, _stream(stream)))


def moe_expert_fc1(cfg, x_perm, offsets, perm_prob, w1, b1, act_save, a, stream=None):
    _check("moe_expert_fc1", _lib.moe_expert_fc1(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(perm_prob), _ptr(w1), _ptr(b1),
        _ptr(act_save), _ptr(a), _stream(stream)))


def moe_expert_fc1_gather(cfg, x, src_token, offsets, perm_prob, w1, b1, act_save, a,
                          stream=None):
    _check("moe_expert_fc1_gather", _lib.moe_expert_fc1_gather(
        ctypes.byref(cfg), _ptr(x), _ptr(src_token), _ptr(offsets), _ptr(perm_prob), _ptr(w1),
        _ptr(b1), _ptr(act_save), _ptr(a), _stream(stream)))


def moe_expert_fc2(cfg, a, offsets, perm_prob, w2, b2, y_perm, stream=None):
    _check("moe_expert_fc2", _lib.moe_expert_fc2(
        ctypes.byref(cfg), _ptr(a), _ptr(offsets), _ptr(perm_prob), _ptr(w2), _ptr(b2),
        _ptr(y_perm), _stream(stream)))


def moe_mxfp8_scale_bytes(rows, K, groups) -> int:
    return int(_lib.moe_mxfp8_scale_bytes(int(rows), int(K), int(groups)))


def moe_mxfp8_quantize(rows, K, groups, offsets, x, q, sf, stream=None):
    _check("moe_mxfp8_quantize", _lib.moe_mxfp8_quantize(
        int(rows), int(K), int(groups), _ptr(offsets), _ptr(x), _ptr(q), _ptr(sf),
        _stream(stream)))


def moe_permute_mxfp8(cfg, x, topk_idx, topk_prob, x_q, x_sf, counts, offsets, dst_row,
                      src_token, perm_prob, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_permute_mxfp8", _lib.moe_permute_mxfp8(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(topk_prob), _ptr(x_q), _ptr(x_sf),
        _ptr(counts), _ptr(offsets), _ptr(dst_row), _ptr(src_token), _ptr(perm_prob), wp, wb,
        _stream(stream)))


def moe_expert_fc1_mxfp8(cfg, x_q, x_sf, offsets, perm_prob, w1_q, w1_sf, a, a_q, a_sf,
                         stream=None):
    _check("moe_expert_fc1_mxfp8", _lib.moe_expert_fc1_mxfp8(
        ctypes.byref(cfg), _ptr(x_q), _ptr(x_sf), _ptr(offsets), _ptr(perm_prob), _ptr(w1_q),
        _ptr(w1_sf), _ptr(a), _ptr(a_q), _ptr(a_sf), _stream(stream)))


def moe_expert_fc2_mxfp8(cfg, a_q, a_sf, offsets, w2_q, w2_sf, y_perm, stream=None):
    _check("moe_expert_fc2_mxfp8", _lib.moe_expert_fc2_mxfp8(
        ctypes.byref(cfg), _ptr(a_q), _ptr(a_sf), _ptr(offsets), _ptr(w2_q), _ptr(w2_sf),
        _ptr(y_perm), _stream(stream)))


def moe_unpermute_combine(cfg, y_perm, dst_row, topk_prob, shared_y, y, stream=None):
    _check("moe_unpermute_combine", _lib.moe_unpermute_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(dst_row), _ptr(topk_prob), _ptr(shared_y), _ptr(y),
        _stream(stream)))


def moe_layer_fwd(cfg, x, w_r, gate_bias, sel_bias, w1, b1, w2, b2, w1_shared, w2_shared, y,
                  topk_idx_out=None, topk_prob_out=None, ws=None, stream=None):
    wp, wb = _ws(ws)
    _check("moe_layer_fwd", _lib.moe_layer_fwd(
        ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(gate_bias), _ptr(sel_bias), _ptr(w1),
        _ptr(b1), _ptr(w2), _ptr(b2), _ptr(w1_shared), _ptr(w2_shared), _ptr(y),
        _ptr(topk_idx_out), _ptr(topk_prob_out), wp, wb, _stream(stream)))


def moe_grouped_mlp_bwd(cfg, dy_perm, x_perm, act_save, a, offsets, perm_prob, w1, w2, dx_perm,
                        dw1, dw2, dprob_perm, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_grouped_mlp_bwd", _lib.moe_grouped_mlp_bwd(
        ctypes.byref(cfg), _ptr(dy_perm), _ptr(x_perm), _ptr(act_save), _ptr(a), _ptr(offsets),
        _ptr(perm_prob), _ptr(w1), _ptr(w2), _ptr(dx_perm), _ptr(dw1), _ptr(dw2), _ptr(dprob_perm),
        wp, wb, _stream(stream)))


def moe_router_bwd(cfg, x, logits, topk_idx, topk_prob, offsets, dst_row, src_token, dprob_perm,
                   w_r, dl_topk, dw_r, db_r, dx_router, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_router_bwd", _lib.moe_router_bwd(
        ctypes.byref(cfg), _ptr(x), _ptr(logits), _ptr(topk_idx), _ptr(topk_prob), _ptr(offsets),
        _ptr(dst_row), _ptr(src_token), _ptr(dprob_perm), _ptr(w_r), _ptr(dl_topk), _ptr(dw_r),
        _ptr(db_r), _ptr(dx_router), wp, wb, _stream(stream)))


def moe_layer_bwd(cfg, x, w_r, w1, w2, w1_shared, w2_shared, dy, dx, dw_r, db_r, dw1, dw2,
                  dw1_shared, dw2_shared, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_layer_bwd", _lib.moe_layer_bwd(
        ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(w1), _ptr(w2), _ptr(w1_shared),
        _ptr(w2_shared), _ptr(dy), _ptr(dx), _ptr(dw_r), _ptr(db_r), _ptr(dw1), _ptr(dw2),
        _ptr(dw1_shared), _ptr(dw2_shared), wp, wb, _stream(stream)))


def moe_router_aux_loss(cfg, logits, topk_idx, aux_coeff, z_coeff, losses, dlogits=None, ws=None,
                        stream=None):
    wp, wb = _ws(ws)
    _check("moe_router_aux_loss", _lib.moe_router_aux_loss(
        ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), float(aux_coeff), float(z_coeff),
        _ptr(losses), _ptr(dlogits), wp, wb, _stream(stream)))


def moe_layer_losses(cfg, losses, ws, stream=None):
    wp, wb = _ws(ws)
    _check("moe_layer_losses", _lib.moe_layer_losses(ctypes.byref(cfg), _ptr(losses), wp, wb,
                                                     _stream(stream)))


def moe_get_error(stream=None) -> int:
    return int(_lib.moe_get_error(_stream(stream)))


MOE_PASS_FWD, MOE_PASS_BWD = 0, 1


def moe_set_stage_events(pass_, events):
    """Registers CUDA events that moe_layer_fwd / moe_layer_bwd record at their
    stage boundaries (moe.h lists them).  `events`: a list of
    torch.cuda.Event (already recorded once, so that the CUDA event exists),
    raw cudaEvent_t integers, or None entries; [] clears the pass."""
    handles = []
    for ev in events:
        if ev is None:
            handles.append(None)
            continue
        hnd = int(getattr(ev, "cuda_event", ev))
        if hnd == 0:
            raise ValueError("a torch.cuda.Event is created lazily: record it once first")
        handles.append(hnd)
    arr = (ctypes.c_void_p * max(len(handles), 1))(*handles)
    _check("moe_set_stage_events", _lib.moe_set_stage_events(int(pass_), arr, len(handles)))


def moe_test_bounded_wait(max_polls, stream=None):
    _check("moe_test_bounded_wait", _lib.moe_test_bounded_wait(int(max_polls), _stream(stream)))


def moe_test_inject_cuda_failure(n) -> int:
    return int(_lib.moe_test_inject_cuda_failure(int(n)))


def raw(name):
    """The raw ctypes function of an entry point (for tests of argument checks)."""
    return getattr(_lib, name)


# ---- seeded device-side inputs (separate library) ------------------------------
_synth = None


def synth_normal(t, seed, tag, std, start=0, stream=None):
    """Fill a contiguous fp32 or bf16 CUDA tensor with the seeded N(0, std^2)
    stream of inputs.py, elements [start, start + numel)."""
    global _synth
    if _synth is None:
        _synth = ctypes.CDLL(SYNTH_PATH)
        _synth.moe_synth_normal.restype = ctypes.c_int
        _synth.moe_synth_normal.argtypes = [_P, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                            ctypes.c_uint64, ctypes.c_double, ctypes.c_int64, _P]
    import torch
    dt = {torch.float32: 0, torch.bfloat16: 1}[t.dtype]
    rc = _synth.moe_synth_normal(_ptr(t), t.numel(), dt, int(seed), int(tag), float(std),
                                 int(start), _stream(stream))
    if rc != 0:
        raise RuntimeError(f"moe_synth_normal failed: cudaError {rc}")
    return t
