"""ctypes front of the C++ oracle (oracle/moe_oracle_ref.cpp): the MoE layer
forward -- route, dispatch maps, layer output -- as plain double-precision
loops.  TEST INFRASTRUCTURE ONLY, like oracle/moe_oracle.py: only tests/,
__graft_entry__.smoke() and bench.py's cpu_baseline / reference legs use it.
It shares no code with the CUDA path; tests pin it against the numpy oracle,
the hand-worked golden files and the layer's invariants."""

from __future__ import annotations

import ctypes

import numpy as np

from oracle import build_oracle

_lib = ctypes.CDLL(build_oracle.build())
_P = ctypes.c_void_p
_i = ctypes.c_int
_lib.moe_oracle_route.argtypes = [_i] * 7 + [_P] * 7
_lib.moe_oracle_dispatch.argtypes = [_i] * 3 + [_P] * 6
_lib.moe_oracle_layer_fwd.argtypes = [_i] * 6 + [_P] * 9 + [_i, _P, _P]
for _f in ("moe_oracle_route", "moe_oracle_dispatch", "moe_oracle_layer_fwd", "moe_oracle_threads"):
    getattr(_lib, _f).restype = _i

SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
ACT_GELU, ACT_SWIGLU = 0, 1


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def threads() -> int:
    return int(_lib.moe_oracle_threads())


def route(x, w_r, K, score, renorm=True, sel_bias=None, gate_bias=None, force_balance=False):
    """(logits [T,E] fp32, idx [T,K] int32, probs [T,K] float64)."""
    x, w_r = _f32(x), _f32(w_r)
    sel_bias, gate_bias = _f32(sel_bias), _f32(gate_bias)
    T, h = x.shape
    E = w_r.shape[0]
    logits = np.empty((T, E), np.float32)
    idx = np.empty((T, K), np.int32)
    probs = np.empty((T, K), np.float64)
    st = _lib.moe_oracle_route(T, h, E, K, int(score), int(bool(renorm)), int(bool(force_balance)),
                               _ptr(x), _ptr(w_r), _ptr(gate_bias), _ptr(sel_bias), _ptr(logits),
                               _ptr(idx), _ptr(probs))
    if st != 0:
        raise ValueError("moe_oracle_route: bad sizes")
    return logits, idx, probs


def dispatch_maps(idx, E):
    """(counts, offsets, dst_row, src_token, src_slot), int64."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, K = idx.shape
    counts, offsets = np.empty(E, np.int64), np.empty(E + 1, np.int64)
    dst_row = np.empty((T, K), np.int64)
    src_token, src_slot = np.empty(T * K, np.int64), np.empty(T * K, np.int64)
    st = _lib.moe_oracle_dispatch(T, E, K, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(dst_row),
                                  _ptr(src_token), _ptr(src_slot))
    if st != 0:
        raise ValueError("moe_oracle_dispatch: expert id out of range")
    return counts, offsets, dst_row, src_token, src_slot


def layer_fwd(x, idx, probs, w1, w2, act, *, b1=None, b2=None, w1_shared=None, w2_shared=None,
              tokens=None):
    """y [n, h] float64 for the listed tokens (all by default) from a given
    routing.  w1 / w2: arrays [E, ...] or {expert: array} holding at least
    the experts the listed tokens select."""
    x = _f32(x)
    idx = np.ascontiguousarray(idx, np.int32)
    probs = np.ascontiguousarray(probs, np.float64)
    T, h = x.shape
    K = idx.shape[1]
    tokens = np.arange(T, dtype=np.int64) if tokens is None else np.ascontiguousarray(tokens, np.int64)
    if isinstance(w1, dict):
        E = max(max(w1) + 1, int(idx.max()) + 1)
        keep1 = {e: _f32(a) for e, a in w1.items()}
        keep2 = {e: _f32(a) for e, a in w2.items()}
    else:
        E = len(w1)
        keep1 = {e: _f32(w1[e]) for e in range(E)}
        keep2 = {e: _f32(w2[e]) for e in range(E)}
    F = next(iter(keep2.values())).shape[1]
    p1 = (ctypes.c_void_p * E)(*[_ptr(keep1.get(e)) for e in range(E)])
    p2 = (ctypes.c_void_p * E)(*[_ptr(keep2.get(e)) for e in range(E)])
    b1, b2 = _f32(b1), _f32(b2)
    w1s, w2s = _f32(w1_shared), _f32(w2_shared)
    y = np.empty((tokens.size, h), np.float64)
    st = _lib.moe_oracle_layer_fwd(T, h, E, K, F, int(act), _ptr(x), _ptr(idx), _ptr(probs), p1, p2,
                                   _ptr(b1), _ptr(b2), _ptr(w1s), _ptr(w2s), int(tokens.size),
                                   _ptr(tokens), _ptr(y))
    if st != 0:
        raise ValueError("moe_oracle_layer_fwd: a listed token selects an expert without weights")
    return y
