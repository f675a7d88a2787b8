"""Pins for the oracle's Dispatch / Combine maps: hand-worked maps, counting
invariants, bijection, stable order, and permute-then-unpermute identity."""

import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    d = {"idx": [], "dst": []}
    for line in open(os.path.join(GOLDEN, "dispatch_4tok.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        vals = [int(v) for v in f[1:]]
        if f[0] in ("idx", "dst"):
            d[f[0]].append(vals)
        else:
            d[f[0]] = vals
    return d


def test_dispatch_hand_example():
    g = _golden()
    idx = np.array(g["idx"], np.int32)
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(idx, 3)
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert dst_row.tolist() == g["dst"]
    assert src_token.tolist() == g["src_token"]


@pytest.mark.parametrize("T,E,K", [(1, 1, 1), (3, 2, 2), (127, 8, 2), (300, 64, 8), (64, 3, 3)])
def test_dispatch_invariants(T, E, K):
    rng = np.random.default_rng(T * 31 + E)
    l = rng.normal(size=(T, E)).astype(np.float32)
    idx, _ = O.route(l, K, O.SCORE_SOFTMAX)
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(idx, E)
    P = T * K
    assert counts.sum() == P
    assert offsets[0] == 0 and offsets[-1] == P
    assert (np.diff(offsets) == counts).all()
    # bijection between (t, k) pairs and rows
    assert sorted(dst_row.ravel().tolist()) == list(range(P))
    for t in range(T):
        for k in range(K):
            r = dst_row[t, k]
            assert src_token[r] == t and src_slot[r] == k
            assert offsets[idx[t, k]] <= r < offsets[idx[t, k] + 1]
    # ascending token order inside every expert segment
    for e in range(E):
        seg = src_token[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()


def test_permute_unpermute_identity():
    rng = np.random.default_rng(7)
    T, E, K, h = 50, 6, 3, 5
    x = rng.normal(size=(T, h))
    idx, _ = O.route(rng.normal(size=(T, E)).astype(np.float32), K, O.SCORE_SOFTMAX)
    _, _, dst_row, src_token, _ = O.dispatch_maps(idx, E)
    xp = O.permute_rows(x, src_token)
    assert xp.shape == (T * K, h)
    back = O.unpermute_combine(xp, dst_row, np.full((T, K), 1.0 / K))
    np.testing.assert_allclose(back, x, rtol=1e-15, atol=1e-15)
    for k in range(K):
        assert (xp[dst_row[:, k]] == x).all()


def test_empty_experts_and_single_expert():
    idx = np.zeros((5, 1), np.int32)
    counts, offsets, dst_row, src_token, _ = O.dispatch_maps(idx, 4)
    assert counts.tolist() == [5, 0, 0, 0]
    assert offsets.tolist() == [0, 5, 5, 5, 5]
    assert dst_row[:, 0].tolist() == [0, 1, 2, 3, 4]


def test_force_balanced_counts():
    T, K, E = 2048, 8, 256
    idx = O.force_balanced_topk(T, K, E)
    counts = O.dispatch_maps(idx, E)[0]
    assert (counts == T * K // E).all()
