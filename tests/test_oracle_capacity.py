"""Pins for the oracle's expert capacity (token dropping): a hand-worked
dispatch (tests/golden/capacity_4tok.txt), the capacity formula, a capacity at
least the largest load reproducing the dropless layer, kept slots being each
expert's first C in token order, the masked-dense formulation (positions from
a cumulative sum) agreeing with the permuted one, and central finite
differences of the layer backward with the drop pattern held fixed."""

import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "capacity_4tok.txt")


def _golden():
    d = {"idx": [], "keep": [], "dst": []}
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        vals = [int(v) for v in f[1:]]
        if f[0] in d and isinstance(d[f[0]], list) and f[0] in ("idx", "keep", "dst"):
            d[f[0]].append(vals)
        else:
            d[f[0]] = vals
    return d


def test_capacity_hand_example():
    g = _golden()
    idx = np.array(g["idx"], np.int32)
    C = g["capacity"][0]
    keep = O.capacity_keep(idx, 3, C)
    assert keep.astype(int).tolist() == g["keep"]
    counts, offsets, dst_row, src_token, _ = O.dispatch_maps(idx, 3, keep)
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert dst_row.tolist() == g["dst"]
    assert src_token[:offsets[-1]].tolist() == g["src_token"]
    assert O.expert_capacity(4, 2, 3, 1.5) == 4 and O.expert_capacity(4, 2, 3, 0.75) == 2


def test_capacity_formula():
    assert O.expert_capacity(4096, 8, 256, 1.25) == 160      # 1.25 * 128
    assert O.expert_capacity(8192, 2, 8, 1.0) == 2048
    assert O.expert_capacity(100, 1, 64, 0.1, min_capacity=4) == 4
    assert O.expert_capacity(1000, 2, 3, 1.0) == 666         # floor


@pytest.mark.parametrize("T,E,K,C", [(200, 8, 2, 30), (333, 16, 4, 50), (64, 4, 1, 5)])
def test_kept_slots_are_each_experts_first_in_token_order(T, E, K, C):
    rng = np.random.default_rng(T + C)
    idx = O.select_topk(rng.normal(size=(T, E)) + np.linspace(2, 0, E)[None, :], K)
    keep = O.capacity_keep(idx, E, C)
    for e in range(E):
        t_list, k_list = np.nonzero(idx == e)
        kept = keep[t_list, k_list]
        n = min(C, t_list.size)
        assert kept[:n].all() and not kept[n:].any()
    counts, offsets, dst_row, src_token, src_slot = O.dispatch_maps(idx, E, keep)
    full = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(counts, np.minimum(full, C))
    assert (dst_row[~keep] == -1).all()
    rows = dst_row[keep]
    np.testing.assert_array_equal(np.sort(rows), np.arange(counts.sum()))


def _problem(seed, T=40, h=8, E=6, K=2, F=6):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, h))
    w_r = rng.normal(size=(E, h)) * 0.8
    w_r[0] += 0.5  # a popular expert, so a small capacity drops slots
    w1 = rng.normal(size=(E, 2 * F, h)) / np.sqrt(h)
    w2 = rng.normal(size=(E, h, F)) / np.sqrt(F)
    dy = rng.normal(size=(T, h))
    return x, w_r, w1, w2, dy


@pytest.mark.parametrize("score", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID])
def test_large_capacity_is_dropless_and_masked_dense_agrees(score):
    x, w_r, w1, w2, _ = _problem(1)
    K = 2
    base = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU)
    big = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU, capacity=x.shape[0] * K)
    np.testing.assert_array_equal(big["y"], base["y"])
    for C in (3, 9, 15):
        perm = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU, capacity=C)
        assert (~perm["keep"]).any()
        dense = O.layer_fwd_masked_dense(x, w_r, w1, w2, K, score, O.ACT_SWIGLU, capacity=C)
        np.testing.assert_allclose(perm["y"], dense, rtol=1e-12, atol=1e-12)
        # a token whose every slot was dropped gets exactly zero output
        none_kept = ~perm["keep"].any(axis=1)
        assert (perm["y"][none_kept] == 0).all()


@pytest.mark.parametrize("score", [O.SCORE_SOFTMAX, O.SCORE_SIGMOID])
def test_capacity_backward_matches_central_differences(score):
    x, w_r, w1, w2, dy = _problem(2, T=24)
    K, C = 2, 6
    kw = dict(logits_dtype=np.float64, capacity=C)
    g = O.layer_bwd(x, w_r, w1, w2, dy, K, score, O.ACT_SWIGLU, **kw)
    y0 = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU, **kw)
    assert (~y0["keep"]).any()
    eps = 1e-6

    def loss():
        r = O.layer_fwd(x, w_r, w1, w2, K, score, O.ACT_SWIGLU, **kw)
        assert (r["idx"] == y0["idx"]).all() and (r["keep"] == y0["keep"]).all()
        return float((dy * r["y"]).sum())

    rng = np.random.default_rng(9)
    for arr, name in ((w_r, "dw_r"), (x, "dx"), (w1, "dw1"), (w2, "dw2")):
        flat = arr.reshape(-1)
        gflat = g[name].reshape(-1)
        for j in rng.choice(flat.size, size=10, replace=False):
            old = flat[j]
            flat[j] = old + eps
            lp = loss()
            flat[j] = old - eps
            lm = loss()
            flat[j] = old
            assert (lp - lm) / (2 * eps) == pytest.approx(gflat[j], rel=1e-5, abs=1e-8), name
