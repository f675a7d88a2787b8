"""GPU parity of the MXFP8 expert GEMMs (moe_mxfp8_quantize,
moe_expert_fc1_mxfp8, moe_expert_fc2_mxfp8) against the MXFP8 oracle.

* Quantisation: codes and E8M0 scales bit-exact (the decisions depend only on
  the bf16 inputs), over ragged groups, empty groups, rows outside every group,
  uniform groups, ties, subnormals, zero blocks and a wide dynamic range.
* GEMMs: the oracle's float64 product of the same dequantised operands; the
  GPU sums exact FP8 x FP8 products in fp32, so |gpu - oracle| <= K 2^-24
  sum_k |a_k b_k| plus the output's rounding (bf16: 2^-9 relative); through
  the SwiGLU epilogue the bound is carried by the derivative (|silu'| <= 1.1).
* The FC1 epilogue's own MXFP8 output of a: every element within the E4M3
  rounding of its block scale (or saturated) of the oracle's a, scales equal
  to the oracle's except where a block maximum lies within the accumulation
  bound of a power of two.
* Full DeepSeek-V3 sizes on sampled experts and rows, and bitwise reruns."""

import numpy as np
import pytest
import torch

from gpu_util import lib, needs_gpu, to_dev, to_np
from mixture_experts_layer_softmax_gb300 import inputs
from oracle import mxfp8_oracle as X

pytestmark = [pytest.mark.gpu, needs_gpu]

U = 2.0 ** -24  # fp32 unit roundoff


def scale_index(rows, K, offsets=None, urows=None, row_ids=None):
    """Byte index of each (row, 32-block) scale in the scale-atom layout that
    include/moe.h documents (rows 0..rows-1, or just row_ids); rows outside
    every group get -1."""
    KB = K // 128
    r = np.arange(rows) if row_ids is None else np.asarray(row_ids, np.int64)
    rows = len(r)
    if offsets is not None:
        offs = np.asarray(offsets, np.int64)
        inside = (r >= offs[0]) & (r < offs[-1])
        g = np.clip(np.searchsorted(offs, r, side="right") - 1, 0, len(offs) - 2)
        m = np.diff(offs)
        rt = np.concatenate([[0], np.cumsum((m + 127) // 128)])
        lr = r - offs[g]
        tile = rt[g] + lr // 128
    else:
        inside = np.ones(rows, bool)
        g = r // urows
        lr = r - g * urows
        tile = g * ((urows + 127) // 128) + lr // 128
    i = lr % 128
    base = (tile[:, None] * KB + np.arange(KB)[None, :]) * 512 + (16 * (i % 32) + 4 * (i // 32))[:, None]
    idx = (base[:, :, None] + np.arange(4)).reshape(rows, KB * 4)
    idx[~inside] = -1
    return idx


def gpu_scales(sf, idx):
    s = sf.cpu().numpy()
    out = np.zeros(idx.shape, np.uint8)
    ok = idx >= 0
    out[ok] = s[idx[ok]]
    return out


def quantize_dev(M, x, groups, offsets=None):
    rows, K = x.shape
    q = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(M.moe_mxfp8_scale_bytes(rows, K, groups), dtype=torch.uint8, device="cuda")
    od = None if offsets is None else torch.from_numpy(np.asarray(offsets, np.int32)).cuda()
    M.moe_mxfp8_quantize(rows, K, groups, od, to_dev(x, "bf16"), q, sf)
    return q, sf


def bf16(a):
    return to_np(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def hard_rows(rng, rows, K):
    """bf16 rows with a wide dynamic range, zero blocks, subnormal blocks and
    exact E4M3 ties after scaling."""
    x = rng.standard_normal((rows, K)) * np.exp2(rng.integers(-40, 40, (rows, 1)))
    if rows > 3 and K >= 64:
        x[1, :32] = 0.0
        x[2, 32:64] = rng.standard_normal(32) * 2.0 ** -130          # bf16 subnormals
        g = X.e4m3_decode(np.arange(0x7F))
        mids = (g[1:] + g[:-1]) / 2
        blk = np.concatenate([[448.0], rng.choice(mids, 31)]) * 2.0 ** 5
        x[3, :32] = blk * np.where(rng.random(32) < 0.5, -1, 1)
    return bf16(x)


@pytest.mark.parametrize("rows,K,offsets,groups", [
    (1000, 256, [0, 300, 300, 301, 900], 4),        # an empty and a one-row group, 100 rows outside
    (300, 7168, None, 3),                            # uniform groups of 100 rows
    (640, 2048, None, 5),                            # uniform groups of 128
    (777, 384, [0, 129, 256, 257, 777], 4),          # groups spanning 2 tiles, 1 row past a tile
    (1, 128, [0, 1], 1),
])
def test_quantize_bit_exact(rows, K, offsets, groups):
    M = lib()
    rng = np.random.default_rng(rows + K)
    x = hard_rows(rng, rows, K)
    q, sf = quantize_dev(M, x, groups, offsets)
    torch.cuda.synchronize()
    oq, os_ = X.quantize(x)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    idx = scale_index(rows, K, offsets, None if offsets is not None else rows // groups)
    ok = idx >= 0
    np.testing.assert_array_equal(gpu_scales(sf, idx)[ok], os_[ok])
    assert ok.any()


def _case(seed, T, K, E, h, F, skew=False, empty=()):
    rng = np.random.default_rng(seed)
    P = T * K
    w = np.ones(E)
    if skew:
        w = rng.dirichlet(np.full(E, 0.3))
    for e in empty:
        w[e] = 0.0
    counts = rng.multinomial(P, w / w.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    x = bf16(rng.standard_normal((P, h)))
    w1 = bf16(rng.standard_normal((E * 2 * F, h)) / np.sqrt(h))
    w2 = bf16(rng.standard_normal((E * h, F)) / np.sqrt(F))
    p = rng.uniform(0.05, 1.0, P).astype(np.float32)
    return dict(T=T, K=K, E=E, h=h, F=F, P=P, offsets=offsets, x=x, w1=w1, w2=w2, p=p)


def _cfg(M, c):
    return M.make_config(c["T"], c["h"], c["E"], c["K"], c["F"], M.MOE_BF16, M.MOE_SCORE_SOFTMAX,
                         M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM)


def _fc1_bounds(aq, as_, offsets, bq, bs, Nb, Kd, p):
    """Oracle a and its elementwise bound for the GPU's fp32 value of a."""
    H = X.grouped_gemm(aq, as_, offsets, bq, bs, Nb)
    S = X.grouped_gemm(aq & 0x7F, as_, offsets, bq & 0x7F, bs, Nb)   # sum |a_k b_k|
    tH = Kd * U * S
    F = Nb // 2
    g, u, tg, tu = H[:, :F], H[:, F:], tH[:, :F], tH[:, F:]
    a = X.fc1_swiglu(H, p.astype(np.float64))
    pp = p.astype(np.float64)[:, None]
    d = pp * (1.1 * tg * (np.abs(u) + tu) + (np.abs(X.silu(g)) + 1.1 * tg) * tu)
    d32 = d + 2.0 ** -18 * np.abs(a) + 1e-30     # fp32 evaluation of p silu(g) up
    return a, d32


def _check_aq(a_ref, d32, codes, scales):
    """The FC1 epilogue's MXFP8 a against the oracle's a."""
    deq = X.dequantize(codes, scales)
    Xe = np.repeat(scales.astype(np.int64) - 127, 32, axis=1).astype(np.float64)
    sc = np.exp2(Xe)
    amag = np.abs(a_ref) + d32
    sat = np.maximum(amag - 448.0 * sc, 0.0)
    tol = d32 + np.maximum(2.0 ** -4 * amag, 2.0 ** -10 * sc) + sat
    err = np.abs(deq - a_ref)
    assert np.all(err <= tol), float((err / tol).max())
    # scales: the oracle's rule on the block maxima, up to the bound
    R, F = a_ref.shape
    amax = np.abs(a_ref).reshape(R, F // 32, 32).max(axis=2)
    dmax = d32.reshape(R, F // 32, 32).max(axis=2)
    lo = X.shared_exponent(np.maximum(amax - dmax, 0.0)) + 127
    hi = X.shared_exponent(amax + dmax) + 127
    assert np.all((scales >= lo) & (scales <= hi))
    # the check is not vacuous: most blocks admit one scale only (the bound is
    # the worst case K 2^-24 sum |a b|, loose at K = 7168)
    assert np.mean(lo == hi) > 0.8


CASES = [
    dict(seed=1, T=300, K=2, E=8, h=256, F=128),
    dict(seed=2, T=500, K=4, E=16, h=384, F=256, skew=True, empty=(3, 7)),
    dict(seed=3, T=100, K=8, E=64, h=512, F=128, skew=True),     # many experts below one tile
    dict(seed=4, T=2048, K=1, E=2, h=1024, F=384),               # multi-tile experts
    dict(seed=6, T=1024, K=2, E=4, h=2048, F=512),               # ~4 tiles per expert, long K
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"T{c['T']}_E{c['E']}_h{c['h']}_F{c['F']}")
def test_fc1_fc2_mxfp8_match_oracle(c):
    M = lib()
    c = _case(**c)
    P, E, h, F, offs = c["P"], c["E"], c["h"], c["F"], c["offsets"]
    cfg = _cfg(M, c)
    od = torch.from_numpy(offs.astype(np.int32)).cuda()
    xq, xsf = quantize_dev(M, c["x"], E, offs)
    w1q, w1sf = quantize_dev(M, c["w1"], E)
    w2q, w2sf = quantize_dev(M, c["w2"], E)
    a = torch.full((P, F), float("nan"), dtype=torch.bfloat16, device="cuda")
    aq = torch.empty(P, F, dtype=torch.uint8, device="cuda")
    asf = torch.zeros(M.moe_mxfp8_scale_bytes(P, F, E), dtype=torch.uint8, device="cuda")
    pd = torch.from_numpy(c["p"]).cuda()
    M.moe_expert_fc1_mxfp8(cfg, xq, xsf, od, pd, w1q, w1sf, a, aq, asf)
    y = torch.full((P, h), float("nan"), dtype=torch.bfloat16, device="cuda")
    M.moe_expert_fc2_mxfp8(cfg, aq, asf, od, w2q, w2sf, y)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    # operands: bit-exact against the oracle quantiser
    oxq, oxs = X.quantize(c["x"])
    ow1q, ow1s = X.quantize(c["w1"])
    np.testing.assert_array_equal(xq.cpu().numpy(), oxq)
    np.testing.assert_array_equal(w1q.cpu().numpy(), ow1q)
    # FC1: bf16 a and the MXFP8 a
    a_ref, d32 = _fc1_bounds(oxq, oxs, offs, ow1q, ow1s, 2 * F, h, c["p"])
    ag = to_np(a).astype(np.float64)
    tol_a = d32 + 2.0 ** -8 * (np.abs(a_ref) + d32)
    assert np.all(np.abs(ag - a_ref) <= tol_a), float((np.abs(ag - a_ref) / tol_a).max())
    a_codes = aq.cpu().numpy()
    a_scales = gpu_scales(asf, scale_index(P, F, offs))
    _check_aq(a_ref, d32, a_codes, a_scales)
    # FC2 on the GPU's own MXFP8 a
    ow2q, ow2s = X.quantize(c["w2"])
    y_ref = X.grouped_gemm(a_codes, a_scales, offs, ow2q, ow2s, h)
    S = X.grouped_gemm(a_codes & 0x7F, a_scales, offs, ow2q & 0x7F, ow2s, h)
    tol_y = F * U * S + 2.0 ** -8 * np.abs(y_ref) + 1e-30
    yg = to_np(y).astype(np.float64)
    assert np.all(np.abs(yg - y_ref) <= tol_y), float((np.abs(yg - y_ref) / tol_y).max())
    # end to end against the oracle's MXFP8 MLP (which quantises a in float64)
    y_mlp = X.expert_mlp_fwd(c["x"], offs, c["p"], c["w1"].reshape(E, 2 * F, h),
                             c["w2"].reshape(E, h, F))
    assert np.abs(yg - y_mlp).max() <= 1e-2 * np.abs(y_mlp).max()


def test_fc1_bf16_output_only_and_reruns_bitwise():
    M = lib()
    c = _case(seed=5, T=400, K=2, E=8, h=256, F=256, skew=True)
    P, E, h, F, offs = c["P"], c["E"], c["h"], c["F"], c["offsets"]
    cfg = _cfg(M, c)
    od = torch.from_numpy(offs.astype(np.int32)).cuda()
    xq, xsf = quantize_dev(M, c["x"], E, offs)
    w1q, w1sf = quantize_dev(M, c["w1"], E)
    outs = []
    for with_q in (False, True, True):
        a = torch.empty(P, F, dtype=torch.bfloat16, device="cuda")
        aq = torch.empty(P, F, dtype=torch.uint8, device="cuda") if with_q else None
        asf = torch.zeros(M.moe_mxfp8_scale_bytes(P, F, E), dtype=torch.uint8,
                          device="cuda") if with_q else None
        M.moe_expert_fc1_mxfp8(cfg, xq, xsf, od, None, w1q, w1sf, a, aq, asf)
        torch.cuda.synchronize()
        outs.append((a.clone(), None if aq is None else aq.clone(), None if asf is None else asf.clone()))
    assert M.moe_get_error() == M.MOE_OK
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[1][0], outs[2][0])
    assert torch.equal(outs[1][1], outs[2][1]) and torch.equal(outs[1][2], outs[2][2])
    # perm_prob NULL: weight 1
    oxq, oxs = X.quantize(c["x"])
    ow1q, ow1s = X.quantize(c["w1"])
    a_ref, d32 = _fc1_bounds(oxq, oxs, offs, ow1q, ow1s, 2 * F, h, np.ones(P, np.float32))
    ag = to_np(outs[0][0]).astype(np.float64)
    assert np.all(np.abs(ag - a_ref) <= d32 + 2.0 ** -8 * (np.abs(a_ref) + d32))


def test_full_size_deepseek_v3_sampled():
    """DeepSeek-V3 expert shapes (P = 4096 x 8 rows, h 7168, F 2048, 256
    experts with a skewed load): weights and activations quantised on the
    GPU, both GEMMs at full size; the oracle checks three experts' weights
    bit-exactly and a sample of their rows through FC1 and FC2."""
    M = lib()
    T, K, E, h, F = 4096, 8, 256, 7168, 2048
    P = T * K
    rng = np.random.default_rng(11)
    counts = rng.multinomial(P, rng.dirichlet(np.full(E, 0.5)))
    counts[17] = 0
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    seed = 97
    dev = torch.device("cuda")
    x = torch.empty(P, h, dtype=torch.bfloat16, device=dev)
    M.synth_normal(x, seed, inputs.TAG["x"], 1.0)
    w1 = torch.empty(E * 2 * F, h, dtype=torch.bfloat16, device=dev)
    M.synth_normal(w1, seed, inputs.TAG["w1"], h ** -0.5)
    w2 = torch.empty(E * h, F, dtype=torch.bfloat16, device=dev)
    M.synth_normal(w2, seed, inputs.TAG["w2"], F ** -0.5)
    cfg = M.make_config(T, h, E, K, F, M.MOE_BF16, M.MOE_SCORE_SIGMOID, M.MOE_ACT_SWIGLU, 0, 0,
                        M.MOE_FLAG_RENORM)
    od = torch.from_numpy(offs.astype(np.int32)).cuda()
    u8 = dict(dtype=torch.uint8, device=dev)
    xq, xsf = torch.empty(P, h, **u8), torch.zeros(M.moe_mxfp8_scale_bytes(P, h, E), **u8)
    w1q, w1sf = torch.empty(E * 2 * F, h, **u8), torch.zeros(M.moe_mxfp8_scale_bytes(E * 2 * F, h, E), **u8)
    w2q, w2sf = torch.empty(E * h, F, **u8), torch.zeros(M.moe_mxfp8_scale_bytes(E * h, F, E), **u8)
    M.moe_mxfp8_quantize(P, h, E, od, x, xq, xsf)
    M.moe_mxfp8_quantize(E * 2 * F, h, E, None, w1, w1q, w1sf)
    M.moe_mxfp8_quantize(E * h, F, E, None, w2, w2q, w2sf)
    p = torch.rand(P, device=dev) * 0.9 + 0.1
    aq, asf = torch.empty(P, F, **u8), torch.zeros(M.moe_mxfp8_scale_bytes(P, F, E), **u8)
    a = torch.empty(P, F, dtype=torch.bfloat16, device=dev)
    y = torch.empty(P, h, dtype=torch.bfloat16, device=dev)
    M.moe_expert_fc1_mxfp8(cfg, xq, xsf, od, p, w1q, w1sf, a, aq, asf)
    M.moe_expert_fc2_mxfp8(cfg, aq, asf, od, w2q, w2sf, y)
    torch.cuda.synchronize()
    assert M.moe_get_error() == M.MOE_OK
    big = int(np.argmax(counts))
    for e in (big, int(np.argsort(counts)[E // 2]), 255):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        w1e = inputs.normal((2 * F, h), h ** -0.5, seed, inputs.TAG["w1"], "bf16", start=e * 2 * F * h)
        w2e = inputs.normal((h, F), F ** -0.5, seed, inputs.TAG["w2"], "bf16", start=e * h * F)
        ow1q, ow1s = X.quantize(w1e)
        ow2q, ow2s = X.quantize(w2e)
        np.testing.assert_array_equal(w1q[e * 2 * F:(e + 1) * 2 * F].cpu().numpy(), ow1q)
        w1_rows = np.arange(e * 2 * F, (e + 1) * 2 * F)
        np.testing.assert_array_equal(gpu_scales(w1sf, scale_index(0, h, None, 2 * F, w1_rows)), ow1s)
        np.testing.assert_array_equal(w2q[e * h:(e + 1) * h].cpu().numpy(), ow2q)
        w2_rows = np.arange(e * h, (e + 1) * h)
        np.testing.assert_array_equal(gpu_scales(w2sf, scale_index(0, F, None, h, w2_rows)), ow2s)
        rows = np.unique(np.concatenate([[r0, r1 - 1], rng.integers(r0, r1, 6)]))
        xr = inputs.rows((P, h), rows, 1.0, seed, inputs.TAG["x"], "bf16")
        oxq, oxs = X.quantize(xr)
        np.testing.assert_array_equal(xq[rows].cpu().numpy(), oxq)
        np.testing.assert_array_equal(gpu_scales(xsf, scale_index(0, h, offs, None, rows)), oxs)
        one = np.array([0, len(rows)])
        pr = p[rows].cpu().numpy()
        a_ref, d32 = _fc1_bounds(oxq, oxs, one, ow1q, ow1s, 2 * F, h, pr)
        ag = to_np(a[rows]).astype(np.float64)
        tol_a = d32 + 2.0 ** -8 * (np.abs(a_ref) + d32)
        assert np.all(np.abs(ag - a_ref) <= tol_a)
        a_codes = aq[rows].cpu().numpy()
        a_scales = gpu_scales(asf, scale_index(0, F, offs, None, rows))
        _check_aq(a_ref, d32, a_codes, a_scales)
        y_ref = X.grouped_gemm(a_codes, a_scales, one, ow2q, ow2s, h)
        S = X.grouped_gemm(a_codes & 0x7F, a_scales, one, ow2q & 0x7F, ow2s, h)
        yg = to_np(y[rows]).astype(np.float64)
        assert np.all(np.abs(yg - y_ref) <= F * U * S + 2.0 ** -8 * np.abs(y_ref) + 1e-30)


@pytest.mark.parametrize("T,E,K,h,cap", [
    (1000, 8, 2, 256, 0), (333, 64, 8, 384, 0), (2048, 256, 8, 7168, 0), (700, 16, 4, 128, 150),
    (0, 8, 2, 256, 0),
])
def test_permute_mxfp8_equals_permute_then_quantize(T, E, K, h, cap):
    M = lib()
    rng = np.random.default_rng(T + E + h)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, 0] += 1.0
    from oracle import moe_oracle as O
    idx, prob = O.route(logits, K, O.SCORE_SOFTMAX) if T else (np.zeros((0, K), np.int32),
                                                                np.zeros((0, K), np.float32))
    x = hard_rows(rng, T, h) if T else np.zeros((0, h), np.float32)
    cfg = M.make_config(T, h, E, K, 128, M.MOE_BF16, 0, M.MOE_ACT_SWIGLU, 0, 0, M.MOE_FLAG_RENORM,
                        capacity=cap)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    P = T * K
    i32 = dict(dtype=torch.int32, device="cuda")
    xd = to_dev(x, "bf16")
    idd = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).cuda()
    pdd = to_dev(prob, "f32")
    sfb = M.moe_mxfp8_scale_bytes(P, h, E)
    outs = {}
    for fused in ((True,) if T == 0 else (True, False)):
        counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
        dst_row, src_token = torch.empty(T, K, **i32), torch.empty(max(P, 1), **i32)
        perm_prob = torch.empty(max(P, 1), dtype=torch.float32, device="cuda")
        q = torch.zeros(max(P, 1), h, dtype=torch.uint8, device="cuda")
        sf = torch.zeros(max(sfb, 16), dtype=torch.uint8, device="cuda")
        if fused:
            M.moe_permute_mxfp8(cfg, xd, idd, pdd, q, sf, counts, offsets, dst_row, src_token,
                                perm_prob, ws)
        else:
            x_perm = torch.zeros(max(P, 1), h, dtype=torch.bfloat16, device="cuda")
            M.moe_permute(cfg, xd, idd, pdd, x_perm, counts, offsets, dst_row, src_token,
                          perm_prob, ws)
            M.moe_mxfp8_quantize(P, h, E, offsets, x_perm, q, sf)
        torch.cuda.synchronize()
        assert M.moe_get_error() == M.MOE_OK
        outs[fused] = dict(q=q.cpu().numpy(), sf=sf, offsets=to_np(offsets),
                           src=src_token.cpu().numpy(), dst=dst_row.cpu().numpy())
    f = outs[True]
    if T == 0:  # no rows: the maps are empty, nothing is written
        assert not f["offsets"].any()
        return
    u = outs[False]
    np.testing.assert_array_equal(f["offsets"], u["offsets"])
    np.testing.assert_array_equal(f["dst"], u["dst"])
    n = int(f["offsets"][-1])
    if n == 0:
        return
    np.testing.assert_array_equal(f["q"][:n], u["q"][:n])
    idx_s = scale_index(n, h, f["offsets"])
    np.testing.assert_array_equal(gpu_scales(f["sf"], idx_s), gpu_scales(u["sf"], idx_s))
    # and against the oracle: row r holds token src_token[r] quantised
    oq, os_ = X.quantize(x[f["src"][:n]])
    np.testing.assert_array_equal(f["q"][:n], oq)
    np.testing.assert_array_equal(gpu_scales(f["sf"], idx_s), os_)
    if cap:
        assert (f["dst"] == -1).any()
