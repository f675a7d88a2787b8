"""Pins for the MXFP8 oracle (oracle/mxfp8_oracle.py): the E4M3 code table
against the format's fixed points, rounding against PyTorch's independent
float8_e4m3fn conversion, saturation, the shared-exponent rule on closed
forms, a hand-worked block (tests/golden/mxfp8_block.txt), the quantisation
error bounds, exact round trips of grid values, and the grouped GEMM against
brute force and a closed form.  Each pin is chosen so that a plausible slip
(an exponent bias off by one, ties away from zero, a scale applied with the
wrong sign, a transposed operand, a wrong expert's weights) fails."""

import os

import numpy as np
import pytest
import torch

from oracle import mxfp8_oracle as X

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_block.txt")


def test_code_table_fixed_points():
    d = X.e4m3_decode
    assert d(0x7E) == 448.0                    # largest finite
    assert d(0x08) == 2.0 ** -6                # smallest normal
    assert d(0x01) == 2.0 ** -9                # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9            # largest subnormal
    assert d(0x38) == 1.0                      # exponent field 7 = bias
    assert d(0x3C) == 1.5
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x80) == 0.0 and np.signbit(d(0x80))
    assert d(0xFE) == -448.0
    g = d(np.arange(0x7F))
    assert np.all(np.diff(g) > 0)              # codes 0..126 increase strictly
    assert len(np.unique(np.abs(d(np.arange(256))[~np.isnan(d(np.arange(256)))]))) == 127


def test_code_table_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = X.e4m3_decode(codes)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_rounding_matches_torch_float8_within_range():
    rng = np.random.default_rng(0)
    g = X.e4m3_decode(np.arange(0x7F))
    mids = (g[1:] + g[:-1]) / 2                # every tie
    v = np.concatenate([g, mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20),
                        rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-14, 8.8, 20000))])
    v = v[v <= 448.0]
    v = np.concatenate([v, -v])
    v32 = v.astype(np.float32)                 # the grid, ties and their neighbours are
    v = v32.astype(np.float64)                 # fp32-exact; the random values are taken as rounded
    ref = torch.from_numpy(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(X.e4m3_encode(v), ref)


def test_saturation():
    np.testing.assert_array_equal(X.e4m3_round([448.0, 449.0, 463.9, 464.0, 511.99, 1e6]),
                                  [448.0] * 6)
    np.testing.assert_array_equal(X.e4m3_round([-500.0]), [-448.0])


def test_shared_exponent_closed_forms():
    se = X.shared_exponent
    assert se(448.0) == 0                      # 448 -> scale 1
    assert se(1.0) == -8                       # 1 * 2^8 = 256
    assert se(0.75) == -9                      # 0.75 * 2^9 = 384
    assert se(3.0) == -7
    assert se(2.0 ** 100) == 92
    assert se(0.0) == -127
    assert se(2.0 ** -130) == -127             # clamped to the E8M0 range
    assert se(np.nextafter(2.0, 0)) == -8      # just below 2: floor(log2) = 0
    assert se(2.0) == -7


def test_hand_worked_block():
    xs, codes, scale = [], [], None
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        f = line.split()
        if f[0] == "scale":
            scale = int(f[1])
        else:
            xs.append(float(f[1]))
            codes.append(int(f[2], 16))
    x = np.zeros((1, 32))
    x[0, :len(xs)] = xs
    q, s = X.quantize(x)
    assert s.tolist() == [[scale]]
    assert q[0, :len(xs)].tolist() == codes
    assert np.all(q[0, len(xs):] == 0)
    assert X.dequantize(q, s)[0, 2] == 6.5 / 64


def test_quantisation_error_bounds():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    x[3, 32:64] = 0.0                          # an all-zero block
    q, s = X.quantize(x)
    back = X.dequantize(q, s)
    Xe = s.astype(np.int64) - 127
    scale = np.repeat(np.exp2(Xe.astype(np.float64)), 32, axis=1)
    a = np.abs(x)
    normal = a >= scale * 2.0 ** -6
    sat = a > scale * 448.0
    # half an E4M3 ulp: 2^-4 relative for normals (3 mantissa bits),
    # 2^-10 x scale absolute in the subnormal range; magnitudes above 448 x
    # scale (at most 512 x scale by the exponent rule) saturate to 448 x scale
    assert np.all(np.abs(back - x)[normal & ~sat] <= 2.0 ** -4 * a[normal & ~sat])
    assert np.all(np.abs(back - x)[~normal] <= 2.0 ** -10 * scale[~normal])
    assert sat.any()
    np.testing.assert_array_equal(np.abs(back)[sat], 448.0 * scale[sat])
    # the block maximum lands in [256, 448] after scaling
    amax = a.reshape(64, 8, 32).max(axis=2)
    r = amax / np.exp2(Xe.astype(np.float64))
    assert np.all((r[amax > 0] >= 256) & (r[amax > 0] < 512))
    assert s[3, 1] == 0 and np.all(q[3, 32:64] == 0)


def test_grid_values_round_trip_exactly():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 0x7F, (8, 64)).astype(np.uint8) | (rng.integers(0, 2, (8, 64)) << 7).astype(np.uint8)
    codes[:, 0] = 0x7E                          # every block holds 448, so X = 0 ...
    codes[:, 32] = 0x7E
    Xs = rng.integers(-30, 30, (8, 2))
    x = X.e4m3_decode(codes) * np.repeat(np.exp2(Xs.astype(np.float64)), 32, axis=1)
    q, s = X.quantize(x)                        # ... relative to its own scale 2^Xs
    np.testing.assert_array_equal(s.astype(np.int64) - 127, Xs)
    np.testing.assert_array_equal(X.dequantize(q, s), x)


def test_grouped_gemm_brute_force():
    rng = np.random.default_rng(3)
    E, Nb, K = 3, 4, 64
    offsets = np.array([0, 2, 2, 5])            # expert 1 empty
    a = rng.standard_normal((5, K))
    b = rng.standard_normal((E * Nb, K)) * 3
    aq, as_ = X.quantize(a)
    bq, bs = X.quantize(b)
    out = X.grouped_gemm(aq, as_, offsets, bq, bs, Nb)
    A, B = X.dequantize(aq, as_), X.dequantize(bq, bs)
    for r in range(5):
        e = int(np.searchsorted(offsets, r, side="right") - 1)
        for n in range(Nb):
            s = 0.0
            for k in range(K):
                s += X.e4m3_decode(aq[r, k]) * 2.0 ** (int(as_[r, k // 32]) - 127) * \
                     X.e4m3_decode(bq[e * Nb + n, k]) * 2.0 ** (int(bs[e * Nb + n, k // 32]) - 127)
            assert out[r, n] == pytest.approx(s, rel=1e-12, abs=1e-300)
            assert out[r, n] == pytest.approx(A[r] @ B[e * Nb + n], rel=1e-12)


def test_grouped_gemm_scales_closed_form():
    # every element code 1.0: out = 32 * sum over blocks of 2^(Xa + Xb)
    R, Nb, K = 2, 2, 96
    aq = np.full((R, K), 0x38, np.uint8)
    bq = np.full((Nb, K), 0x38, np.uint8)
    as_ = np.array([[120, 127, 130], [127, 127, 127]], np.uint8)
    bs = np.array([[127, 127, 127], [100, 110, 127]], np.uint8)
    out = X.grouped_gemm(aq, as_, [0, R], bq, bs, Nb)
    for r in range(R):
        for n in range(Nb):
            want = 32 * sum(2.0 ** (int(as_[r, j]) - 127 + int(bs[n, j]) - 127) for j in range(3))
            assert out[r, n] == want


def test_expert_mlp_matches_exact_math_within_fp8_error():
    # the MXFP8 MLP against the exact float64 MLP: within the error that
    # 1 x 32 E4M3 quantisation of all four operands allows
    rng = np.random.default_rng(4)
    E, h, F, P = 2, 64, 32, 40
    offsets = np.array([0, 25, 40])
    x = rng.standard_normal((P, h))
    w1 = rng.standard_normal((E, 2 * F, h)) / np.sqrt(h)
    w2 = rng.standard_normal((E, h, F)) / np.sqrt(F)
    p = rng.uniform(0.2, 1.0, P)
    y = X.expert_mlp_fwd(x, offsets, p, w1, w2)
    ref = np.zeros((P, h))
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        H = x[r0:r1] @ w1[e].T
        a = p[r0:r1, None] * X.silu(H[:, :F]) * H[:, F:]
        ref[r0:r1] = a @ w2[e].T
    err = np.abs(y - ref).max() / np.abs(ref).max()
    assert err < 0.08, err
    assert err > 1e-4                           # quantisation really happened
