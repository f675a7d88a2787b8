"""Plain CPU oracle for the MXFP8 expert GEMMs (microscaled FP8 operands).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
call it.  It shares no code with the CUDA path and computes in float64 with
numpy primitives.

Sources:

* "Scalable Training of Mixture-of-Experts Models with Megatron Core" (review
  page), §5.3.3 "MXFP8 (Blackwell)": activations and weights are both
  quantised in 1 x 32 blocks, each block with an E8M0 scale factor; §5.4
  "Dynamic shape alignment": MXFP8 GEMMs want their dimensions aligned to 32.
* The element format and the scale rule are not spelled out on the pages;
  they are read from the published OCP Microscaling (MX) v1.0 format
  definition, which MXFP8 names:
  - element: FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    subnormals, no infinities, S.1111.111 is NaN; largest finite 448);
  - scale: E8M0, an unsigned biased exponent (code c means 2^(c - 127),
    c = 255 is NaN);
  - shared exponent of a block: X = floor(log2(max |x|)) - emax_elem with
    emax_elem = 8 for E4M3, clamped to the E8M0 range; an all-zero block
    takes the smallest scale;
  - element code: x / 2^X rounded to nearest, ties to even, values beyond the
    largest finite magnitude saturated to +-448.

Readings where the pages leave a step open:

* Blocks run along the reduction (K) dimension of each GEMM operand: along h
  for x_perm and W1, along F for a and W2.  K is a multiple of 32.
* Saturation rather than overflow to NaN ("satfinite"); the scale rule keeps
  |x| / 2^X below 512, so only magnitudes in [448, 512) saturate.
* Inputs are finite.
* In the MXFP8 expert MLP the FC1 output a = p * silu(gate) * up is
  quantised again (1 x 32 blocks along F) as FC2's left operand; the oracle
  quantises the float64 a, with no intermediate rounding.

Pins live in tests/test_oracle_mxfp8.py.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8          # 448 = 1.75 * 2^8
E8M0_BIAS = 127
BLOCK = 32             # elements sharing one scale


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8) as float64; S.1111.111 decodes to NaN."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the 127 finite non-negative magnitudes, indexed by their code 0x00 .. 0x7E
# (value increases with the code)
_GRID = e4m3_decode(np.arange(0x7F))


def e4m3_encode(v) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest magnitude on the grid, a
    tie going to the even code (the one whose mantissa ends in 0), magnitudes
    above 448 saturated to 448; the sign bit is the input's (so -0.0 and tiny
    negatives give 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("inputs are finite")
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.clip(np.searchsorted(_GRID, a, side="left"), 0, 0x7E)  # first grid value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _GRID[lo]
    d_hi = _GRID[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a == _GRID[hi], hi, mag)  # exact grid values
    return (mag | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def e4m3_round(v) -> np.ndarray:
    """v rounded to E4M3 (round to nearest even, saturating), as float64."""
    return e4m3_decode(e4m3_encode(v))


def shared_exponent(amax) -> np.ndarray:
    """X = floor(log2 amax) - 8, clamped to [-127, 127]; amax == 0 gives -127.
    floor(log2) is taken exactly from the binary exponent (frexp)."""
    amax = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(amax)                # amax = m 2^e, m in [0.5, 1)
    x = (e.astype(np.int64) - 1) - E4M3_EMAX
    x = np.where(amax == 0.0, -E8M0_BIAS, x)
    return np.clip(x, -E8M0_BIAS, E8M0_BIAS)


def quantize(x, block: int = BLOCK):
    """MXFP8 quantisation of the rows of x [R, K] in 1 x block blocks along K.
    Returns (codes [R, K] uint8, scale codes [R, K / block] uint8 = X + 127)."""
    x = np.asarray(x, dtype=np.float64)
    R, K = x.shape
    if K % block:
        raise ValueError("K must be a multiple of the block size")
    xb = x.reshape(R, K // block, block)
    X = shared_exponent(np.abs(xb).max(axis=2))                    # [R, K/block]
    scaled = np.ldexp(xb, -X[:, :, None])                          # exact: a power of 2
    codes = e4m3_encode(scaled).reshape(R, K)
    return codes, (X + E8M0_BIAS).astype(np.uint8)


def dequantize(codes, scales, block: int = BLOCK) -> np.ndarray:
    """Float64 values of MXFP8 data: code value x 2^(scale code - 127)."""
    codes = np.asarray(codes)
    R, K = codes.shape
    v = e4m3_decode(codes).reshape(R, K // block, block)
    X = np.asarray(scales, dtype=np.int64) - E8M0_BIAS
    return np.ldexp(v, X[:, :, None]).reshape(R, K)


def grouped_gemm(a_codes, a_scales, offsets, b_codes, b_scales, Nb: int) -> np.ndarray:
    """out[r, n] = sum_k A[r, k] B_e[n, k] over the dequantised operands, for
    the rows r of each expert e (offsets[e] .. offsets[e+1]); B is [E * Nb, K]."""
    A = dequantize(a_codes, a_scales)
    B = dequantize(b_codes, b_scales)
    offsets = np.asarray(offsets)
    out = np.zeros((A.shape[0], Nb))
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            out[r0:r1] = A[r0:r1] @ B[e * Nb:(e + 1) * Nb].T
    return out


def silu(z):
    return z / (1.0 + np.exp(-z))


def fc1_swiglu(h, prob):
    """The FC1 epilogue of a bias-free SwiGLU expert: a = p * silu(gate) * up,
    the gate in the first F columns of h [R, 2F]."""
    F = h.shape[1] // 2
    p = np.ones(h.shape[0]) if prob is None else np.asarray(prob, dtype=np.float64)
    return p[:, None] * silu(h[:, :F]) * h[:, F:]


def expert_mlp_fwd(x_perm, offsets, prob, w1, w2):
    """MXFP8 expert MLP on permuted rows: quantise x_perm and W1 along h,
    FC1 + SwiGLU with the routing weight p, quantise a and W2 along F, FC2.
    w1 [E, 2F, h], w2 [E, h, F]; returns y_perm [P, h] (float64)."""
    E, F2, h = w1.shape
    xq, xs = quantize(x_perm)
    w1q, w1s = quantize(np.asarray(w1, dtype=np.float64).reshape(E * F2, h))
    H = grouped_gemm(xq, xs, offsets, w1q, w1s, F2)
    a = fc1_swiglu(H, prob)
    aq, as_ = quantize(a)
    w2q, w2s = quantize(np.asarray(w2, dtype=np.float64).reshape(E * h, F2 // 2))
    return grouped_gemm(aq, as_, offsets, w2q, w2s, h)
