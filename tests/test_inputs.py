"""The seeded input generator against its published definitions."""

import numpy as np
import torch

from mixture_experts_layer_softmax_gb300 import inputs, workloads


def test_splitmix64_published_sequence():
    # SplitMix64 from state 0: the first three outputs as published.
    key = 0
    outs = [inputs.mix64_int(key + (i + 1) * inputs.GAMMA) for i in range(3)]
    assert outs == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_vectorised_matches_scalar():
    seed, tag = 7, 3
    key = inputs.stream_key(seed, tag)
    v = inputs.raw_u64(seed, tag, 100, 5)
    for j in range(5):
        assert int(v[j]) == inputs.mix64_int(key + (100 + j + 1) * inputs.GAMMA)


def test_normal_moments_and_slices():
    a = inputs.normal((1 << 20,), 1.0, 0, 1)
    assert abs(a.mean()) < 5e-3 and abs(a.std() - 1) < 5e-3
    b = inputs.normal((1000,), 1.0, 0, 1, start=5000)
    np.testing.assert_array_equal(a[5000:6000], b)


def test_bf16_rounding_matches_torch():
    a = inputs.normal((100000,), 3.0, 1, 2)
    ours = inputs.bf16_bits_to_f32(inputs.f32_to_bf16_bits(a))
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(ours, ref)


def test_rows_helper():
    full = inputs.normal((6, 4, 3), 0.5, 2, 5, "bf16")
    r = inputs.rows((6, 4, 3), [4, 1], 0.5, 2, 5, "bf16")
    np.testing.assert_array_equal(r, full[[4, 1]])


def test_zipf_gate_bias_recipe():
    w = workloads.QWEN3
    b = w.gate_bias()
    r = inputs.random_ranks(w.E, w.seed)
    assert sorted(r.tolist()) == list(range(1, w.E + 1))
    assert b.max() == np.float32(2.0)
    np.testing.assert_allclose(b, 2.0 * r.astype(np.float64) ** -1.1, rtol=1e-7)
