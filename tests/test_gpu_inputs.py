"""The device-side input generator (used to fill full-size benchmark tensors)
reproduces the host generator of inputs.py bit for bit, on slices taken far
into the stream."""

import numpy as np
import pytest
import torch

from gpu_util import lib, needs_gpu
from mixture_experts_layer_softmax_gb300 import inputs

pytestmark = [pytest.mark.gpu, needs_gpu]


@pytest.mark.parametrize("dtype,std,start", [("bf16", 1.0, 0), ("bf16", 0.0156, 123_456_789_001),
                                              ("f32", 0.02, 7), ("f32", 1.0, 4_000_000_000)])
def test_device_generator_matches_host(dtype, std, start):
    M = lib()
    n = 1 << 21
    t = torch.empty(n, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    M.synth_normal(t, 4, 5, std, start=start)
    host = inputs.normal((n,), std, 4, 5, dtype, start=start)
    got = t.float().cpu().numpy()
    mism = int((got != host).sum())
    assert mism == 0, f"{mism} of {n} elements differ"
