"""Synthetic MoE-layer workloads shaped like the layers the pages train
(Mixtral-8x7B, Qwen3-235B-A22B, DeepSeek-V3) plus a tiny fp32 case and a
fine-grained sweep.  A workload is a shape, a recipe for its seeded inputs,
and the layer options; nothing here computes any part of the layer.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import inputs

SOFTMAX, SIGMOID = 0, 1
GELU, SWIGLU = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    K: int
    F: int
    dtype: str = "bf16"          # "f32" or "bf16": activations and expert weights
    score: int = SOFTMAX
    act: int = SWIGLU
    has_bias: bool = False       # b1/b2 on the experts (GELU tiny case)
    n_shared: int = 0
    renorm: bool = True
    force_balance: bool = False
    router_std: float | None = 0.02   # None: 1/sqrt(h)
    zipf_s: float = 0.0          # >0: gate bias 2.0 * rank^-s on a seeded ranking
    zipf_scale: float = 2.0
    sel_bias_std: float = 0.0    # >0: selection-only bias ~ N(0, std^2)
    backward: bool = False
    seed: int = 0

    @property
    def P(self) -> int:
        return self.T * self.K

    @property
    def w1_rows(self) -> int:
        return 2 * self.F if self.act == SWIGLU else self.F

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ---- input recipe -------------------------------------------------
    def std(self, role: str) -> float:
        if role == "x" or role == "dy":
            return 1.0
        if role == "w_r":
            return self.router_std if self.router_std is not None else 1.0 / math.sqrt(self.h)
        if role in ("w1", "b1", "w1_shared"):
            return 1.0 / math.sqrt(self.h)
        if role in ("w2", "b2", "w2_shared"):
            return 1.0 / math.sqrt(self.F)
        if role == "sel_bias":
            return self.sel_bias_std
        raise KeyError(role)

    def shape(self, role: str):
        T, h, E, F = self.T, self.h, self.E, self.F
        return dict(x=(T, h), dy=(T, h), w_r=(E, h), w1=(E, self.w1_rows, h), b1=(E, self.w1_rows),
                    w2=(E, h, F), b2=(E, h), w1_shared=(self.w1_rows, h), w2_shared=(h, F),
                    sel_bias=(E,), gate_bias=(E,))[role]

    def tensor_dtype(self, role: str) -> str:
        # the router weight, the biases of the router are fp32 (kept in FP32)
        if role in ("w_r", "gate_bias", "sel_bias"):
            return "f32"
        return self.dtype

    def roles(self):
        r = ["x", "w_r", "w1", "w2"]
        if self.has_bias:
            r += ["b1", "b2"]
        if self.n_shared:
            r += ["w1_shared", "w2_shared"]
        if self.sel_bias_std > 0:
            r += ["sel_bias"]
        if self.zipf_s > 0:
            r += ["gate_bias"]
        if self.backward:
            r += ["dy"]
        return r

    def host(self, role: str) -> np.ndarray:
        """The seeded tensor on the host (float32; bf16 tensors hold exactly
        representable bf16 values)."""
        if role == "gate_bias":
            return self.gate_bias()
        return inputs.normal(self.shape(role), self.std(role), self.seed, inputs.TAG[role],
                             self.tensor_dtype(role))

    def gate_bias(self) -> np.ndarray | None:
        if self.zipf_s <= 0:
            return None
        r = inputs.random_ranks(self.E, self.seed)
        return (self.zipf_scale * r.astype(np.float64) ** (-self.zipf_s)).astype(np.float32)

    def flops_fwd(self) -> int:
        mats = 3 if self.act == SWIGLU else 2
        f = 2 * self.T * self.K * mats * self.h * self.F
        f += 2 * self.T * self.n_shared * mats * self.h * self.F
        return f


TINY = Workload("tiny_fp32_T256_h128_E8_K2_F512_gelu", T=256, h=128, E=8, K=2, F=512,
                dtype="f32", act=GELU, has_bias=True, router_std=None, seed=0)
MIXTRAL = Workload("mixtral8x7b_T8192_h4096_E8_K2_F14336", T=8192, h=4096, E=8, K=2, F=14336,
                   seed=2)
QWEN3 = Workload("qwen3_235b_T16384_h4096_E128_K8_F1536_zipf", T=16384, h=4096, E=128, K=8,
                 F=1536, zipf_s=1.1, seed=3)
DSV3 = Workload("deepseek_v3_T4096_h7168_E256_K8_F2048_sigmoid_shared", T=4096, h=7168, E=256,
                K=8, F=2048, score=SIGMOID, n_shared=1, sel_bias_std=0.1, backward=True, seed=4)


def sweep():
    out = []
    for E in (64, 128, 256):
        for T in (2048, 8192, 32768):
            for fb in (False, True):
                out.append(Workload(f"sweep_T{T}_h2048_E{E}_K8_F1024_{'balanced' if fb else 'random'}",
                                    T=T, h=2048, E=E, K=8, F=1024, force_balance=fb, seed=5))
    return out


ALL = {w.name: w for w in [TINY, MIXTRAL, QWEN3, DSV3] + sweep()}
