#!/usr/bin/env python3
"""MoE-layer forward benchmark on GB300 (one process per GPU).

A step is one pass of the whole layer -- Route, Dispatch, the tensor-core
expert GEMMs (FC1, FC2, and the shared expert when the workload has one) and
Combine -- over one batch of seeded synthetic tokens, issued through the C
ABI (include/moe.h) one stage at a time so each stage is timed with CUDA
events on the launching stream.  L2 is flushed (a 512 MB write) before every
step, outside the timed events.

Default workload: the Mixtral-8x7B-shaped layer (T=8192, h=4096, E=8, top-2,
SwiGLU F=14336, bf16).  With N GPUs every rank runs its own replica on its own
tokens (weak scaling, no collective on the data path); the per-step time is
the max over ranks.

Printed line (rank 0): value = tokens/s over all ranks with inputs resident;
e2e = the same through moe_layer_fwd with the tokens copied in from pinned host
memory and the output copied back every step; roofline of the dominant kernel
(FC1 grouped GEMM); cpu_baseline = the float64 CPU oracle on a bounded sample.
`--impl reference` times that oracle alone as the reference arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; grouped-GEMM % bf16 peak; permute/combine % HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# stage boundaries recorded by moe_layer_fwd / moe_layer_bwd (moe_set_stage_events)
FWD_STAGES = ["route", "dispatch", "fc1", "fc2", "shared", "combine"]
BWD_STAGES = ["dy_scatter", "fc2_dgrad", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad", "shared",
              "router", "combine"]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None, help="workload name (default: the Mixtral-shaped layer)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-mxfp8", action="store_true",
                   help="skip the MXFP8 expert-MLP measurement reported beside the bf16 line")
    p.add_argument("--gather", action="store_true",
                   help="time the forward with the gather-fused FC1 (no x_perm) instead of the "
                        "x_perm scatter")
    p.add_argument("--no-graph", action="store_true",
                   help="time eager launches only (default: the step is also captured in a CUDA "
                        "graph and the graph replays give the headline time)")
    p.add_argument("--sample-tokens", type=int, default=0, help="oracle sample size (0: auto)")
    p.add_argument("--tiling", choices=["auto", "1cta", "2cta"], default="auto",
                   help="expert GEMM tiling: auto (CTA pairs when experts average >= 512 rows)")
    p.add_argument("--tokens", type=int, default=0,
                   help="override T (smaller cases for profiler captures; not a bench line)")
    p.add_argument("--hbm-write", action="store_true",
                   help="only measure this GPU's write-only and copy HBM bandwidth (torch fill_ / "
                        "copy_ over 16 GB, best of 10, CUDA events) and print one JSON line")
    p.add_argument("--shape", default="",
                   help="override workload fields, e.g. T=512,h=4096,E=32,F=2048 (profiler cases)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (each rank gets it): the job's step
    time is the slowest replica's."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job throughput of weak-scaled replicas: every rank processes its
    own tokens_per_rank tokens per step of `ms` (the max over ranks)."""
    return world * tokens_per_rank / (ms / 1000.0)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def window(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sel = [r for t, r in self.rows if self.t_on and self.t_on - 0.06 <= t <= (self.t_off or t) + 0.06]
        if not sel:
            sel = [r for _, r in self.rows]
        mhz, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in sel:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
class OracleSample:
    """Host inputs for a sample of tokens that route to few experts, so the
    oracle only needs those experts' weights (generated on the host by the
    same seeded generator as the device inputs)."""

    def __init__(self, w, want: int):
        import numpy as np
        from mixture_experts_layer_softmax_gb300 import inputs
        from oracle import moe_oracle as O
        self.w = w
        self.x = w.host("x")
        self.w_r = w.host("w_r")
        self.sel_bias = w.host("sel_bias") if w.sel_bias_std > 0 else None
        self.gate_bias = w.gate_bias()
        logits = O.gating_logits(self.x, self.w_r, self.gate_bias)
        idx, probs = O.route(logits, w.K, w.score, w.renorm, self.sel_bias, w.force_balance)
        self.routing = (logits, idx, probs)
        # Grow an expert set token by token (in token order) while the host
        # weights it needs stay under a budget; the sample is the tokens whose
        # experts all lie in the set.
        per_expert = (w.w1_rows * w.h + w.h * w.F)
        budget = 4.0e8  # elements generated on the host
        chosen = set()
        for t in range(w.T):
            new = set(idx[t].tolist()) - chosen
            if (len(chosen) + len(new)) * per_expert > budget:
                continue
            chosen |= new
            if np.isin(idx, sorted(chosen)).all(axis=1).sum() >= want:
                break
        toks = np.nonzero(np.isin(idx, sorted(chosen)).all(axis=1))[0]
        self.tokens = toks[:want]
        need = sorted(set(idx[self.tokens].ravel().tolist()))
        R1, h, F = w.w1_rows, w.h, w.F
        st = w.std
        self.w1 = {e: inputs.normal((R1, h), st("w1"), w.seed, inputs.TAG["w1"], w.dtype, start=e * R1 * h)
                   for e in need}
        self.w2 = {e: inputs.normal((h, F), st("w2"), w.seed, inputs.TAG["w2"], w.dtype, start=e * h * F)
                   for e in need}
        self.b1 = self.b2 = None
        if w.has_bias:
            b1, b2 = w.host("b1"), w.host("b2")
            self.b1, self.b2 = b1, b2
        self.w1s = w.host("w1_shared") if w.n_shared else None
        self.w2s = w.host("w2_shared") if w.n_shared else None
        self.experts = need
        if w.backward:
            # The training step on the sampled tokens as a compact layer of its
            # own: only their experts (renumbered 0..n-1), their routing kept.
            # Each token's dx, and its share of the weight gradients, depend
            # only on its own experts, so the sample's work and its dx are the
            # full step's for those tokens.
            remap = {e: i for i, e in enumerate(need)}
            logits, idx, probs = self.routing
            tk = self.tokens
            self.sub_routing = (logits[tk][:, need], np.vectorize(remap.get)(idx[tk]).astype(np.int32),
                                probs[tk])
            self.sub_x = self.x[tk]
            self.sub_dy = w.host("dy")[tk]
            self.sub_w_r = self.w_r[need]
            self.sub_w1 = np.stack([self.w1[e] for e in need])
            self.sub_w2 = np.stack([self.w2[e] for e in need])

    def run(self):
        """The sampled tokens' layer output by the plain C++ oracle (double
        loops, OpenMP over tokens), from the routing decided for every token."""
        from oracle import moe_oracle_c as C
        w = self.w
        _, idx, probs = self.routing
        return C.layer_fwd(self.x, idx, probs, self.w1, self.w2, w.act, b1=self.b1, b2=self.b2,
                           w1_shared=self.w1s, w2_shared=self.w2s, tokens=self.tokens)

    def cores(self):
        from oracle import moe_oracle_c as C
        return (blas_threads() if self.w.backward else C.threads()) or 1

    def kind(self):
        return ("float64 numpy oracle forward + backward" if self.w.backward else
                "plain C++ oracle (double loops, OpenMP over tokens) forward")

    def run_train(self):
        """Forward then backward of the sampled tokens; returns their dx."""
        from oracle import moe_oracle as O
        w = self.w
        args = (self.sub_x, self.sub_w_r, self.sub_w1, self.sub_w2)
        O.layer_fwd(*args, w.K, w.score, w.act, w1_shared=self.w1s, w2_shared=self.w2s,
                    routing=self.sub_routing)
        return O.layer_bwd(*args, self.sub_dy, w.K, w.score, w.act, w1_shared=self.w1s,
                           w2_shared=self.w2s, routing=self.sub_routing)["dx"]


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count()


def auto_sample(w):
    per_tok = 2.0 * (w.K + w.n_shared) * (3 if w.act == 1 else 2) * w.h * w.F
    if w.backward:  # forward + backward: about three times the forward's work
        per_tok *= 3
    return int(max(16, min(1024, 1.5e11 / per_tok)))


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    S = args.sample_tokens or auto_sample(w)
    samp = OracleSample(w, S)
    run = samp.run_train if w.backward else samp.run
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    n = len(samp.tokens)
    ms = 1000.0 * statistics.mean(times)
    value = n / (ms / 1000.0)
    cores = samp.cores()
    sample = (f"{n} tokens of {w.name} routed only to experts {samp.experts}; {samp.kind()}, "
              f"one sample per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def workload_config(w):
    return {"workload": w.name, "T": w.T, "h": w.h, "E": w.E, "K": w.K, "F": w.F,
            "score": "sigmoid" if w.score == 1 else "softmax",
            "act": "swiglu" if w.act == 1 else "gelu", "n_shared": w.n_shared,
            "routing": "force-balanced" if w.force_balance else "router",
            "l2": "flushed before every timed step (512 MB write, outside the events)",
            "timing": "CUDA events per step; value from CUDA-graph replays of the step, stage "
                      "breakdown from eager launches queued behind a GPU-side sleep",
            "inputs": "seeded synthetic (SplitMix64 + Box-Muller), generated on the device"}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def kernel_hash(sources=None):
    h = hashlib.sha256()
    for f in sources or ("gemm_tc.cu", "gemm_tc2.cu", "tc_ptx.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "mixture_experts_layer_softmax_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(w, stage="fc1"):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum
    from one ncu capture) of the kernel of `stage`, if profiles/traffic.json
    holds a record for this workload taken with the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(w.name)
    except Exception:
        return None
    if rec and stage != "fc1":
        rec = rec.get("stages", {}).get(stage)
    if not rec or rec.get("kernel_hash") != kernel_hash(rec.get("sources")):
        return None
    return rec.get("bytes_per_launch", rec.get("fc1_bytes_per_launch"))


def expert_gemm_work(w):
    """Algorithmic work of each routed-expert grouped GEMM of the training
    step: (FLOPs, bytes) per launch, every operand read once and every result
    written once (b = 2 bytes, P = T*K permuted rows, R1 = 2F for SwiGLU)."""
    T, h, E, K, F = w.T, w.h, w.E, w.K, w.F
    P, R1, b = T * K, w.w1_rows, 2
    nt = (F + 255) // 256  # dprob partials of the FC2 data gradient
    return {
        # x_perm, W1 in; a and the saved pre-activation H out
        "fc1": (2.0 * P * h * R1, b * (P * h + E * R1 * h + P * F + P * R1)),
        # a, W2 in; y_perm out
        "fc2": (2.0 * P * F * h, b * (P * F + E * h * F + P * h)),
        # dy_perm, W2, H in; dH and the dprob partials out
        "fc2_dgrad": (2.0 * P * h * F, b * (P * h + E * h * F + P * R1 + P * R1) + 4 * P * nt),
        # dy_perm, a in; dW2 out
        "fc2_wgrad": (2.0 * P * h * F, b * (P * h + P * F + E * h * F)),
        # dH, W1 in; dx_perm out
        "fc1_dgrad": (2.0 * P * R1 * h, b * (P * R1 + E * R1 * h + P * h)),
        # dH, x_perm in; dW1 out
        "fc1_wgrad": (2.0 * P * R1 * h, b * (P * R1 + P * h + E * R1 * h)),
    }


GEMM_KERNELS = {
    "fc1": "grouped_gemm_tc_kernel<FC1>", "fc2": "grouped_gemm_tc_kernel<FC2>",
    "fc2_dgrad": "grouped_gemm_tc_bwd_kernel<dgrad> (FC2, dSwiGLU + dprob epilogue)",
    "fc2_wgrad": "grouped_gemm_tc_bwd_kernel<wgrad> (dW2)",
    "fc1_dgrad": "grouped_gemm_tc_bwd_kernel<dgrad> (FC1)",
    "fc1_wgrad": "grouped_gemm_tc_bwd_kernel<wgrad> (dW1)",
}


def kernel_roofline(name, flops, nbytes, ms, pk, pk_kind, peak_tf):
    """Roofline of one launch: bound by HBM when its arithmetic intensity is
    below the ridge point of the measured peaks, else by the tensor cores."""
    gbs = nbytes / (ms / 1000.0) / 1e9
    tfs = flops / (ms / 1000.0) / 1e12
    ridge = peak_tf * 1e12 / (pk["hbm_gbs"] * 1e9)
    hbm = flops / nbytes < ridge
    r = {"kernel": name, "bound": "hbm" if hbm else "tensor",
         "achieved": gbs if hbm else tfs, "peak": pk["hbm_gbs"] if hbm else peak_tf,
         "unit": "GB/s" if hbm else "TFLOP/s",
         "peak_kind": (f"{pk_kind} HBM copy" if hbm else f"{pk_kind} bf16 burst (cuBLAS)"),
         "bytes_per_launch": nbytes, "flops_per_launch": flops, "ms_per_launch": ms,
         "hbm_gbs": gbs, "tflops": tfs, "tensor_frac": tfs / peak_tf,
         "hbm_frac": gbs / pk["hbm_gbs"]}
    r["frac"] = r["achieved"] / r["peak"]
    return r


def time_mxfp8(M, torch, w, cfg, x, w_r, gate_bias, sel_bias, w1, w2, w1s, w2s, flush_buf, hold,
               stream, steps):
    """The layer forward with MXFP8 expert GEMMs: the bf16 router, the dispatch
    with the quantisation fused in (moe_permute_mxfp8: maps + x_perm in
    MXFP8), FC1 with the SwiGLU epilogue writing a in MXFP8, FC2, the shared
    expert the same way (its x quantised on its own), and the combine.  The
    weights are quantised once beforehand (timed on their own).  Device times
    with CUDA events per stage, L2 flushed before every step; the whole step
    is also replayed from a CUDA graph."""
    T, h, E, K, F = w.T, w.h, w.E, w.K, w.F
    P = T * K
    dev = x.device
    u8 = dict(dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    R1 = 2 * F
    w1q, w1sf = torch.empty(E * R1, h, **u8), torch.empty(M.moe_mxfp8_scale_bytes(E * R1, h, E), **u8)
    w2q, w2sf = torch.empty(E * h, F, **u8), torch.empty(M.moe_mxfp8_scale_bytes(E * h, F, E), **u8)
    ws = torch.empty(M.moe_workspace_size(cfg), **u8)
    idx, prob = torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device=dev)
    xq, xsf = torch.empty(P, h, **u8), torch.empty(M.moe_mxfp8_scale_bytes(P, h, E), **u8)
    aq, asf = torch.empty(P, F, **u8), torch.empty(M.moe_mxfp8_scale_bytes(P, F, E), **u8)
    y_perm = torch.empty(P, h, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, h, dtype=torch.bfloat16, device=dev)
    if w.n_shared:
        cs = M.make_config(T, h, 1, 1, F, cfg.dtype, cfg.score, cfg.act, 0, 0, cfg.flags)
        soff = torch.tensor([0, T], **i32)
        s1q, s1sf = torch.empty(R1, h, **u8), torch.empty(M.moe_mxfp8_scale_bytes(R1, h, 1), **u8)
        s2q, s2sf = torch.empty(h, F, **u8), torch.empty(M.moe_mxfp8_scale_bytes(h, F, 1), **u8)
        sxq, sxsf = torch.empty(T, h, **u8), torch.empty(M.moe_mxfp8_scale_bytes(T, h, 1), **u8)
        saq, sasf = torch.empty(T, F, **u8), torch.empty(M.moe_mxfp8_scale_bytes(T, F, 1), **u8)
        y_s = torch.empty(T, h, dtype=torch.bfloat16, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    wq0, wq1 = ev(), ev()
    flush_buf.fill_(1)
    wq0.record(stream)
    M.moe_mxfp8_quantize(E * R1, h, E, None, w1, w1q, w1sf)
    M.moe_mxfp8_quantize(E * h, F, E, None, w2, w2q, w2sf)
    if w.n_shared:
        M.moe_mxfp8_quantize(R1, h, 1, None, w1s, s1q, s1sf)
        M.moe_mxfp8_quantize(h, F, 1, None, w2s, s2q, s2sf)
    wq1.record(stream)
    stages = ["route", "dispatch_mxfp8", "fc1", "fc2", "shared", "combine"]

    def step(marks=None):
        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        mark(0)
        M.moe_router_topk(cfg, x, w_r, gate_bias, sel_bias, None, idx, prob, None, ws)
        mark(1)
        M.moe_permute_mxfp8(cfg, x, idx, prob, xq, xsf, counts, offsets, dst_row, src_token,
                            perm_prob, ws)
        mark(2)
        M.moe_expert_fc1_mxfp8(cfg, xq, xsf, offsets, perm_prob, w1q, w1sf, None, aq, asf)
        mark(3)
        M.moe_expert_fc2_mxfp8(cfg, aq, asf, offsets, w2q, w2sf, y_perm)
        mark(4)
        if w.n_shared:
            M.moe_mxfp8_quantize(T, h, 1, soff, x, sxq, sxsf)
            M.moe_expert_fc1_mxfp8(cs, sxq, sxsf, soff, None, s1q, s1sf, None, saq, sasf)
            M.moe_expert_fc2_mxfp8(cs, saq, sasf, soff, s2q, s2sf, y_s)
        mark(5)
        M.moe_unpermute_combine(cfg, y_perm, dst_row, None, y_s if w.n_shared else None, y)
        mark(6)

    for _ in range(3):
        flush_buf.fill_(1)
        step()
    torch.cuda.synchronize()
    marks = [[ev() for _ in range(len(stages) + 1)] for _ in range(steps)]
    for i in range(steps):
        flush_buf.fill_(1)
        hold()
        step(marks[i])
    torch.cuda.synchronize()
    st = M.moe_get_error()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status after the MXFP8 steps: {M.moe_status_string(st)}")
    stage_ms = {n: statistics.mean(m[j].elapsed_time(m[j + 1]) for m in marks)
                for j, n in enumerate(stages)}
    ms = statistics.mean(m[0].elapsed_time(m[-1]) for m in marks)
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        gev = [(ev(), ev()) for _ in range(steps)]
        for i in range(steps):
            flush_buf.fill_(1)
            gev[i][0].record(stream)
            g.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        graph_ms = statistics.mean(a.elapsed_time(b) for a, b in gev)
        ms = graph_ms
    except Exception as exc:  # keep the eager number
        print(f"MXFP8 graph capture unavailable: {exc}", file=sys.stderr)
    return {"layer_fwd_ms": ms, "tokens_per_s": T / (ms / 1000.0), "cuda_graph": graph_ms is not None,
            "stages_ms": stage_ms, "fc1_ms": stage_ms["fc1"], "fc2_ms": stage_ms["fc2"],
            "weight_quantize_ms": wq0.elapsed_time(wq1), "y": y,
            "how": "moe_router_topk + moe_permute_mxfp8 + moe_expert_fc1_mxfp8 (a written in "
                   "MXFP8) + moe_expert_fc2_mxfp8 (+ shared expert in MXFP8) + "
                   "moe_unpermute_combine; weights quantised once beforehand "
                   "(weight_quantize_ms); reported beside the bf16 headline, not in it"}


def run_ours(args, w):
    import numpy as np
    import torch
    from mixture_experts_layer_softmax_gb300 import _build, inputs
    _build.build()
    from mixture_experts_layer_softmax_gb300 import moe as M

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    bf = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    T, h, E, K, F = w.T, w.h, w.E, w.K, w.F
    P = T * K
    seed = w.seed + 1000 * rank  # each replica its own tokens

    def gen(role, shape, dtype, s=None):
        t = torch.empty(shape, dtype=dtype, device=dev)
        M.synth_normal(t, w.seed if s is None else s, inputs.TAG[role], w.std(role))
        return t

    x = gen("x", (T, h), bf, seed)
    w_r = torch.from_numpy(w.host("w_r")).to(dev)
    w1 = gen("w1", (E, w.w1_rows, h), bf)
    w2 = gen("w2", (E, h, F), bf)
    b1 = gen("b1", (E, F), bf) if w.has_bias else None
    b2 = gen("b2", (E, h), bf) if w.has_bias else None
    w1s = gen("w1_shared", (w.w1_rows, h), bf) if w.n_shared else None
    w2s = gen("w2_shared", (h, F), bf) if w.n_shared else None
    sel_bias = torch.from_numpy(w.host("sel_bias")).to(dev) if w.sel_bias_std > 0 else None
    gb = w.gate_bias()
    gate_bias = torch.from_numpy(gb).to(dev) if gb is not None else None

    tiling = {"auto": 0, "1cta": M.MOE_FLAG_GEMM_1CTA, "2cta": M.MOE_FLAG_GEMM_2CTA}[args.tiling]
    # the router hands the dispatch its per-chunk expert histograms (as
    # moe_layer_fwd does internally)
    cfg = M.config_for(w, tiling | M.MOE_FLAG_HIST_FROM_ROUTER)
    ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.empty(T, K, **i32)
    prob = torch.empty(T, K, dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    dst_row, src_token = torch.empty(T, K, **i32), torch.empty(P, **i32)
    perm_prob = torch.empty(P, dtype=torch.float32, device=dev)
    x_perm = torch.empty(P, h, dtype=bf, device=dev)
    a = torch.empty(P, F, dtype=bf, device=dev)
    y_perm = torch.empty(P, h, dtype=bf, device=dev)
    y = torch.empty(T, h, dtype=bf, device=dev)
    if w.n_shared:
        cs = M.make_config(T, h, 1, 1, F, cfg.dtype, cfg.score, cfg.act, 0, 0, cfg.flags)
        soff = torch.tensor([0, T], **i32)
        a_s = torch.empty(T, F, dtype=bf, device=dev)
        y_s = torch.empty(T, h, dtype=bf, device=dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    stages = ["route", "dispatch", "fc1", "fc2", "shared", "combine"]
    train = w.backward
    # --gather: dispatch builds only the maps and FC1 gathers the token rows
    # (moe_expert_fc1_gather); by default the rows are scattered into x_perm
    # once, as moe_layer_fwd does
    gather = w.dtype == "bf16" and args.gather
    if train:
        # training step: the whole forward (saving for backward) then the whole
        # backward, each one C-ABI call, on the same workspace
        cfg = M.config_for(w, M.MOE_FLAG_SAVE_FOR_BWD | tiling)
        ws = torch.empty(M.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
        dy = gen("dy", (T, h), bf, seed)
        dx = torch.empty(T, h, dtype=bf, device=dev)
        dw_r = torch.empty(E, h, dtype=torch.float32, device=dev)
        dw1 = torch.empty_like(w1)
        dw2 = torch.empty_like(w2)
        dw1s = torch.empty_like(w1s) if w.n_shared else None
        dw2s = torch.empty_like(w2s) if w.n_shared else None
        stages = ["forward", "backward"]

        def step(ev=None, x_=None, dy_=None, dx_=None):
            if ev is not None:
                ev[0].record(stream)
            M.moe_layer_fwd(cfg, x if x_ is None else x_, w_r, gate_bias, sel_bias, w1, b1, w2,
                            b2, w1s, w2s, y, None, None, ws)
            if ev is not None:
                ev[1].record(stream)
            M.moe_layer_bwd(cfg, x if x_ is None else x_, w_r, w1, w2, w1s, w2s,
                            dy if dy_ is None else dy_, dx if dx_ is None else dx_, dw_r, None,
                            dw1, dw2, dw1s, dw2s, ws)
            if ev is not None:
                ev[2].record(stream)
    else:
        def step(ev=None):
            def mark(i):
                if ev is not None:
                    ev[i].record(stream)
            mark(0)
            M.moe_router_topk(cfg, x, w_r, gate_bias, sel_bias, None, idx, prob, None, ws)
            mark(1)
            if gather:  # maps only: FC1 gathers the token rows itself
                M.moe_permute(cfg, None, idx, prob, None, counts, offsets, dst_row, src_token,
                              perm_prob, ws)
            else:
                M.moe_permute(cfg, x, idx, prob, x_perm, counts, offsets, dst_row, src_token,
                              perm_prob, ws)
            mark(2)
            if gather:
                M.moe_expert_fc1_gather(cfg, x, src_token, offsets, perm_prob, w1, b1, None, a)
            else:
                M.moe_expert_fc1(cfg, x_perm, offsets, perm_prob, w1, b1, None, a)
            mark(3)
            M.moe_expert_fc2(cfg, a, offsets, perm_prob, w2, b2, y_perm)
            mark(4)
            if w.n_shared:
                M.moe_expert_fc1(cs, x, soff, None, w1s, None, None, a_s)
                M.moe_expert_fc2(cs, a_s, soff, None, w2s, None, y_s)
            mark(5)
            M.moe_unpermute_combine(cfg, y_perm, dst_row, None, y_s if w.n_shared else None, y)
            mark(6)

    # kernels of this library per step: route (bf16: one kernel for E <= 8,
    # else split W_r, the gating GEMM, selection; fp32: one fused kernel for
    # E <= 32, else GEMM and selection), dispatch (maps, row scatter), FC1 and
    # FC2, the shared expert's two GEMMs (+ its offsets in moe_layer_fwd),
    # combine
    # The router also hands the dispatch its per-chunk expert histograms: the
    # one-launch router (bf16, E <= 8) from its epilogue, the other paths by
    # the histogram step launched right after them.
    if w.dtype == "bf16":
        route_k = 1 if E <= 8 else 3 + 1
    else:
        route_k = (1 if E <= 32 else 2) + 1
    # dispatch: per-expert scan (folded into the ranks kernel when
    # ceil(T/32) * E <= 8192), ranks, and the row scatter unless FC1 gathers
    maps_k = 1 if ((T + 31) // 32) * E <= 8192 else 2
    dispatch_k = maps_k + (0 if (gather and not train) else 1)
    launches_per_step = route_k + dispatch_k + 2 + ((3 if train else 2) if w.n_shared else 0) + 1
    if train:  # backward: scatter, 4 GEMMs (+4 shared), dprob, router, router wgrad, combine
        launches_per_step += 1 + 4 + (4 if w.n_shared else 0) + 4
    # Eager stage timing: a GPU-side sleep after the L2 flush lets the host
    # enqueue the whole step before the GPU reaches it, so the events between
    # stages measure device time, not the host's launch rate.
    def hold():
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(2_000_000)
    n_ev = len(stages) + 1

    for _ in range(max(args.warmup, 3)):
        flush_buf.fill_(1)
        step()
    torch.cuda.synchronize()
    st = M.moe_get_error()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {M.moe_status_string(st)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    # Training: the library records these events at the stage boundaries
    # inside moe_layer_fwd / moe_layer_bwd (moe_set_stage_events), on the
    # stream that launches the kernels, so every expert GEMM of the step is
    # timed on its own inside the timed steps.
    st_fwd = st_bwd = None
    if train:
        st_fwd = [[torch.cuda.Event(enable_timing=True) for _ in FWD_STAGES + ["end"]]
                  for _ in range(args.steps)]
        st_bwd = [[torch.cuda.Event(enable_timing=True) for _ in BWD_STAGES + ["end"]]
                  for _ in range(args.steps)]
        for e in [e for row in st_fwd + st_bwd for e in row]:
            e.record(stream)  # creates the CUDA event
        torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.window(True)
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush_buf.fill_(1)
        if train:
            M.moe_set_stage_events(M.MOE_PASS_FWD, st_fwd[i])
            M.moe_set_stage_events(M.MOE_PASS_BWD, st_bwd[i])
        hold()
        step(evs[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if train:
        M.moe_set_stage_events(M.MOE_PASS_FWD, [])
        M.moe_set_stage_events(M.MOE_PASS_BWD, [])
    sampler.window(False)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    st = M.moe_get_error()
    if st != M.MOE_OK:
        raise RuntimeError(f"device status after the timed steps: {M.moe_status_string(st)}")

    # the standalone permute (maps + x_perm row scatter), as the training path
    # and moe_permute callers run it, timed on its own
    permute_ms = None
    if not train:
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush_buf.fill_(1)
            hold()
            pev[i][0].record(stream)
            M.moe_permute(cfg, x, idx, prob, x_perm, counts, offsets, dst_row, src_token,
                          perm_prob, ws)
            pev[i][1].record(stream)
        torch.cuda.synchronize()
        permute_ms = statistics.mean(a.elapsed_time(b) for a, b in pev)

    # The router and the dispatch on their own, each captured in a CUDA graph
    # and replayed with the L2 flush in between (as the layer runs in the
    # headline), so their launches follow one another without host gaps.
    def graph_time(fn):
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                flush_buf.fill_(1)
                hold()  # as in the eager timing: the flush's write-backs drain first
                ev[i][0].record(stream)
                g.replay()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b) for a, b in ev)
        except Exception as exc:
            print(f"graph capture unavailable: {exc}", file=sys.stderr)
            return None

    route_graph_ms = permute_graph_ms = None
    if not train and not args.no_graph:
        route_graph_ms = graph_time(lambda: M.moe_router_topk(cfg, x, w_r, gate_bias, sel_bias,
                                                              None, idx, prob, None, ws))
        permute_graph_ms = graph_time(lambda: M.moe_permute(cfg, x, idx, prob, x_perm, counts,
                                                            offsets, dst_row, src_token,
                                                            perm_prob, ws))
    per_step = [e[0].elapsed_time(e[n_ev - 1]) for e in evs]
    stage_ms = {s: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, s in enumerate(stages)}
    sub_ms = None
    if train:
        sub_ms = {"forward": {n: statistics.mean(r[j].elapsed_time(r[j + 1]) for r in st_fwd)
                              for j, n in enumerate(FWD_STAGES)},
                  "backward": {n: statistics.mean(r[j].elapsed_time(r[j + 1]) for r in st_bwd)
                               for j, n in enumerate(BWD_STAGES)}}
    ms_eager = ms = statistics.mean(per_step)

    # The same step captured once in a CUDA graph (the layer never syncs or
    # allocates, so it captures as is), replayed with the L2 flush in between.
    graph_ms = None
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
            torch.cuda.synchronize()
            gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            for i in range(args.steps):
                flush_buf.fill_(1)
                hold()
                gev[i][0].record(stream)
                g.replay()
                gev[i][1].record(stream)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            graph_ms = statistics.mean(a.elapsed_time(b) for a, b in gev)
            st = M.moe_get_error()
            if st != M.MOE_OK:
                raise RuntimeError(M.moe_status_string(st))
            ms = graph_ms
        except Exception as exc:  # report, keep the eager number
            print(f"graph capture unavailable: {exc}", file=sys.stderr)
            graph_ms = None
    ms = max_over_ranks(ms, world, dev)
    value = job_tokens_per_s(world, T, ms)

    # ---- end to end through the public calls with host buffers ----
    # Every step copies its inputs in from pinned host memory and its result
    # back to pinned host memory; a copy stream overlaps step i+1's upload and
    # step i's download with step i's compute (double-buffered on both sides).
    # All copies lie inside the timed region.  Forward: x in, y out through
    # moe_layer_fwd.  Training: x and dy in, dx out (the gradient handed to
    # the layer below) through moe_layer_fwd + moe_layer_bwd; the weight
    # gradients stay on the device, where an optimizer step would use them.
    e2e = None
    if not args.no_e2e:
        K2 = max(args.steps, 2)
        srcs = [x, dy] if train else [x]
        dsts = [dx] if train else [y]
        host_in = [[t.cpu().pin_memory() for t in srcs] for _ in range(2)]
        host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dsts]
                    for _ in range(2)]
        dev_in = [[torch.empty_like(t) for t in srcs] for _ in range(2)]
        dev_out = [[torch.empty_like(t) for t in dsts] for _ in range(2)]
        cs = torch.cuda.Stream(dev)
        ev_up = [torch.cuda.Event(), torch.cuda.Event()]
        ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
        ev_down = [torch.cuda.Event(), torch.cuda.Event()]

        def compute_eager(b):
            if train:
                step(x_=dev_in[b][0], dy_=dev_in[b][1], dx_=dev_out[b][0])
            else:
                M.moe_layer_fwd(cfg, dev_in[b][0], w_r, gate_bias, sel_bias, w1, b1, w2, b2, w1s,
                                w2s, dev_out[b][0], None, None, ws)

        # As for `value`, the layer's calls are captured in a CUDA graph (one
        # per buffer set) and replayed each step; the copies stay outside.
        comp_graphs = None
        if not args.no_graph:
            try:
                comp_graphs = []
                for b in range(2):
                    g_ = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g_):
                        compute_eager(b)
                    comp_graphs.append(g_)
                torch.cuda.synchronize()
            except Exception as exc:  # report, keep eager launches
                print(f"e2e graph capture unavailable: {exc}", file=sys.stderr)
                comp_graphs = None

        def compute(b):
            if comp_graphs is not None:
                comp_graphs[b].replay()
            else:
                compute_eager(b)

        def upload(b):
            for d_, h_ in zip(dev_in[b], host_in[b]):
                d_.copy_(h_, non_blocking=True)

        def pipeline(n):
            with torch.cuda.stream(cs):
                upload(0)
                ev_up[0].record(cs)
            for i in range(n):
                b = i % 2
                stream.wait_event(ev_up[b])
                if i >= 2:
                    stream.wait_event(ev_down[b])  # dev_out[b] has been read back
                compute(b)
                ev_comp[b].record(stream)
                with torch.cuda.stream(cs):
                    if i + 1 < n:
                        nb_ = (i + 1) % 2
                        if i >= 1:
                            cs.wait_event(ev_comp[nb_])  # step i-1 is done reading dev_in[nb_]
                        upload(nb_)
                        ev_up[nb_].record(cs)
                    cs.wait_event(ev_comp[b])
                    for h_, d_ in zip(host_out[b], dev_out[b]):
                        h_.copy_(d_, non_blocking=True)
                    ev_down[b].record(cs)

        pipeline(3)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        pipeline(K2)
        cs.wait_stream(stream)
        t1.record(cs)
        torch.cuda.synchronize()
        ems = t0.elapsed_time(t1) / K2
        ems = max_over_ranks(ems, world, dev)
        nbytes = lambda ts: sum(t.numel() * t.element_size() for t in ts)
        e2e = {"value": job_tokens_per_s(world, T, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": nbytes(srcs), "d2h_bytes_per_step": nbytes(dsts),
               "ms_per_step": ems,
               "how": ("moe_layer_fwd + moe_layer_bwd per step; x and dy copied in from pinned "
                       "host memory and dx copied back every step" if train else
                       "moe_layer_fwd per step; tokens copied in from pinned host memory and the "
                       "output copied back every step") +
                      ", on a copy stream overlapped with compute" +
                      (", the layer's calls replayed from a CUDA graph per buffer set"
                       if comp_graphs is not None else ", eager launches")}

    mx = None
    if (not train and not args.no_mxfp8 and w.dtype == "bf16" and w.act == 1
            and not w.has_bias and h % 128 == 0 and F % 128 == 0):
        mx = time_mxfp8(M, torch, w, cfg, x, w_r, gate_bias, sel_bias, w1, w2, w1s, w2s,
                        flush_buf, hold, stream, args.steps)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    pk, pk_kind = peaks()
    esz = 2 if w.dtype == "bf16" else 4
    # the timed region is short and the SM clock stays at its maximum (see
    # "clocks"), so the denominator is the burst cuBLAS bf16 figure
    peak_tf = pk["bf16_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic", "config": workload_config(w), "stages_ms": stage_ms,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks, "e2e": e2e,
        "wall_s_timed": t_wall, "ms_per_step_eager": ms_eager, "cuda_graph": graph_ms is not None,
        "gemm_tiling": args.tiling,
        "forward_path": ("dispatch maps, token rows gathered inside FC1 (no x_perm)"
                         if (gather and not train) else "dispatch maps + x_perm row scatter"),
    }
    if train:
        fwd_fl = w.flops_fwd()
        tot_fl = 3 * fwd_fl  # backward GEMMs: data + weight gradients = 2x forward
        line["config"]["step"] = "forward + backward"
        line["layer_tflops"] = tot_fl / (ms / 1000.0) / 1e12
        line["layer_pct_bf16_peak"] = 100.0 * line["layer_tflops"] / peak_tf
        line["forward_tflops"] = fwd_fl / (stage_ms["forward"] / 1000.0) / 1e12
        line["backward_tflops"] = 2 * fwd_fl / (stage_ms["backward"] / 1000.0) / 1e12
        line["stages_ms"] = {"forward": stage_ms["forward"], "backward": stage_ms["backward"],
                             **{f"fwd_{k}": v for k, v in sub_ms["forward"].items()},
                             **{f"bwd_{k}": v for k, v in sub_ms["backward"].items()}}
        # every routed-expert GEMM timed alone inside the timed steps (events the
        # library records at the stage boundaries, on the launching stream)
        work = expert_gemm_work(w)
        times = {"fc1": sub_ms["forward"]["fc1"], "fc2": sub_ms["forward"]["fc2"],
                 **{k: sub_ms["backward"][k] for k in
                    ("fc2_dgrad", "fc2_wgrad", "fc1_dgrad", "fc1_wgrad")}}
        kern = {k: kernel_roofline(GEMM_KERNELS[k], work[k][0], work[k][1], times[k], pk,
                                   pk_kind, peak_tf) for k in work}
        for k, r in kern.items():
            r["traffic"] = traffic_record(w, k)
        top = max(kern, key=lambda k: kern[k]["ms_per_launch"])
        line["roofline"] = dict(kern[top], stage=top)
        line["expert_gemms"] = kern
        line["expert_gemms_how"] = (
            "bytes: every operand read once and every result written once (weights, permuted "
            "activations, saved pre-activations, weight gradients); bound hbm when FLOP/byte is "
            "below the ridge point of the measured peaks; the weight-gradient kernels only write "
            "to HBM what they produce, so `python bench.py --hbm-write`'s write-only rate is "
            "their practical ceiling")
        w_bytes = 2 * (w.E + w.n_shared) * (w.w1_rows * h + h * F)
        line["forward_weight_stream_frac"] = (w_bytes / (stage_ms["forward"] / 1000.0) / 1e9
                                              / pk["hbm_gbs"])
    else:
        fc1_flops = 2.0 * P * h * w.w1_rows
        fc2_flops = 2.0 * P * F * h
        fc1_tf = fc1_flops / (stage_ms["fc1"] / 1000.0) / 1e12
        gemm_tf = (fc1_flops + fc2_flops) / ((stage_ms["fc1"] + stage_ms["fc2"]) / 1000.0) / 1e12
        perm_bytes = T * h * esz + P * h * esz
        comb_bytes = P * h * esz + T * h * esz + (T * h * esz if w.n_shared else 0)
        perm_gbs = perm_bytes / (permute_ms / 1000.0) / 1e9
        comb_gbs = comb_bytes / (stage_ms["combine"] / 1000.0) / 1e9
        pair = args.tiling == "2cta" or (args.tiling == "auto" and P >= 512 * E)
        fc1_kernel = ("grouped_gemm_tc2_kernel<FC1> (CTA pairs)" if pair
                      else "grouped_gemm_tc_kernel<FC1>")
        if w.dtype == "bf16":
            line["roofline"] = {"kernel": fc1_kernel, "bound": "tensor",
                                "achieved": fc1_tf, "peak": peak_tf, "unit": "TFLOP/s",
                                "frac": fc1_tf / peak_tf,
                                "peak_kind": f"{pk_kind} bf16 burst (cuBLAS)",
                                "traffic": traffic_record(w), "flops_per_launch": fc1_flops,
                                "ms_per_launch": stage_ms["fc1"]}
        else:
            # fp32 runs the SIMT grouped GEMM on the FP32 ALUs: the peak is the SM count
            # x 128 FP32 lanes x 2 FLOP (FMA) x the maximum SM clock (2.07 GHz)
            n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
            alu_peak = n_sm * 128 * 2 * 2.07e9 / 1e12
            line["roofline"] = {"kernel": "grouped_gemm_simt_kernel<FC1> (fp32)", "bound": "alu",
                                "achieved": fc1_tf, "peak": alu_peak, "unit": "TFLOP/s",
                                "frac": fc1_tf / alu_peak,
                                "peak_kind": f"nominal fp32 FMA rate ({n_sm} SMs x 128 lanes x 2.07 GHz)",
                                "traffic": None, "flops_per_launch": fc1_flops,
                                "ms_per_launch": stage_ms["fc1"]}
        line["grouped_gemm_pct_bf16_peak"] = 100.0 * gemm_tf / peak_tf
        line["grouped_gemm_tflops"] = gemm_tf
        line["permute_pct_hbm"] = 100.0 * perm_gbs / pk["hbm_gbs"]
        line["permute_ms"] = permute_ms
        line["permute_how"] = ("moe_permute with the row scatter (maps + x_perm), timed alone; the "
                               "forward above " + ("gathers the rows inside FC1 instead"
                                                   if gather else "uses it"))
        line["combine_pct_hbm"] = 100.0 * comb_gbs / pk["hbm_gbs"]
        cnt = counts.cpu().numpy().astype(np.float64)  # the last step's expert loads
        line["expert_counts"] = {"min": int(cnt.min()), "max": int(cnt.max()),
                                 "mean": float(cnt.mean()),
                                 "cv": float(cnt.std() / cnt.mean()) if cnt.mean() > 0 else 0.0}
        line["route_ms"] = stage_ms["route"]
        # the router reads every token row once (its weight stays in L2/shared memory)
        line["route_pct_hbm"] = 100.0 * (T * h * esz) / (stage_ms["route"] / 1000.0) / 1e9 / pk["hbm_gbs"]
        if route_graph_ms and permute_graph_ms:
            line["graph_replays"] = {
                "route_ms": route_graph_ms,
                "route_pct_hbm": 100.0 * (T * h * esz) / (route_graph_ms / 1000.0) / 1e9 / pk["hbm_gbs"],
                "permute_ms": permute_graph_ms,
                "permute_pct_hbm": 100.0 * perm_bytes / (permute_graph_ms / 1000.0) / 1e9 / pk["hbm_gbs"],
                "how": "moe_router_topk and moe_permute each captured alone in a CUDA graph, "
                       "replayed with the L2 flushed (and its write-backs drained behind a "
                       "GPU-side sleep) before every replay"}
        if mx is not None:
            # FP8 tensor peak: the measured bf16 burst x the nominal fp8/bf16 ratio (4.5 / 2.25)
            fp8_peak = 2.0 * peak_tf
            mx["fc1_tflops"] = fc1_flops / (mx["fc1_ms"] / 1000.0) / 1e12
            mx["fc2_tflops"] = fc2_flops / (mx["fc2_ms"] / 1000.0) / 1e12
            mx["fp8_peak_tflops"] = fp8_peak
            mx["fp8_peak_kind"] = f"{pk_kind} bf16 burst x 2 (nominal fp8/bf16 ratio)"
            mx["fc1_frac_fp8_peak"] = mx["fc1_tflops"] / fp8_peak
            mx["expert_gemms_speedup_vs_bf16"] = ((stage_ms["fc1"] + stage_ms["fc2"])
                                                  / (mx["fc1_ms"] + mx["fc2_ms"]))
            mx["layer_speedup_vs_bf16"] = ms / mx["layer_fwd_ms"]
            y_mx = mx.pop("y")
            # output drift of the MXFP8 layer against this run's bf16 layer output
            d = (y_mx.float() - y.float()).abs().max().item()
            mx["max_abs_diff_vs_bf16_output"] = d
            mx["rel_diff_vs_bf16_output"] = d / max(y.float().abs().max().item(), 1e-30)
            line["mxfp8"] = mx
    if not args.no_cpu_baseline:
        S = args.sample_tokens or auto_sample(w)
        samp = OracleSample(w, S)
        run = samp.run_train if train else samp.run
        t0 = time.perf_counter()
        reps = 0
        ref = None
        while True:
            ref = run()
            reps += 1
            if time.perf_counter() - t0 > 10.0 or reps >= 50:
                break
        el = time.perf_counter() - t0
        n = len(samp.tokens)
        line["cpu_baseline"] = {
            "value": reps * n / el, "unit": "tokens/s", "cores": samp.cores(), "kind": "oracle",
            "sample": f"{n} tokens of the timed workload routed only to experts {samp.experts}, "
                      f"{samp.kind()} repeated {reps}x ({el:.1f} s)"}
        # correctness column: the same tokens from the GPU result of the last
        # step (y for the forward, dx for the training step)
        out = dx if train else y
        gpu_rows = out[torch.from_numpy(samp.tokens).to(dev)].float().cpu().numpy().astype(np.float64)
        err = float(np.abs(gpu_rows - ref).max())
        bound = 2e-2 * float(np.abs(ref).max()) + 1e-3
        line["check"] = {"tokens": n, "tensor": "dx" if train else "y", "max_abs_err": err,
                         "bound": bound, "ok": err <= bound}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def hbm_write_probe():
    """Write-only bandwidth (writes, no reads) beside the copy bandwidth the
    roofline peaks use: the expert weight gradients write dW and read little.
    Writes are timed as zero_() (a memset) and as fill_() of an int64 view
    (8-byte stores); a uint8 fill_ is not bandwidth-bound (about half of
    either) and is reported only for comparison."""
    import torch
    dev = torch.device("cuda")
    n = 16 << 30
    buf = torch.empty(n, dtype=torch.uint8, device=dev)
    src = torch.empty(n // 2, dtype=torch.uint8, device=dev)
    dst = torch.empty(n // 2, dtype=torch.uint8, device=dev)
    ops = {"zero_": lambda: buf.zero_(), "fill_int64": lambda: buf.view(torch.int64).fill_(1),
           "fill_uint8": lambda: buf.fill_(1), "copy": lambda: dst.copy_(src)}
    for f in ops.values():
        f()
    torch.cuda.synchronize()
    best = {}
    for name, f in ops.items():
        ts = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        best[name] = n / (min(ts) / 1000) / 1e9
    print(json.dumps({"write_only_gbs": max(best["zero_"], best["fill_int64"]),
                      "copy_gbs": best["copy"], "by_op_gbs": best,
                      "how": "16 GiB written by zero_ / an int64 fill_ (writes only), 8 GiB copied "
                             "(8 GiB read + 8 GiB written), best of 10, CUDA events"}), flush=True)


def main():
    args = parse()
    if args.hbm_write:
        hbm_write_probe()
        return
    from mixture_experts_layer_softmax_gb300 import workloads
    w = workloads.ALL[args.workload] if args.workload else workloads.MIXTRAL
    if args.tokens:
        w = w.replace(name=f"{w.name}_T{args.tokens}", T=args.tokens)
    if args.shape:
        kv = dict(item.split("=") for item in args.shape.split(","))
        w = w.replace(name=f"{w.name}_{args.shape.replace(',', '_').replace('=', '')}",
                      **{k: int(v) for k, v in kv.items()})
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
