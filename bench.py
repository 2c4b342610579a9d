#!/usr/bin/env python3
"""Throughput of the NVFP4 prefill layer block on GB300.

Workload (one "step"): one ubatch of T=1024 tokens through one layer block of
the 27B-class dense model -- RMSNorm + NVFP4 quantize, QKV projection
(7168 x 5120), attention-core stand-in (Q slice) + quantize, O projection
(5120 x 5120) + residual, and the MLP (RMSNorm prologue, fused gate/up
2 x 17408 x 5120 with SwiGLU + FP4 requant, down 5120 x 17408 + residual) --
as one launch set of libnvfp4 kernels, captured in a CUDA graph.  Weights are
seeded synthetic bf16 quantized once on the device (cold path, untimed).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
same workload instead (host cores, bounded sample per step).

Multi-GPU: one process per GPU (torchrun); each rank runs its own replica of
the block on its own ubatches (no collective on the data path); the timed
region is bracketed by barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "NVFP4 MLP prefill tokens/s at T=1024; GEMM TFLOPS and % of dense-FP4 peak"
EV_EVERY = 10   # steps of the timed graph between two steps with per-GEMM events
T_DEFAULT, H, I, QKV = 1024, synthetic.H, synthetic.I, synthetic.QKV
FP4_PER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor ratio
L2_BYTES = 129 * 2 ** 20


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------- inputs
def make_inputs(T):
    """bf16 bit patterns of the layer-0 weights, norms and a T-token ubatch."""
    w = synthetic.attn_weights(0)
    w.update(synthetic.mlp_weights(0))
    x = synthetic.activations(T, seed=2)
    return w, x


def weight_bytes():
    n = QKV * H + H * H + 2 * I * H + H * I
    return n // 2 + n // 16          # codes + scales


def block_flops(T):
    return 2 * T * (QKV * H + H * H + 2 * I * H + H * I)


# ---------------------------------------------------------------- peaks
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d["bf16_tflops_sustained"], "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def recorded_traffic():
    """Per-launch DRAM traffic of the fused gate/up GEMM from the committed
    ncu summary, or None if the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "gemm_swiglu_T1024.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != kernel_source_hash():
        return None
    try:
        return int(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm2.cu", "gemm_epilogue.cuh", "common.cuh", "internal.h"):
        h.update(open(os.path.join(ROOT, "nvfp4_block_scaled_device_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ CPU oracle
def oracle_weights(wbits):
    import oracle
    q = {}
    for k, name in (("qkv", "w_qkv"), ("o", "w_o"), ("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        g = oracle.global_scale(wbits[name])
        c, s = oracle.quantize(wbits[name], g)
        q[k] = (c, s, g)
    return q


def oracle_block(x_rows, wq, wbits, g_inter):
    """The oracle's layer block on a batch of token rows (the CPU statement of
    the same launch set)."""
    import oracle
    h = oracle.rmsnorm(x_rows, wbits["attn_norm"])
    g = oracle.global_scale(h)
    hc, hs = oracle.quantize(h, g)
    _, _, qkv = oracle.gemm(hc, hs, g, *wq["qkv"])
    q = np.ascontiguousarray(qkv[:, :H])
    ga = oracle.global_scale(q)
    ac, asf = oracle.quantize(q, ga)
    _, _, x1 = oracle.gemm(ac, asf, ga, *wq["o"], residual=x_rows)
    return oracle.mlp(x1, wbits["mlp_norm"], wq["gate"], wq["up"], wq["down"], g_inter=g_inter)["out"]


def cpu_baseline(wbits, x, T, budget_s=15.0):
    """Oracle tokens/s on the host cores: S tokens of the ubatch through the
    whole block, S grown until the timed call takes ~budget_s."""
    import oracle
    oracle.build()
    wq = oracle_weights(wbits)               # cold path, not timed
    g_inter = np.float32(0.0)
    S, rate, elapsed = 8, None, 0.0
    while True:
        rows = x[:S]
        # intermediate scale of this batch (per-call), fixed before timing
        if g_inter == 0.0:
            g_inter = oracle.mlp(rows[:1], wbits["mlp_norm"], wq["gate"], wq["up"], wq["down"])["g_inter"]
        t0 = time.perf_counter()
        oracle_block(rows, wq, wbits, g_inter)
        elapsed = time.perf_counter() - t0
        rate = S / elapsed
        if elapsed >= budget_s / 3 or S >= T:
            break
        S = int(min(T, max(S * 2, S * budget_s / max(elapsed, 1e-3))))
    return {"value": rate, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{S} of the {T} ubatch tokens through the whole block (oracle.gemm batch path), "
                      f"{elapsed:.1f} s; weights quantized beforehand (untimed)"}


def run_reference(args):
    """--impl reference: the oracle on the host cores, W + K steps of one
    token each; per step every GEMM is evaluated on a sampled fraction f of
    its output columns (the rest zero-filled), elementwise work in full."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    T = args.T
    wbits, x = make_inputs(T)
    wq = oracle_weights(wbits)
    rng = np.random.default_rng(5)
    g_inter = oracle.mlp(x[:1], wbits["mlp_norm"], wq["gate"], wq["up"], wq["down"])["g_inter"]
    total_macs = QKV * H + H * H + 2 * I * H + H * I

    def sampled_gemm(ac, asf, g, W, f):
        codes, sf, gw = W
        N = codes.shape[0]
        n = np.sort(rng.choice(N, size=max(1, int(round(f * N))), replace=False))
        dot, _ = oracle.dot_sampled(ac, asf, codes, sf, np.zeros(n.size, np.int64), n)
        out = np.zeros((1, N), np.float64)
        out[0, n] = float(np.float32(np.float32(g) * np.float32(gw))) * dot
        return synthetic.f32_to_bf16_bits(out.astype(np.float32)), n.size * codes.shape[1] * 2

    def step(t, f):
        row = x[t % T: t % T + 1]
        macs = 0
        h = oracle.rmsnorm(row, wbits["attn_norm"])
        g = oracle.global_scale(h)
        hc, hs = oracle.quantize(h, g)
        qkv, m = sampled_gemm(hc, hs, g, wq["qkv"], f); macs += m
        q = np.ascontiguousarray(qkv[:, :H])
        ga = oracle.global_scale(q)
        ac, asf = oracle.quantize(q, ga)
        o, m = sampled_gemm(ac, asf, ga, wq["o"], f); macs += m
        x1 = synthetic.f32_to_bf16_bits(synthetic.bf16_bits_to_f32(o) + synthetic.bf16_bits_to_f32(row))
        h2 = oracle.rmsnorm(x1, wbits["mlp_norm"])
        g2 = oracle.global_scale(h2)
        c2, s2 = oracle.quantize(h2, g2)
        gate, m = sampled_gemm(c2, s2, g2, wq["gate"], f); macs += m
        up, m = sampled_gemm(c2, s2, g2, wq["up"], f); macs += m
        s = oracle.swiglu(gate, up)
        sc, ss = oracle.quantize(s, g_inter)
        _, m = sampled_gemm(sc, ss, g_inter, wq["down"], f); macs += m
        return macs

    # size the column fraction so W + K steps take ~120 s
    t0 = time.perf_counter()
    probe_f = 1.0 / 64
    step(0, probe_f)
    per_full = (time.perf_counter() - t0) / probe_f
    f = min(1.0, max(1.0 / 4096, 120.0 / max(1, args.steps + args.warmup) / per_full))
    for i in range(args.warmup):
        step(i, f)
    t0 = time.perf_counter()
    macs = 0
    for i in range(args.steps):
        macs += step(args.warmup + i, f)
    el = time.perf_counter() - t0
    tokens = macs / total_macs
    value = tokens / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
            "data": "synthetic (seeded)",
            "config": {"workload": "prefill layer block, T=1024 ubatch: RMSNorm+QKV(7168x5120)+O(5120x5120)"
                                   "+MLP(5120->2x17408->5120), NVFP4 W4A4, H=5120", "T": T},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"each step: 1 token; every GEMM on a random {f:.4f} fraction of its output "
                                       f"columns (others zero), elementwise steps in full; tokens = MACs done / "
                                       f"MACs per token"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ multi-rank timing
def slowest_rank_ms(ms, dist=None, device=None):
    """Duration of the timed region as the whole job sees it: the maximum over
    the ranks (all-reduce MAX), or the local value in a single process."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, ms):
    """Units per second over all ranks (weak scaling: every rank processed
    units_per_rank within the slowest rank's time)."""
    return world * units_per_rank / (ms / 1e3)


# ------------------------------------------------- side measurements
def side_measurements(nv, W, stream, hbm_gbs, fp4_peak):
    """After the timed region, outside the metric: the one-launch scale +
    quantize at R=16384 x K=5120 (168 MB of bf16 per pass; achieved GB/s on
    the algorithmic bytes 2RK read + 0.5625RK written) and every GEMM shape of
    the block at T=1 (decode: weights streamed from HBM, launches in a CUDA
    graph) and T=16384 (long prefill), with the block's weights, each timed
    over a few launches with CUDA events."""
    def timed(fn, iters):
        with torch.cuda.stream(stream):
            fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(iters):
                fn()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / iters * 1e3      # us

    dev = W["o"].codes.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    out = {}
    R, K = 16384, H
    x = torch.randn((R, K), generator=gen, device=dev).bfloat16()
    w = (1 + 0.05 * torch.randn((K,), generator=gen, device=dev)).bfloat16()
    t = nv.NVFP4Tensor.empty(R, K, dev)
    ws = nv.workspace(256, dev)
    alg = 2 * R * K + 0.5625 * R * K
    for name, nw in (("scale_quantize_R16384", None), ("norm_scale_quantize_R16384", w)):
        us = timed(lambda: nv.nvfp4_scale_quantize(x, t, ws, nw, 1e-6, stream), 10)
        out[name] = {"us": us, "GB/s": alg / us / 1e3, "frac_of_hbm": alg / us / 1e3 / hbm_gbs}
    del x, t
    gws = nv.workspace(nv.gemm_workspace_bytes(), dev)
    # T=1: each GEMM streams its weights from HBM, as a decode step does:
    # launches back to back in a CUDA graph, cycling over copies of the
    # weights that together exceed twice the L2
    l2 = 129e6
    A1 = {Kk: nv.NVFP4Tensor.empty(1, Kk, dev) for Kk in (H, I)}
    for Kk, a in A1.items():
        nv.nvfp4_scale_quantize(torch.randn((1, Kk), generator=gen, device=dev).bfloat16(), a, ws, None, 1e-6, stream)

    def copies(Wt):
        n = max(2, int(2.2 * l2 // (Wt.codes.numel() + Wt.sf.numel())) + 1)
        return [nv.NVFP4Tensor(codes=Wt.codes.clone(), sf=Wt.sf.clone(), g=Wt.g.clone(), rows=Wt.rows, cols=Wt.cols)
                for _ in range(n)]

    def rotating_us(launch, n):
        k = [0]

        def fn():
            launch(k[0] % n)
            k[0] += 1
        return graph_time_us(fn, stream, 4 * n)

    res = {}
    for name, Kk in (("qkv", H), ("o", H), ("down", I)):
        Ws = copies(W[name])
        o = torch.empty((1, W[name].rows), dtype=torch.bfloat16, device=dev)
        us = rotating_us(lambda i: nv.nvfp4_gemm(A1[Kk], Ws[i], o, None, stream, gws), len(Ws))
        b = W[name].codes.numel() + W[name].sf.numel()
        res[name] = {"us": us, "TFLOP/s": 2 * W[name].rows * Kk / us / 1e6, "weight_GB/s": b / us / 1e3,
                     "frac_of_hbm": b / us / 1e3 / hbm_gbs, "weight_copies": len(Ws)}
        del Ws
    Gs, Us = copies(W["gate"]), copies(W["up"])
    s1 = nv.NVFP4Tensor.empty(1, I, dev)
    g1 = torch.tensor([0.01], dtype=torch.float32, device=dev)
    sws1 = nv.workspace(nv.swiglu_workspace_bytes(1, I, nv.NVFP4_INTER_STATIC), dev)
    us = rotating_us(lambda i: nv.nvfp4_gemm_swiglu(A1[H], Gs[i], Us[i], nv.NVFP4_INTER_STATIC, g1, s1, sws1, None,
                                                    stream), len(Gs))
    b = sum(x_.codes.numel() + x_.sf.numel() for x_ in (W["gate"], W["up"]))
    res["gate_up_swiglu"] = {"us": us, "TFLOP/s": 2 * 2 * I * H / us / 1e6, "weight_GB/s": b / us / 1e3,
                             "frac_of_hbm": b / us / 1e3 / hbm_gbs, "weight_copies": len(Gs)}
    del Gs, Us
    for v in res.values():
        v["frac_of_fp4_peak"] = v["TFLOP/s"] / fp4_peak
    res["weights"] = "HBM-resident: launches cycle over weight copies > 2x L2"
    out["gemm_T1"] = res
    del A1
    for T in (16384,):
        A = {Kk: nv.NVFP4Tensor.empty(T, Kk, dev) for Kk in (H, I)}
        for Kk, a in A.items():
            nv.nvfp4_scale_quantize(torch.randn((T, Kk), generator=gen, device=dev).bfloat16(), a, ws, None, 1e-6,
                                    stream)
        res = {}
        for name, Wt, Kk in (("qkv", W["qkv"], H), ("o", W["o"], H), ("down", W["down"], I)):
            o = torch.empty((T, Wt.rows), dtype=torch.bfloat16, device=dev)
            us = timed(lambda: nv.nvfp4_gemm(A[Kk], Wt, o, None, stream, gws), 5)
            res[name] = {"us": us, "TFLOP/s": 2 * T * Wt.rows * Kk / us / 1e6}
        s_t = nv.NVFP4Tensor.empty(T, I, dev)
        g_i = torch.tensor([0.01], dtype=torch.float32, device=dev)
        sws = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_STATIC), dev)
        us = timed(lambda: nv.nvfp4_gemm_swiglu(A[H], W["gate"], W["up"], nv.NVFP4_INTER_STATIC, g_i, s_t, sws,
                                                None, stream), 5)
        res["gate_up_swiglu"] = {"us": us, "TFLOP/s": 2 * T * 2 * I * H / us / 1e6}
        for v in res.values():
            v["frac_of_fp4_peak"] = v["TFLOP/s"] / fp4_peak
        out[f"gemm_T{T}"] = res
        del A
    assert nv.device_status() == 0
    return out


# ------------------------------------------------ the other workloads
def graph_time_us(fn, stream, n, reps=3):
    """Mean device time of fn() over n launches captured in one CUDA graph
    (best of `reps` replays, after one warm replay)."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            fn()
    best = None
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e3 / n
            best = t if best is None else min(best, t)
    return best


def mlp_weight_bytes(h=H, i=I):
    n = 3 * i * h
    return n // 2 + n // 16


def oracle_mlp_rate(T_list, budget_s=4.0):
    """Oracle MLP tokens/s on the host cores (configs 2 and 5): each T with
    T <= 17 timed in full; larger T extrapolated linearly from the T=17
    per-token time (every MLP step after the two global scales is per token)."""
    import oracle
    oracle.build()
    w = synthetic.mlp_weights(0, zero_block_frac=0.01)
    q = {}
    for k in ("gate", "up", "down"):
        g = oracle.global_scale(w["w_" + k])
        c, sf = oracle.quantize(w["w_" + k], g)
        q[k] = (c, sf, g)
    out = {}
    per_token = None
    for T in T_list:
        if T <= 17:
            x = synthetic.activations(T, seed=4, outliers=True)
            t0 = time.perf_counter()
            oracle.mlp(x, w["mlp_norm"], q["gate"], q["up"], q["down"])
            el = time.perf_counter() - t0
            out[T] = {"value": T / el, "how": f"timed in full ({el:.2f} s)"}
            per_token = el / T
        else:
            out[T] = {"value": 1.0 / per_token, "how": "extrapolated linearly from the T=17 per-token time"}
    return out, oracle.num_threads()


def config_measurements(nv, W, blk_factory, stream, hbm_gbs, fp4_peak):
    """Configs other than the headline one, each on its own workload and
    reported with its roofline bound; timed as CUDA graphs of the launch
    sets (device time, inputs resident)."""
    dev = W["o"].codes.device
    res = {}
    # config 1: the single NVFP4 linear (16 x 512 x 256): latency-bound
    a_bits, w_bits = synthetic.single_linear(16, 512, 256, seed=0)
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    ws = nv.workspace(256, dev)
    A1, W1 = nv.quantize_new(to_dev(a_bits), ws), nv.quantize_new(to_dev(w_bits), ws)
    o1 = torch.empty((16, 512), dtype=torch.bfloat16, device=dev)
    us = graph_time_us(lambda: nv.nvfp4_gemm(A1, W1, o1, None, stream), stream, 200)
    res["cfg1_single_linear_16x512x256"] = {"us_per_gemm": us, "TFLOP/s": 2 * 16 * 512 * 256 / us / 1e6,
                                            "bound": "launch latency"}
    # config 2: the decode MLP (T=1) as a graph; two layers' weights
    # alternate so that each call streams its weights (300 MB > L2)
    wb = {}
    for layer in (0, 1):
        m = synthetic.mlp_weights(layer)
        wb[layer] = {k: nv.quantize_new(to_dev(m["w_" + k]), ws) for k in ("gate", "up", "down")}
        wb[layer]["norm"] = to_dev(m["mlp_norm"])
    x = to_dev(synthetic.activations(1, seed=1))
    y = torch.empty_like(x)
    gi = {l: torch.zeros(1, dtype=torch.float32, device=dev) for l in (0, 1)}
    mws = nv.workspace(nv.mlp_workspace_bytes(1, H, I, nv.NVFP4_INTER_DYNAMIC), dev)
    with torch.cuda.stream(stream):
        for l in (0, 1):
            nv.nvfp4_mlp(x, wb[l]["norm"], wb[l]["gate"], wb[l]["up"], wb[l]["down"], nv.NVFP4_INTER_DYNAMIC, gi[l],
                         y, mws, True, 1e-6, stream)

    def two_layers():
        for l in (0, 1):
            nv.nvfp4_mlp(x, wb[l]["norm"], wb[l]["gate"], wb[l]["up"], wb[l]["down"], nv.NVFP4_INTER_STATIC, gi[l],
                         y, mws, True, 1e-6, stream)
    us2 = graph_time_us(two_layers, stream, 50) / 2
    wbytes = mlp_weight_bytes()
    res["cfg2_decode_mlp_T1"] = {"us_per_mlp": us2, "tokens_per_s_per_layer": 1e6 / us2,
                                 "weight_GB/s": wbytes / us2 / 1e3, "frac_of_hbm": wbytes / us2 / 1e3 / hbm_gbs,
                                 "bound": "hbm", "launches": "3 per MLP, CUDA graph",
                                 "weights": "two layers alternate (300 MB > L2)"}
    del wb
    # config 5: MLP T sweep, Student-t(3) activations with 0.1% of channels
    # x100, weights with 1% all-zero blocks
    m = synthetic.mlp_weights(0, zero_block_frac=0.01)
    wz = {k: nv.quantize_new(to_dev(m["w_" + k]), ws) for k in ("gate", "up", "down")}
    nz = to_dev(m["mlp_norm"])
    sweep = {}
    for T in (1, 3, 17, 128, 777, 4096, 8192):
        xt = to_dev(synthetic.activations(T, seed=4, outliers=True))
        yt = torch.empty_like(xt)
        g5 = torch.zeros(1, dtype=torch.float32, device=dev)
        w5 = nv.workspace(nv.mlp_workspace_bytes(T, H, I, nv.NVFP4_INTER_DYNAMIC), dev)
        with torch.cuda.stream(stream):
            nv.nvfp4_mlp(xt, nz, wz["gate"], wz["up"], wz["down"], nv.NVFP4_INTER_DYNAMIC, g5, yt, w5, True, 1e-6,
                         stream)
        n = max(2, min(50, int(2e4 / max(T, 1) ** 0.8)))
        us5 = graph_time_us(lambda: nv.nvfp4_mlp(xt, nz, wz["gate"], wz["up"], wz["down"], nv.NVFP4_INTER_STATIC,
                                                 g5, yt, w5, True, 1e-6, stream), stream, n)
        flops = 2 * T * 3 * I * H
        nbytes = wbytes + 45824 * T
        t_roof = max(flops / (fp4_peak * 1e12), nbytes / (hbm_gbs * 1e9)) * 1e6
        sweep[T] = {"us": us5, "tokens_per_s": T / us5 * 1e6, "TFLOP/s": flops / us5 / 1e6,
                    "GB/s": nbytes / us5 / 1e3,
                    "bound": "tensor" if flops / (fp4_peak * 1e12) > nbytes / (hbm_gbs * 1e9) else "hbm",
                    "frac_of_roofline": t_roof / us5}
        del xt, yt, w5
    res["cfg5_mlp_T_sweep_outliers_zero_blocks"] = sweep
    del wz
    # the routed-expert projection (next row: grouped GEMM for MoE experts):
    # T=1024 tokens, top-4 of 64 experts, each expert 1536 x 5120, skewed
    # routing (half of the tokens send a slot to expert 0); HBM-bound (the
    # experts' 283 MB of weights stream once)
    Tm, topk, E, Nm = EXPERTS_SHAPE
    ax, wx, ids, ox, wsx = experts_inputs(nv, dev, ws)
    usx = graph_time_us(lambda: nv.nvfp4_gemm_experts(ax, wx, E, ids, ox, wsx, stream), stream, 20)
    xbytes = E * Nm * H * 9 // 16
    res["experts_T1024_top4_of_64_N1536_K5120"] = {
        "us": usx, "TFLOP/s": 2 * Tm * topk * Nm * H / usx / 1e6, "weight_GB/s": xbytes / usx / 1e3,
        "frac_of_hbm": xbytes / usx / 1e3 / hbm_gbs, "bound": "hbm", "launches": 3}
    del wx, ax, ox, wsx
    # config 4: T=16384 as 16 ubatches of 1024 through 8 stacked layers, ONE
    # graph (capture fails on any host synchronisation: 0 per layer)
    L, U, T = 8, 16, 1024
    blocks = [blk_factory(layer) for layer in range(L)]
    xs = [to_dev(synthetic.activations(T, seed=3 + 1000 * u)) for u in range(U)]
    bufs = [[torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)] for _ in range(U)]
    with torch.cuda.stream(stream):
        for b in blocks:
            b.calibrate(xs[0], bufs[0][0], stream)

    def all_layers():
        for u in range(U):
            inp = xs[u]
            for layer in range(L):
                out = bufs[u][layer % 2]
                blocks[layer].forward(inp, out, stream)
                inp = out
    us4 = graph_time_us(all_layers, stream, 1, reps=3)
    res["cfg4_long_prefill_T16384_8_layers"] = {
        "ms_per_pass": us4 / 1e3, "tokens_per_s": U * T / us4 * 1e6,
        "layer_tokens_per_s": L * U * T / us4 * 1e6, "TFLOP/s": L * U * block_flops(T) / us4 / 1e6,
        "frac_of_fp4_peak": L * U * block_flops(T) / us4 / 1e6 / fp4_peak,
        "host_syncs_per_layer": 0, "launches_per_pass": L * U * PrefillBlockLaunches(),
        "how": "16 ubatches x 8 layers (seeded weights per layer) captured as one CUDA graph; a host "
               "synchronisation anywhere in the launch set would fail the capture"}
    del blocks, xs, bufs
    torch.cuda.empty_cache()
    return res


def PrefillBlockLaunches():
    from nvfp4_block_scaled_device_gb300.block import PrefillBlock
    return PrefillBlock.LAUNCHES_PER_FORWARD


# ------------------------------------------------ decode-kernel timeline
def decode_timeline(nv, W, dev):
    """Per-CTA timeline of the tensor-core decode GEMM at T=1 (QKV, O, down),
    one cold launch each (L2 flushed, weights from HBM), from a library
    built with the kernel's debug timeline (-DNVFP4_TRACE_DECODE; the
    product library carries none of it).  Prints one JSON line per GEMM:
    medians / maxima over the CTAs of the time (us from the first CTA's
    entry) each reached a point, and per-CTA stall totals (us)."""
    import ctypes
    from nvfp4_block_scaled_device_gb300.build import build, PKG
    path = build(extra_flags=["-DNVFP4_TRACE_DECODE"], out=os.path.join(PKG, "_build", "libnvfp4_trace.so"))
    L = nv.lib(path)
    L.nvfp4_debug_decode_trace.argtypes = [ctypes.c_void_p]
    L.nvfp4_debug_decode_trace_clear.argtypes = []
    nv._lib = L
    names = ["entry", "setup_done", "first_stage_full", "last_segment_issued", "first_acc_full", "last_ticket",
             "block_done", "exit"]
    stalls = ["producer_wait_slot", "mma_wait_data", "mma_wait_acc", "epilogue_busy", "epi_store", "epi_ticket",
              "epi_combine", "epi_block"]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    gws = nv.workspace(nv.gemm_workspace_bytes(), dev)
    ws = nv.workspace(256, dev)
    A = {k: nv.NVFP4Tensor.empty(1, k, dev) for k in (H, I)}
    for k, a in A.items():
        nv.nvfp4_scale_quantize(torch.randn((1, k), device=dev).bfloat16(), a, ws, None, 1e-6, None)
    for name, Kk in (("qkv", H), ("o", H), ("down", I)):
        o = torch.empty((1, W[name].rows), dtype=torch.bfloat16, device=dev)
        for rep in range(3):
            flush.fill_(rep)
            torch.cuda.synchronize()
            assert L.nvfp4_debug_decode_trace_clear() == 0
            nv.nvfp4_gemm(A[Kk], W[name], o, None, None, gws)
            torch.cuda.synchronize()
        buf = (ctypes.c_ulonglong * (256 * 16))()
        assert L.nvfp4_debug_decode_trace(buf) == 0
        t = np.array(buf, dtype=np.int64).reshape(256, 16)[:torch.cuda.get_device_properties(dev).multi_processor_count]
        t0 = t[:, 0].min()
        rec = {"gemm": name, "T": 1, "weight_MB": (W[name].codes.numel() + W[name].sf.numel()) / 1e6}
        for k, n in enumerate(names):
            col = (t[:, k][t[:, k] >= t0] - t0) / 1e3
            rec[n] = {"med": round(float(np.median(col)), 2), "max": round(float(col.max()), 2)} if len(col) else None
        for k, n in enumerate(stalls):
            col = t[:, 8 + k] / 1e3
            rec["stall_" + n] = {"med": round(float(np.median(col)), 2), "max": round(float(col.max()), 2)}
        print(json.dumps(rec), flush=True)
    assert nv.device_status() == 0


# routed-expert projection: tokens, experts per token, experts, expert rows
EXPERTS_SHAPE = (1024, 4, 64, 1536)


def experts_inputs(nv, dev, ws):
    """Inputs of the expert-indexed GEMM measurement: T=1024 quantized
    token rows, 64 experts of 1536 x 5120 NVFP4 weights, top-4 routing ids
    with half of the tokens sending their first slot to expert 0."""
    Tm, topk, E, Nm = EXPERTS_SHAPE
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    rng = np.random.default_rng(8)
    wx = nv.quantize_new(to_dev(synthetic.normal(rng, (E * Nm, H), std=0.02)), ws)
    gx = torch.cat([nv.quantize_new(to_dev(synthetic.normal(rng, (Nm, H), std=0.02)), ws).g for _ in range(E)])
    wx.g = gx                                           # per-expert global scales (values immaterial to timing)
    ax = nv.quantize_new(to_dev(synthetic.activations(Tm, seed=9)), ws)
    ids = np.stack([rng.choice(E, size=topk, replace=False) for _ in range(Tm)]).astype(np.int32)
    ids[rng.random(Tm) < 0.5, 0] = 0
    ids = torch.from_numpy(ids).to(dev)
    ox = torch.empty((Tm * topk, Nm), dtype=torch.bfloat16, device=dev)
    wsx = nv.workspace(nv.experts_workspace_bytes(Tm, topk, H, E), dev)
    return ax, wx, ids, ox, wsx


def experts_only(nv, dev, reps):
    """Profiling target: the expert-indexed GEMM (three launches per call)
    on the inputs of experts_inputs, `reps` calls after one untimed call;
    prints the mean call time from CUDA events."""
    E = EXPERTS_SHAPE[2]
    ws = nv.workspace(256, dev)
    ax, wx, ids, ox, wsx = experts_inputs(nv, dev, ws)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        nv.nvfp4_gemm_experts(ax, wx, E, ids, ox, wsx, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            nv.nvfp4_gemm_experts(ax, wx, E, ids, ox, wsx, stream)
        e1.record(stream)
    stream.synchronize()
    assert nv.device_status() == 0
    log(f"[bench] expert-indexed GEMM: {e0.elapsed_time(e1) / reps * 1e3:.1f} us per call (eager), {reps} calls")


def row_kernel_only(nv, dev, norm, reps):
    """Profiling target: the one-launch scale + quantize (with the RMSNorm
    when norm) at R=16384 x K=5120, `reps` launches on one stream after one
    untimed launch; prints the mean launch time from CUDA events (a time
    taken under a profiler is not a measurement)."""
    R, K = 16384, H
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    x = torch.randn((R, K), generator=gen, device=dev).bfloat16()
    w = (1 + 0.05 * torch.randn((K,), generator=gen, device=dev)).bfloat16() if norm else None
    t = nv.NVFP4Tensor.empty(R, K, dev)
    ws = nv.workspace(256, dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        nv.nvfp4_scale_quantize(x, t, ws, w, 1e-6, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            nv.nvfp4_scale_quantize(x, t, ws, w, 1e-6, stream)
        e1.record(stream)
    stream.synchronize()
    assert nv.device_status() == 0
    us = e0.elapsed_time(e1) / reps * 1e3
    alg = 2 * R * K + 0.5625 * R * K
    log(f"[bench] scale_quantize R={R} K={K} norm={norm}: {us:.1f} us per launch, {alg / us / 1e3:.0f} GB/s "
        f"(algorithmic bytes), {reps} launches")


# ----------------------------------------------------------- GPU (ours)
def run_ours(args):
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as nv
    from nvfp4_block_scaled_device_gb300.block import HostPipeline, PrefillBlock

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    T = args.T
    if args.only in ("quantize_R16384", "norm_quantize_R16384"):
        row_kernel_only(nv, dev, args.only.startswith("norm"), args.only_reps)
        return
    if args.only == "experts":
        experts_only(nv, dev, args.only_reps)
        return

    t_in = time.perf_counter()
    wbits, x_bits = make_inputs(T)
    to_dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(dev)
    ws = nv.workspace(256, dev)
    W = {}
    for k, name in (("qkv", "w_qkv"), ("o", "w_o"), ("gate", "w_gate"), ("up", "w_up"), ("down", "w_down")):
        W[k] = nv.quantize_new(to_dev(wbits[name]), ws)      # cold path: once, untimed
    blk = PrefillBlock(T, W, to_dev(wbits["attn_norm"]), to_dev(wbits["mlp_norm"]))
    x = to_dev(x_bits)
    out = torch.empty_like(x)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    log(f"[bench] inputs ready in {time.perf_counter() - t_in:.1f} s")

    with torch.cuda.stream(stream):
        blk.calibrate(x, out, stream)                       # on-device intermediate scale
        for _ in range(2):
            blk.forward(x, out, stream)
    stream.synchronize()
    assert nv.device_status() == 0

    if args.only == "decode_timeline":
        decode_timeline(nv, W, dev)
        return
    if args.only:
        # profiling target: launch one kernel of the step a few times, eagerly
        ev = {k: torch.cuda.Event(enable_timing=True) for k in PrefillBlock.EVENT_NAMES}
        with torch.cuda.stream(stream):
            blk.forward_timed(x, out, ev, stream)            # fills the decomposed MLP's buffers
            for _ in range(args.only_reps):
                if args.only == "swiglu":
                    nv.nvfp4_gemm_swiglu(blk.hm, W["gate"], W["up"], nv.NVFP4_INTER_STATIC, blk.g_inter, blk.s,
                                         blk.ws_swiglu, None, stream)
                elif args.only == "down":
                    nv.nvfp4_gemm(blk.s, W["down"], out, blk.x1, stream, blk.ws_gemm)
                elif args.only == "qkv":
                    nv.nvfp4_gemm(blk.h, W["qkv"], blk.qkv, None, stream, blk.ws_gemm)
                elif args.only == "o":
                    nv.nvfp4_gemm(blk.a, W["o"], blk.x1, x, stream, blk.ws_gemm)
                elif args.only == "norm_quantize":
                    nv.nvfp4_scale_quantize(x, blk.h, blk.ws_amax, blk.attn_norm, 1e-6, stream)
                elif args.only == "step":
                    blk.forward_timed(x, out, ev, stream)
                elif args.only == "mma_probe":
                    log(f"[bench] MMA issue rate: {nv.mma_issue_rate():.0f} MAC/clk/SM")
        stream.synchronize()
        assert nv.device_status() == 0
        log(f"[bench] --only {args.only}: {args.only_reps} launches done")
        return

    # ---- CUDA graphs: a 1-step graph (warm-up, e2e) and a U-step graph with
    # per-step timing events around each GEMM (timed region)
    try:
        ev_new = lambda: torch.cuda.Event(enable_timing=True, external=True)
        ev_new()
        external = True
    except TypeError:
        external = False
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        blk.forward(x, out, stream)
    U = min(args.steps, 50)
    while args.steps % U:
        U -= 1
    # events around the GEMMs on every EV_EVERY-th step only: event nodes
    # between the kernels of a step cost it several microseconds each
    evs = []
    gU = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gU, stream=stream):
        for u in range(U):
            if external and (u % EV_EVERY == EV_EVERY - 1 or (U < EV_EVERY and u == U - 1)):
                ev = {k: ev_new() for k in PrefillBlock.EVENT_NAMES}
                blk.forward_timed(x, out, ev, stream)
                evs.append(ev)
            else:
                blk.forward(x, out, stream)
    stream.synchronize()

    # ---- warm-up (graphs replay on the current stream: keep it `stream`)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g1.replay()
    stream.synchronize()

    # ---- timed region
    clocks = ClockSampler(local)
    time.sleep(0.2)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // U):
            gU.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    ms_total = slowest_rank_ms(e0.elapsed_time(e1), dist, dev)
    ms_step = ms_total / args.steps
    value = whole_job_rate(world, T * args.steps, ms_total)

    # per-GEMM times from the last replay's evented steps
    gemm = {}
    if evs:
        def avg(a, b):
            return statistics.mean(e[a].elapsed_time(e[b]) for e in evs) * 1e3   # us
        gemm = {"qkv_us": avg("qkv0", "qkv1"), "o_us": avg("o0", "o1"), "gate_up_swiglu_us": avg("gu0", "gu1"),
                "down_us": avg("gu1", "dn1"), "mlp_us": avg("mlp0", "dn1")}
    assert nv.device_status() == 0

    # ---- end to end through the public API with host buffers: every step
    # copies its ubatch in from pinned host memory and its output back; the
    # copies of the neighbouring steps overlap each step's compute
    # (HostPipeline: two device buffer pairs, separate copy streams)
    x_host = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).pin_memory()
    out_host = [torch.empty(x_host.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ke = max(10, min(args.steps, 200))
    pipe = HostPipeline(blk, stream)
    for i in range(4):
        pipe.submit(x_host, out_host[i % 2])
    pipe.wait()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    pipe.h2d.wait_event(s0)
    for i in range(ke):
        pipe.submit(x_host, out_host[i % 2])
    pipe.join()
    s1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = slowest_rank_ms(s0.elapsed_time(s1), dist, dev)
    e2e = {"value": whole_job_rate(world, T * ke, ms_e2e), "unit": "tokens/s", "h2d_bytes_per_step": x.numel() * 2,
           "d2h_bytes_per_step": out.numel() * 2, "steps": ke,
           "copies": "pinned host <-> device every step, overlapped with the neighbouring steps' compute"}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    hbm_gbs, bf16_burst_peak, _, _ = peaks()
    side = side_measurements(nv, W, stream, hbm_gbs, bf16_burst_peak * FP4_PER_BF16) if args.side else None
    mma_rate = nv.mma_issue_rate()
    clk_stats = clk
    configs = None
    if args.configs:
        def blk_factory(layer):
            aw = synthetic.attn_weights(layer)
            mw = synthetic.mlp_weights(layer)
            Wl = {}
            for k, name, src in (("qkv", "w_qkv", aw), ("o", "w_o", aw), ("gate", "w_gate", mw), ("up", "w_up", mw),
                                 ("down", "w_down", mw)):
                Wl[k] = nv.quantize_new(to_dev(src[name]), ws)
            return PrefillBlock(T, Wl, to_dev(aw["attn_norm"]), to_dev(mw["mlp_norm"]))
        configs = config_measurements(nv, W, blk_factory, stream, hbm_gbs, bf16_burst_peak * FP4_PER_BF16)
        assert nv.device_status() == 0

    hbm, bf16_burst, bf16_sust, src = peaks()
    # the timed region is milliseconds long: the burst figure applies
    fp4_peak = bf16_burst * FP4_PER_BF16
    fp4_sust = bf16_sust * FP4_PER_BF16
    gu_flops = 2 * T * 2 * I * H
    roofline = None
    if "gate_up_swiglu_us" in gemm:
        achieved = gu_flops / (gemm["gate_up_swiglu_us"] * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp4_peak, "traffic": recorded_traffic(),
                    "kernel": "fused gate/up GEMM + SwiGLU + FP4 requant (T=1024, N=2x17408, K=5120)",
                    "peak_source": f"{src}: bf16 burst {bf16_burst} TFLOP/s x {FP4_PER_BF16:g} (nominal FP4/BF16), "
                                   "of measured",
                    "peak_sustained": fp4_sust, "frac_of_sustained": achieved / fp4_sust}
        if mma_rate:
            sm_mhz = (clk_stats or {}).get("sm_mhz") or 2070.0
            mma_peak = 2 * mma_rate * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6 / 1e12
            roofline["mma_issue"] = {
                "mac_per_clk_per_sm": mma_rate, "sm_mhz": sm_mhz, "peak_TFLOP/s": mma_peak,
                "frac": achieved / mma_peak,
                "how": "nvfp4_mma_issue_rate: the kernels' fused K-stage block (12 scale copies + 4 MMAs of "
                       "256x256x64) issued back to back on one SM pair, operands in shared memory"}
    tflops = {}
    for k, fl in (("qkv", 2 * T * QKV * H), ("o", 2 * T * H * H), ("gate_up_swiglu", gu_flops),
                  ("down", 2 * T * H * I)):
        if f"{k}_us" in gemm:
            tflops[k] = fl / (gemm[f"{k}_us"] * 1e-6) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x ue4m3/16 x fp32) with fp32 accumulate, bf16 activations",
        "data": "synthetic (seeded numpy PCG64; weights ~N(0,0.02), activations ~N(0,1))",
        "config": {"workload": "prefill layer block, T=1024 ubatch: RMSNorm+QKV(7168x5120)+O(5120x5120)"
                               "+MLP(5120->2x17408->5120), NVFP4 W4A4, H=5120",
                   "T": T, "H": H, "I": I, "qkv": QKV, "launch": "CUDA graph (7 kernels/step)",
                   "gemm_timing": f"CUDA events around each GEMM on every {EV_EVERY}th step of the timed graph",
                   "intermediate_scale": "static, set by one on-device calibration ubatch",
                   "l2": f"weights {weight_bytes() / 2**20:.0f} MiB > {L2_BYTES / 2**20:.0f} MiB L2 "
                         "(inputs larger than L2, no flush)",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": PrefillBlock.LAUNCHES_PER_FORWARD * args.steps,
        "mlp_tokens_per_s": T / (gemm["mlp_us"] * 1e-6) if "mlp_us" in gemm else None,
        "gemm_tflops": tflops,
        "block_tflops": block_flops(T) / (ms_step * 1e-3) / 1e12,
        "fp4_peak_tflops": fp4_peak,
        "roofline": roofline,
        "e2e": e2e,
        "side": side,
        "configs": configs,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wbits, x_bits, T)
        if configs:
            T_list = sorted(configs["cfg5_mlp_T_sweep_outliers_zero_blocks"])
            rates, cores = oracle_mlp_rate(T_list)
            for Tk in T_list:
                configs["cfg5_mlp_T_sweep_outliers_zero_blocks"][Tk]["oracle_tokens_per_s"] = rates[Tk]
            configs["cfg2_decode_mlp_T1"]["oracle_tokens_per_s"] = rates[1]
            configs["cfg4_long_prefill_T16384_8_layers"]["oracle_tokens_per_s"] = {
                "value": line["cpu_baseline"]["value"] / 8,
                "how": "extrapolated: the oracle's per-token block rate over one layer (cpu_baseline) / 8 layers"}
            configs["oracle_cores"] = cores
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--T", type=int, default=T_DEFAULT)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", dest="side", action="store_false",
                    help="skip the side measurements (quantize at R=16384, GEMMs at T=1 and T=16384)")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the other workloads (single linear, decode MLP, T sweep, 8-layer long prefill)")
    ap.add_argument("--only", choices=("swiglu", "down", "qkv", "o", "norm_quantize", "step", "mma_probe",
                                       "decode_timeline", "quantize_R16384", "norm_quantize_R16384", "experts"),
                    help="profiling target: run one kernel of the step --only-reps times and exit "
                         "(decode_timeline: the T=1 decode GEMMs' per-CTA timeline from a debug build)")
    ap.add_argument("--only-reps", type=int, default=3)
    args = ap.parse_args()
    assert args.warmup >= 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
