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
    the block at T=1 (decode) and T=16384 (long prefill), with the block's
    weights, each timed over a few launches with CUDA events."""
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
    for T in (1, 16384):
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
        if T == 1:
            wbytes = sum(Wt.codes.numel() + Wt.sf.numel() for Wt in W.values())
            for name in res:
                Wt = {"qkv": [W["qkv"]], "o": [W["o"]], "down": [W["down"]],
                      "gate_up_swiglu": [W["gate"], W["up"]]}[name]
                b = sum(x_.codes.numel() + x_.sf.numel() for x_ in Wt)
                res[name]["weight_GB/s"] = b / res[name]["us"] / 1e3
            res["weights_MB"] = wbytes / 1e6
        out[f"gemm_T{T}"] = res
        del A
    assert nv.device_status() == 0
    return out


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
                elif args.only == "norm_quantize":
                    nv.nvfp4_scale_quantize(x, blk.h, blk.ws_amax, blk.attn_norm, 1e-6, stream)
                elif args.only == "step":
                    blk.forward_timed(x, out, ev, stream)
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
    hbm_gbs, _, bf16_sust_peak, _ = peaks()
    side = side_measurements(nv, W, stream, hbm_gbs, bf16_sust_peak * FP4_PER_BF16) if args.side else None

    hbm, bf16_burst, bf16_sust, src = peaks()
    fp4_peak = bf16_sust * FP4_PER_BF16
    gu_flops = 2 * T * 2 * I * H
    roofline = None
    if "gate_up_swiglu_us" in gemm:
        achieved = gu_flops / (gemm["gate_up_swiglu_us"] * 1e-6) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp4_peak, "traffic": recorded_traffic(),
                    "kernel": "fused gate/up GEMM + SwiGLU + FP4 requant (T=1024, N=2x17408, K=5120)",
                    "peak_source": f"{src}: bf16 sustained {bf16_sust} TFLOP/s x {FP4_PER_BF16:g} (nominal FP4/BF16)"}
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
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wbits, x_bits, T)
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
    ap.add_argument("--only", choices=("swiglu", "down", "qkv", "norm_quantize", "step"),
                    help="profiling target: run one kernel of the step --only-reps times and exit")
    ap.add_argument("--only-reps", type=int, default=3)
    args = ap.parse_args()
    assert args.warmup >= 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
