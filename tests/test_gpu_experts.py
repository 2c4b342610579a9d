"""GPU parity of the expert-indexed GEMM (nvfp4_gemm_experts: the routed
projection of a mixture-of-experts layer) against the oracle's
expert-indexed GEMM, which is pinned on the CPU by explicit fp64 sums over
an independent decode.  The GPU quantizes the activations and each
expert's weights itself; those operands are first asserted bit-identical
to the oracle's quantization, then every output row is compared within the
GEMM tolerance.  Routing tables stay on the device: the call is also
captured in a CUDA graph and replayed with new routing."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from _gpu import assert_same_quant, check_close, dev, f64, host, oracle_quant, quantize_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as m
    return m


def make_experts(nv, rng, E, N, K):
    ws = nv.workspace(256)
    gpu, orc = [], []
    for _ in range(E):
        w = synthetic.normal(rng, (N, K), std=0.02)
        t = quantize_gpu(w, ws)
        o = oracle_quant(w)
        assert_same_quant(t, *o, what="expert")
        gpu.append(t)
        orc.append(o)
    W = nv.NVFP4Tensor(codes=torch.cat([t.codes for t in gpu]), sf=torch.cat([t.sf for t in gpu]),
                       g=torch.cat([t.g for t in gpu]), rows=E * N, cols=K)
    return W, (np.stack([o[0] for o in orc]), np.stack([o[1] for o in orc]),
               np.array([o[2] for o in orc], np.float32))


def routing(rng, T, topk, E, skew):
    """ids [T, topk]: distinct experts per token; with skew, half of the
    (token, slot) pairs go to expert 0 and a quarter of the experts get none."""
    ids = np.empty((T, topk), np.int32)
    live = np.arange(E) if not skew else np.arange(E)[: max(topk + 1, 3 * E // 4)]
    for t in range(T):
        if skew and rng.random() < 0.5:
            rest = rng.choice(live[1:], size=topk - 1, replace=False) if topk > 1 else []
            ids[t] = np.concatenate([[0], rest]).astype(np.int32)
        else:
            ids[t] = rng.choice(live, size=topk, replace=False)
    return ids


def run(nv, A, W, E, ids_np, N, stream=None):
    T, topk = ids_np.shape
    ids = torch.from_numpy(ids_np).cuda()
    out = torch.full((T * topk, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = nv.workspace(nv.experts_workspace_bytes(T, topk, A.cols, E))
    nv.nvfp4_gemm_experts(A, W, E, ids, out, ws, stream)
    return out, ids, ws


@pytest.mark.parametrize("T,topk,E,N,K,skew", [(1, 1, 4, 256, 256, False), (5, 2, 8, 256, 512, False),
                                               (130, 2, 8, 512, 512, True), (300, 4, 64, 256, 1024, True),
                                               (1024, 2, 16, 1536, 512, True), (77, 8, 128, 128, 256, True),
                                               # many experts, most of them empty: the routing kernel's
                                               # prefix sum over experts spans several warps
                                               (200, 3, 1000, 128, 256, True), (40, 2, 2500, 128, 256, False)])
def test_experts_vs_oracle(nv, T, topk, E, N, K, skew):
    rng = np.random.default_rng(T * 7 + E + N + K)
    a = synthetic.normal(rng, (T, K))
    ws = nv.workspace(256)
    A = quantize_gpu(a, ws)
    ac, asf, ga = oracle_quant(a)
    assert_same_quant(A, ac, asf, ga, "A")
    W, (wc, wsf, gw) = make_experts(nv, rng, E, N, K)
    ids_np = routing(rng, T, topk, E, skew)
    out, _, _ = run(nv, A, W, E, ids_np, N)
    out2, _, _ = run(nv, A, W, E, ids_np, N)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert torch.equal(out, out2)                       # the pair order within an expert does not matter
    ref, absref, _ = oracle.gemm_id(ac, asf, ga, wc, wsf, gw, ids_np)
    got = f64(host(out)).reshape(T, topk, N)
    check_close(got, ref, absref, f"experts T={T} topk={topk} E={E} N={N} K={K}")


def test_experts_max_experts(nv):
    """E = 4096, the largest expert count: the routing kernel's prefix sum
    spans all of its threads.  The stacked weights are quantized as one
    matrix (each expert's 128 rows are whole scale tiles, so the stack's
    layout is the experts' layouts end to end), every expert carrying that
    one global scale."""
    T, topk, E, N, K = 96, 2, 4096, 128, 64
    rng = np.random.default_rng(41)
    a = synthetic.normal(rng, (T, K))
    A = quantize_gpu(a, nv.workspace(256))
    ac, asf, ga = oracle_quant(a)
    w = synthetic.normal(rng, (E * N, K), std=0.02)
    Wt = quantize_gpu(w, nv.workspace(256))
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(Wt, wc, wsf, gw, "stacked experts")
    W = nv.NVFP4Tensor(codes=Wt.codes, sf=Wt.sf, g=Wt.g.repeat(E), rows=E * N, cols=K)
    ids_np = routing(rng, T, topk, E, True)
    out, _, _ = run(nv, A, W, E, ids_np, N)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref, absref, _ = oracle.gemm_id(ac, asf, ga, wc.reshape(E, N, K // 2), wsf.reshape(E, N, K // 16),
                                    np.full(E, gw, np.float32), ids_np)
    check_close(f64(host(out)).reshape(T, topk, N), ref, absref, "experts E=4096")


def test_experts_out_of_range_id(nv):
    """An id outside [0, E) leaves its row unwritten and records a status;
    the other rows are still right."""
    T, topk, E, N, K = 9, 2, 4, 256, 256
    rng = np.random.default_rng(5)
    a = synthetic.normal(rng, (T, K))
    A = quantize_gpu(a, nv.workspace(256))
    W, (wc, wsf, gw) = make_experts(nv, rng, E, N, K)
    ids_np = routing(rng, T, topk, E, False)
    ids_np[3, 1] = E
    out, _, _ = run(nv, A, W, E, ids_np, N)
    torch.cuda.synchronize()
    assert nv.device_status() == 1 * 100 + 30
    got = host(out).reshape(T, topk, N)
    assert np.isnan(f64(got[3, 1])).all()              # untouched (NaN-filled)
    ok = np.ones((T, topk), bool)
    ok[3, 1] = False
    ids_ok = np.where(ok, ids_np, 0)
    ac, asf, ga = oracle_quant(a)
    ref, absref, _ = oracle.gemm_id(ac, asf, ga, wc, wsf, gw, ids_ok)
    check_close(f64(got)[ok], ref[ok], absref[ok], "experts with one bad id")


def test_experts_graph_replay_new_routing(nv):
    """Captured once in a CUDA graph (capture fails on any host
    synchronisation), replayed after the routing table changed on the
    device: each replay equals the eager call with that routing."""
    T, topk, E, N, K = 64, 2, 8, 256, 512
    rng = np.random.default_rng(6)
    A = quantize_gpu(synthetic.normal(rng, (T, K)), nv.workspace(256))
    W, _ = make_experts(nv, rng, E, N, K)
    r1, r2 = routing(rng, T, topk, E, True), routing(rng, T, topk, E, False)
    ids = torch.from_numpy(r1).cuda()
    out = torch.empty((T * topk, N), dtype=torch.bfloat16, device="cuda")
    ws = nv.workspace(nv.experts_workspace_bytes(T, topk, K, E))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        nv.nvfp4_gemm_experts(A, W, E, ids, out, ws, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        nv.nvfp4_gemm_experts(A, W, E, ids, out, ws, stream)
    for r in (r2, r1):
        ids.copy_(torch.from_numpy(r))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        eager, _, _ = run(nv, A, W, E, r, N)
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert nv.device_status() == 0
