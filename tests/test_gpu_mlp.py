"""GPU parity of the fused gate/up GEMM (SwiGLU + FP4 requant epilogue), the
down projection with residual, and the whole MLP launch set, against the
oracle.  Float outputs use the GEMM/MLP tolerance; the fused requant is also
checked bit-for-bit against the unfused path on the GPU (same scale)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from _gpu import (ELEM_ABS, ELEM_REL, assert_same_quant, check_close, dev, f64, host, oracle_mlp_rows,
                  oracle_quant, quantize_gpu)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as m
    return m


@pytest.fixture()
def ws(nv):
    return nv.workspace(256)


def make_weights(nv, ws, H, I, seed, zero_block_frac=0.0):
    rng = np.random.default_rng(seed)
    bits = {"gate": synthetic.normal(rng, (I, H), std=0.02), "up": synthetic.normal(rng, (I, H), std=0.02),
            "down": synthetic.normal(rng, (H, I), std=0.02)}
    if zero_block_frac:
        for k in bits:
            synthetic.zero_blocks(rng, bits[k], zero_block_frac)
    gpu = {k: quantize_gpu(v, ws) for k, v in bits.items()}
    orc = {k: oracle_quant(v) for k, v in bits.items()}
    for k in bits:
        assert_same_quant(gpu[k], *orc[k], what=f"W_{k}")
    return bits, gpu, orc


def test_swiglu_fused_equals_unfused(nv, ws):
    """STATIC (requant inside the GEMM epilogue) with the scale a DYNAMIC call
    computed must reproduce that call's codes and scales bit for bit."""
    T, K, I = 77, 512, 1024
    rng = np.random.default_rng(21)
    A = quantize_gpu(synthetic.normal(rng, (T, K)), ws)
    Wg = quantize_gpu(synthetic.normal(rng, (I, K), std=0.02), ws)
    Wu = quantize_gpu(synthetic.normal(rng, (I, K), std=0.02), ws)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_dyn = nv.NVFP4Tensor.empty(T, I)
    s_bf_dyn = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_DYNAMIC, g, s_dyn, wsd, s_bf16=s_bf_dyn)
    s_st = nv.NVFP4Tensor.empty(T, I)
    s_bf_st = torch.empty_like(s_bf_dyn)
    wss = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_STATIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_STATIC, g, s_st, wss, s_bf16=s_bf_st)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert torch.equal(s_bf_st, s_bf_dyn)
    assert g.item() == oracle.global_scale(host(s_bf_dyn))   # per-call scale of this s
    assert torch.equal(s_st.codes, s_dyn.codes)
    assert torch.equal(s_st.sf, s_dyn.sf)


@pytest.mark.parametrize("T,K,I", [(1, 256, 256), (33, 512, 1024), (130, 1024, 2048), (300, 5120, 512)])
def test_swiglu_values_vs_oracle(nv, ws, T, K, I):
    """The bf16 SwiGLU output against the oracle's, from the oracle's exact
    gate/up GEMMs; error bound propagated from the GEMM tolerance."""
    rng = np.random.default_rng(T + K + I)
    a = synthetic.normal(rng, (T, K))
    wg = synthetic.normal(rng, (I, K), std=0.02)
    wu = synthetic.normal(rng, (I, K), std=0.02)
    A, Wg, Wu = quantize_gpu(a, ws), quantize_gpu(wg, ws), quantize_gpu(wu, ws)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_out = nv.NVFP4Tensor.empty(T, I)
    s_bf = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_DYNAMIC, g, s_out, wsd, s_bf16=s_bf)
    ac, asf, ga = oracle_quant(a)
    gc, gsf, gg = oracle_quant(wg)
    uc, usf, gu = oracle_quant(wu)
    assert_same_quant(A, ac, asf, ga, "A")
    gref, gabs, gate = oracle.gemm(ac, asf, ga, gc, gsf, gg)
    uref, uabs, up = oracle.gemm(ac, asf, ga, uc, usf, gu)
    s_ref = f64(oracle.swiglu(gate, up))
    got = f64(host(s_bf))
    G, U = f64(gate), f64(up)
    dg = ELEM_REL * np.abs(gref) + ELEM_ABS * gabs
    du = ELEM_REL * np.abs(uref) + ELEM_ABS * uabs
    silu = G / (1 + np.exp(-G))
    bound = 1.1 * dg * (np.abs(U) + du) + np.abs(silu) * du + 2.0 ** -7 * np.abs(s_ref) + 1e-30
    bad = np.argwhere(np.abs(got - s_ref) > bound)
    assert bad.size == 0, f"{len(bad)} SwiGLU values outside the bound, first {bad[:3].tolist()}"
    rel = np.linalg.norm(got - s_ref) / np.linalg.norm(s_ref)
    assert rel <= 5e-3, rel


@pytest.mark.parametrize("T,H,I,mode", [(5, 256, 2048, "static"), (17, 512, 2048, "dynamic"),
                                        (130, 1024, 2048, "static"), (1, 5120, 2048, "static")])
def test_mlp_small_vs_oracle(nv, ws, T, H, I, mode):
    rng = np.random.default_rng(T * 3 + H)
    x = synthetic.normal(rng, (T, H))
    nw = synthetic.normal(rng, (H,), mean=1.0, std=0.05)
    bits, gpu, orc = make_weights(nv, ws, H, I, seed=H + I)
    # the intermediate scale: the oracle's per-call scale of this batch
    full = oracle.mlp(x, nw, orc["gate"], orc["up"], orc["down"], g_inter=None, add_residual=True)
    g_inter_val = full["g_inter"]
    g_inter = torch.tensor([g_inter_val], dtype=torch.float32, device="cuda")
    m = nv.NVFP4_INTER_STATIC if mode == "static" else nv.NVFP4_INTER_DYNAMIC
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    mws = nv.workspace(nv.mlp_workspace_bytes(T, H, I, m))
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], m, g_inter, out, mws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    if m == nv.NVFP4_INTER_DYNAMIC:
        # the device's per-call scale of its own SwiGLU output; the oracle's
        # from its exact GEMMs -- equal up to a rounding of the amax element
        assert abs(g_inter.item() - g_inter_val) <= 2 ** -7 * g_inter_val
    # the reference always uses the oracle's own scale (no device value feeds the oracle)
    ref, absref, _ = oracle_mlp_rows(x, np.arange(T), nw, orc, g_inter_val)
    assert np.array_equal(full["out"], oracle.mlp(x, nw, orc["gate"], orc["up"], orc["down"],
                                                  g_inter=g_inter_val)["out"])
    check_close(f64(host(out)), ref, absref, f"mlp T={T}")


@pytest.fixture(scope="module")
def big_weights(nv):
    """The 27B-class MLP shape: gate/up [17408 x 5120], down [5120 x 17408]."""
    ws = nv.workspace(256)
    w = synthetic.mlp_weights(0)
    gpu = {k: quantize_gpu(w["w_" + k], ws) for k in ("gate", "up", "down")}
    orc = {k: oracle_quant(w["w_" + k]) for k in ("gate", "up", "down")}
    for k in gpu:
        assert_same_quant(gpu[k], *orc[k], what=f"W_{k}")
    return w, gpu, orc


@pytest.mark.parametrize("T,outliers", [(1, False), (1024, False), (3, True), (777, True), (17, True), (128, True),
                                        (4096, True), (8192, False)])
def test_mlp_full_size(nv, big_weights, T, outliers):
    """Decode (T=1) and prefill-ubatch (T=1024) MLP at H=5120, I=17408, and
    the T sweep with the outlier stress (Student-t(3) with 0.1% of channels
    x100), up to T=8192 (the SM-pair kernel and its split).  STATIC
    intermediate scale fixed by the oracle on the first rows; outputs
    compared on sampled rows (every row is independent given the scales)."""
    w, gpu, orc = big_weights
    x = synthetic.activations(T, seed=4 if outliers else (1 if T == 1 else 2), outliers=outliers)
    nw = w["mlp_norm"]
    cal_rows = np.arange(min(T, 4))
    _, _, s_cal = oracle_mlp_rows(x, cal_rows, nw, orc, np.float32(1.0))
    g_inter_val = oracle.global_scale(s_cal)
    g_inter = torch.tensor([g_inter_val], dtype=torch.float32, device="cuda")
    out = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
    mws = nv.workspace(nv.mlp_workspace_bytes(T, 5120, 17408, nv.NVFP4_INTER_STATIC))
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], nv.NVFP4_INTER_STATIC, g_inter, out, mws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    rows = np.unique(np.concatenate([[0, T - 1], np.random.default_rng(T).integers(0, T, 4)]))
    ref, absref, _ = oracle_mlp_rows(x, rows, nw, orc, g_inter_val)
    check_close(f64(host(out))[rows], ref, absref, f"mlp full T={T}")
