"""GPU parity of the GEMMs with one or two activation rows against the
oracle.  Weight streams up to 32 MiB go to the decode kernel (CUDA cores),
larger ones to the tensor-core kernels; the cases cover both.  The bf16
epilogue with and without residual (in place too); ragged K whose last
1024-element unit has only a few valid lanes; column counts that split
unevenly over the SMs (down to one column per CTA); pitched weights; the
SwiGLU epilogues (FP4 requant bit-equal to the per-call-scale path, bf16
values against the oracle); the full projection sizes; the MLP launch set;
determinism."""
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


def pitched(nv, t, extra_bytes):
    """The same quantized matrix with its code rows extra_bytes further apart."""
    buf = torch.zeros((t.rows, t.cols // 2 + extra_bytes), dtype=torch.uint8, device="cuda")
    buf[:, :t.cols // 2] = t.codes
    return nv.NVFP4Tensor(codes=buf[:, :t.cols // 2], sf=t.sf, g=t.g, rows=t.rows, cols=t.cols)


def linear(nv, ws, M, N, K, seed, residual=False, pitch=0):
    rng = np.random.default_rng(seed)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(A, ac, asf, ga, "A")
    assert_same_quant(W, wc, wsf, gw, "W")
    if pitch:
        W = pitched(nv, W, pitch)
    r = synthetic.normal(rng, (M, N)) if residual else None
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(A, W, out, residual=None if r is None else dev(r))
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)   # ref excludes the residual
    if r is not None:
        ref = ref + f64(r)
    return f64(host(out)), ref, absref


# N = 16: one column per CTA; N = 1040, 4096: columns split unevenly over the
# SMs; K = 64, 1088, 2112: a last unit of 32, 32 and 32 valid code bytes
# (two lanes); K = 17408: 17 units per weight row
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(16, 64), (48, 1088), (256, 2112), (1040, 320), (4096, 5120), (512, 17408)])
def test_decode_shapes(nv, ws, M, N, K):
    got, ref, absref = linear(nv, ws, M, N, K, seed=M * 7 + N + K)
    check_close(got, ref, absref, f"decode {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2])
def test_decode_residual(nv, ws, M):
    got, ref, absref = linear(nv, ws, M, 768, 2048, seed=40 + M, residual=True)
    check_close(got, ref, absref, f"decode residual M={M}")


def test_decode_residual_in_place(nv, ws):
    M, N, K = 2, 640, 1024
    rng = np.random.default_rng(44)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    r = synthetic.normal(rng, (M, N))
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    buf = dev(r)
    nv.nvfp4_gemm(A, W, buf, residual=buf)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)
    check_close(f64(host(buf)), ref + f64(r), absref, "decode residual in place")


def test_decode_pitched_weights(nv, ws):
    got, ref, absref = linear(nv, ws, 2, 320, 1088, seed=45, pitch=48)
    check_close(got, ref, absref, "decode pitched W")


@pytest.mark.parametrize("M,N,K", [(1, 7168, 5120), (2, 5120, 5120), (2, 5120, 17408), (1, 5120, 17408)])
def test_decode_full_size(nv, ws, M, N, K):
    """The QKV, O (decode kernel) and down (tensor-core kernels) projection
    sizes, every output compared."""
    got, ref, absref = linear(nv, ws, M, N, K, seed=M + N + K)
    check_close(got, ref, absref, f"decode full {M}x{N}x{K}")


def test_decode_deterministic(nv, ws):
    rng = np.random.default_rng(46)
    A = quantize_gpu(synthetic.normal(rng, (1, 17408)), ws)
    W = quantize_gpu(synthetic.normal(rng, (3584, 17408), std=0.02), ws)   # 31 MB: the decode kernel
    o1 = torch.empty((1, 3584), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    nv.nvfp4_gemm(A, W, o1)
    nv.nvfp4_gemm(A, W, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def swiglu_inputs(nv, ws, T, K, I, seed, pitch_gate=0, pitch_up=0):
    rng = np.random.default_rng(seed)
    a = synthetic.normal(rng, (T, K))
    wg = synthetic.normal(rng, (I, K), std=0.02)
    wu = synthetic.normal(rng, (I, K), std=0.02)
    A, Wg, Wu = quantize_gpu(a, ws), quantize_gpu(wg, ws), quantize_gpu(wu, ws)
    if pitch_gate:
        Wg = pitched(nv, Wg, pitch_gate)
    if pitch_up:
        Wu = pitched(nv, Wu, pitch_up)
    return (a, wg, wu), (A, Wg, Wu)


@pytest.mark.parametrize("T,K,I", [(1, 5120, 2048), (2, 1088, 1024), (2, 5120, 17408)])
def test_decode_swiglu_fused_equals_dynamic(nv, ws, T, K, I):
    """STATIC requant (in the epilogue) with the scale a DYNAMIC call computed
    reproduces that call's codes and scales (padding rows included) bit for
    bit; the two calls' bf16 SwiGLU outputs are identical."""
    _, (A, Wg, Wu) = swiglu_inputs(nv, ws, T, K, I, seed=50 + T + K, pitch_gate=32 if K == 1088 else 0,
                                   pitch_up=96 if K == 1088 else 0)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_dyn = nv.NVFP4Tensor.empty(T, I)
    s_dyn.sf.fill_(0xAB)
    s_bf_dyn = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_DYNAMIC, g, s_dyn, wsd, s_bf16=s_bf_dyn)
    s_st = nv.NVFP4Tensor.empty(T, I)
    s_st.sf.fill_(0xCD)   # padding rows must be rewritten as zeros
    s_bf_st = torch.empty_like(s_bf_dyn)
    wss = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_STATIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_STATIC, g, s_st, wss, s_bf16=s_bf_st)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert torch.equal(s_bf_st, s_bf_dyn)
    assert g.item() == oracle.global_scale(host(s_bf_dyn))
    assert torch.equal(s_st.codes, s_dyn.codes)
    assert torch.equal(s_st.sf, s_dyn.sf)
    # and the FP4 output is the oracle's quantization of the bf16 output
    sc, ss = oracle.quantize(host(s_bf_st), np.float32(g.item()))
    assert np.array_equal(s_st.codes.cpu().numpy(), sc)
    assert np.array_equal(s_st.sf.cpu().numpy(), oracle.sf_swizzle(ss))


@pytest.mark.parametrize("T,K,I", [(1, 256, 256), (2, 5120, 2048), (2, 2112, 1024)])
def test_decode_swiglu_values_vs_oracle(nv, ws, T, K, I):
    """The bf16 SwiGLU output against the oracle's, from the oracle's exact
    gate/up GEMMs; error bound propagated from the GEMM tolerance."""
    (a, wg, wu), (A, Wg, Wu) = swiglu_inputs(nv, ws, T, K, I, seed=60 + T + K + I)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_out = nv.NVFP4Tensor.empty(T, I)
    s_bf = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_DYNAMIC, g, s_out, wsd, s_bf16=s_bf)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ac, asf, ga = oracle_quant(a)
    gc, gsf, gg = oracle_quant(wg)
    uc, usf, gu = oracle_quant(wu)
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


@pytest.mark.parametrize("mode", ["static", "dynamic"])
def test_decode_mlp(nv, ws, mode):
    """The whole MLP launch set at T=2 (both GEMMs on the decode kernel)."""
    T, H, I = 2, 1024, 3072
    rng = np.random.default_rng(70)
    x = synthetic.normal(rng, (T, H))
    nw = synthetic.normal(rng, (H,), mean=1.0, std=0.05)
    wb = {"gate": synthetic.normal(rng, (I, H), std=0.02), "up": synthetic.normal(rng, (I, H), std=0.02),
          "down": synthetic.normal(rng, (H, I), std=0.02)}
    gpu = {k: quantize_gpu(v, ws) for k, v in wb.items()}
    orc = {k: oracle_quant(v) for k, v in wb.items()}
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
        assert abs(g_inter.item() - g_inter_val) <= 2 ** -7 * g_inter_val
    ref, absref, _ = oracle_mlp_rows(x, np.arange(T), nw, orc, g_inter_val)
    check_close(f64(host(out)), ref, absref, f"decode mlp {mode}")
