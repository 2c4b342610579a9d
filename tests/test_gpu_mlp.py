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


def _big(nv, zero_block_frac):
    ws = nv.workspace(256)
    w = synthetic.mlp_weights(0, zero_block_frac=zero_block_frac)
    gpu = {k: quantize_gpu(w["w_" + k], ws) for k in ("gate", "up", "down")}
    orc = {k: oracle_quant(w["w_" + k]) for k in ("gate", "up", "down")}
    for k in gpu:
        assert_same_quant(gpu[k], *orc[k], what=f"W_{k}")
    return w, gpu, orc


@pytest.fixture(scope="module")
def big_weights(nv):
    """The 27B-class MLP shape: gate/up [17408 x 5120], down [5120 x 17408]."""
    return _big(nv, 0.0)


@pytest.fixture(scope="module")
def big_weights_zb(nv):
    """The same shape with 1% of the weights' 16-element blocks all zero (the
    outlier / ragged stress workload)."""
    w, gpu, orc = _big(nv, 0.01)
    assert (orc["gate"][1] == 0).any() and (orc["down"][1] == 0).any()   # zero blocks -> zero scales
    return w, gpu, orc


def pair_tile_rows(T, rng, extra=16):
    """Sampled token rows that cover both 128-row halves of the first, second
    and last 256-row pair tiles (first, middle and last rows of each half),
    plus random rows."""
    rows = []
    for t in sorted({0, 1, (T - 1) // 256}):
        for off in (0, 1, 63, 64, 126, 127, 128, 129, 191, 192, 254, 255):
            if t * 256 + off < T:
                rows.append(t * 256 + off)
    rows += [0, T - 1] + list(rng.integers(0, T, extra))
    return np.unique(np.array(rows, np.int64))


@pytest.mark.parametrize("T,outliers", [(1, False), (2, False), (8, True), (1024, False), (3, True), (777, True),
                                        (17, True), (128, True), (4096, True), (8192, False)])
def test_mlp_full_size(nv, big_weights, big_weights_zb, T, outliers):
    """Decode (T=1) and prefill-ubatch (T=1024) MLP at H=5120, I=17408, and
    the T sweep with the outlier stress (Student-t(3) with 0.1% of channels
    x100, weights with 1% zero blocks), up to T=8192 (the SM-pair kernel and
    its split).  STATIC intermediate scale fixed by the oracle on the first
    rows; outputs compared on sampled rows that cover both halves of
    several pair tiles (every row is independent given the scales)."""
    w, gpu, orc = big_weights_zb if outliers else big_weights
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
    rows = pair_tile_rows(T, np.random.default_rng(T))
    ref, absref, _ = oracle_mlp_rows(x, rows, nw, orc, g_inter_val)
    check_close(f64(host(out))[rows], ref, absref, f"mlp full T={T}")


def test_swiglu_requant_bitexact_pair_full_size(nv, big_weights):
    """The fused gate/up GEMM at the prefill ubatch shape (T=1024, K=5120,
    I=17408: SM-pair tiles) with its bf16 SwiGLU output exported.  Over the
    whole T x I output: the per-call scale (DYNAMIC) is the global scale of
    that bf16 output; the quantize kernel's codes and scales (DYNAMIC), the
    pair epilogue's fused requant (STATIC with the same scale) and a stale
    quarter scale that forces E4M3 saturation at 448 (STATIC, g/4) all equal
    the oracle's quantization of the GPU's own bf16 SwiGLU output, bit for
    bit.  The bf16 values themselves are checked against the oracle's exact
    gate/up GEMMs on rows that cover both halves of several pair tiles."""
    w, gpu, orc = big_weights
    T, K, I = 1024, 5120, 17408
    rng = np.random.default_rng(1024)
    a = synthetic.normal(rng, (T, K))
    ws = nv.workspace(256)
    A = quantize_gpu(a, ws)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_dyn = nv.NVFP4Tensor.empty(T, I)
    bf_dyn = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_gemm_swiglu(A, gpu["gate"], gpu["up"], nv.NVFP4_INTER_DYNAMIC, g, s_dyn, wsd, s_bf16=bf_dyn)
    s_st = nv.NVFP4Tensor.empty(T, I)
    bf_st = torch.empty_like(bf_dyn)
    wss = nv.workspace(nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_STATIC))
    nv.nvfp4_gemm_swiglu(A, gpu["gate"], gpu["up"], nv.NVFP4_INTER_STATIC, g, s_st, wss, s_bf16=bf_st)
    g4 = g / 4
    s_q = nv.NVFP4Tensor.empty(T, I)
    nv.nvfp4_gemm_swiglu(A, gpu["gate"], gpu["up"], nv.NVFP4_INTER_STATIC, g4, s_q, wss)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    s_bits = host(bf_dyn)
    assert torch.equal(bf_st, bf_dyn)
    g_val = np.float32(g.item())
    assert g_val == oracle.global_scale(s_bits)
    codes, sf = oracle.quantize(s_bits, g_val)
    swz = oracle.sf_swizzle(sf)
    for what, t in (("DYNAMIC (quantize kernel)", s_dyn), ("STATIC (pair epilogue)", s_st)):
        bad = np.argwhere(t.codes.cpu().numpy() != codes)
        assert bad.size == 0, f"{what}: codes differ at {bad[:4].tolist()} ({len(bad)})"
        bad = np.nonzero(t.sf.cpu().numpy() != swz)[0]
        assert bad.size == 0, f"{what}: scales differ at {bad[:4].tolist()} ({bad.size})"
    g4_val = np.float32(g4.item())
    assert g4_val == np.float32(g_val / np.float32(4))
    codes4, sf4 = oracle.quantize(s_bits, g4_val)
    assert (sf4 == 0x7E).any(), "the quarter scale must saturate some block scales at 448"
    assert np.array_equal(s_q.codes.cpu().numpy(), codes4)
    assert np.array_equal(s_q.sf.cpu().numpy(), oracle.sf_swizzle(sf4))
    # bf16 SwiGLU values on sampled rows against the oracle's exact GEMMs
    rows = pair_tile_rows(T, rng)
    ac, asf, ga = oracle_quant(a)
    assert_same_quant(A, ac, asf, ga, "A")
    gref, gabs, gate = oracle.gemm(ac[rows], asf[rows], ga, *orc["gate"])
    uref, uabs, up = oracle.gemm(ac[rows], asf[rows], ga, *orc["up"])
    s_ref = f64(oracle.swiglu(gate, up))
    got = f64(s_bits[rows])
    G, U = f64(gate), f64(up)
    dg = ELEM_REL * np.abs(gref) + ELEM_ABS * gabs
    du = ELEM_REL * np.abs(uref) + ELEM_ABS * uabs
    silu = G / (1 + np.exp(-G))
    bound = 1.1 * dg * (np.abs(U) + du) + np.abs(silu) * du + 2.0 ** -7 * np.abs(s_ref) + 1e-30
    bad = np.argwhere(np.abs(got - s_ref) > bound)
    assert bad.size == 0, f"{len(bad)} SwiGLU values outside the bound, first {bad[:3].tolist()}"


def test_mlp_full_size_dynamic_and_stale_scale(nv, big_weights_zb):
    """The outlier / ragged stress MLP at full size (H=5120, I=17408,
    zero-block weights, Student-t activations), T=256 (one row of SM-pair
    tiles):
      - DYNAMIC: the device's per-call intermediate scale against the
        oracle's over all rows (equal up to the rounding of the amax
        element), the output against the oracle on sampled rows;
      - DYNAMIC output == STATIC output with the scale it produced, bit for
        bit (the two requant paths of the full-size MLP agree);
      - STATIC with a stale quarter scale (E4M3 saturation at 448 in the
        intermediate) against the oracle taking the same quarter scale."""
    w, gpu, orc = big_weights_zb
    T, H, I = 256, 5120, 17408
    x = synthetic.activations(T, seed=44, outliers=True)
    nw = w["mlp_norm"]
    _, _, s_all = oracle_mlp_rows(x, np.arange(T), nw, orc, np.float32(1.0))
    g_oracle = oracle.global_scale(s_all)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    out_dyn = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    mws = nv.workspace(nv.mlp_workspace_bytes(T, H, I, nv.NVFP4_INTER_DYNAMIC))
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], nv.NVFP4_INTER_DYNAMIC, g, out_dyn, mws)
    g_copy = g.clone()
    out_st = torch.empty_like(out_dyn)
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], nv.NVFP4_INTER_STATIC, g_copy, out_st, mws)
    g_stale = torch.tensor([np.float32(g_oracle / np.float32(4))], dtype=torch.float32, device="cuda")
    out_q = torch.empty_like(out_dyn)
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], nv.NVFP4_INTER_STATIC, g_stale, out_q, mws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert abs(g.item() - g_oracle) <= 2 ** -7 * g_oracle
    assert torch.equal(out_dyn, out_st)
    rows = pair_tile_rows(T, np.random.default_rng(5))
    ref, absref, _ = oracle_mlp_rows(x, rows, nw, orc, g_oracle)
    check_close(f64(host(out_dyn))[rows], ref, absref, "mlp full DYNAMIC")
    gq = np.float32(g_oracle / np.float32(4))
    ref, absref, s_rows = oracle_mlp_rows(x, rows, nw, orc, gq)
    _, sf_rows = oracle.quantize(s_rows, gq)
    assert (sf_rows == 0x7E).any(), "the stale scale must saturate block scales of the sampled rows"
    check_close(f64(host(out_q))[rows], ref, absref, "mlp full stale quarter scale")
