"""GPU parity of the GEMMs with a handful of activation rows against the
oracle.  Given the split workspace, up to 8 rows go to the tensor-core
decode kernel (stream-K over all SMs, per-block tickets; a SwiGLU GEMM
whose blocks fill the GPU to the whole-tile prefill kernel); without it,
one or two rows and weight streams up to 32 MiB go to the CUDA-core decode
kernel, the rest to the prefill kernels; the cases cover each path.  The bf16
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


PATHS = ["cuda_cores", "tensor_cores"]


def split_ws(nv, path):
    """The workspace that selects the decode path: none (CUDA-core kernel)
    or the split workspace (tensor-core decode kernel)."""
    return nv.workspace(nv.gemm_workspace_bytes()) if path == "tensor_cores" else None


def linear(nv, ws, M, N, K, seed, residual=False, pitch=0, path="cuda_cores"):
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
    nv.nvfp4_gemm(A, W, out, residual=None if r is None else dev(r), workspace=split_ws(nv, path))
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)   # ref excludes the residual
    if r is not None:
        ref = ref + f64(r)
    return f64(host(out)), ref, absref


# N = 16: one column per CTA; N = 1040, 4096: columns split unevenly over the
# SMs; K = 64, 1088, 2112: a last unit of 32, 32 and 32 valid code bytes
# (two lanes); K = 17408: 17 units per weight row
# (tensor cores: K = 64, 320, 1088, 2112 end in a stage of 1, 1, 1, 1
# K-steps; N = 16, 48, 1040 a last 128-row block of 16, 48, 16 rows; the
# SM count splits the K stages of each block unevenly)
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 2])
@pytest.mark.parametrize("N,K", [(16, 64), (48, 1088), (256, 2112), (1040, 320), (4096, 5120), (512, 17408)])
def test_decode_shapes(nv, ws, M, N, K, path):
    got, ref, absref = linear(nv, ws, M, N, K, seed=M * 7 + N + K, path=path)
    check_close(got, ref, absref, f"decode {path} {M}x{N}x{K}")


@pytest.mark.parametrize("M", [3, 5, 8])
@pytest.mark.parametrize("N,K", [(144, 192), (528, 384), (1040, 2112), (4096, 5120)])
def test_decode_tc_more_rows(nv, ws, M, N, K):
    """3 to 8 activation rows: the tensor-core decode kernel's other B columns."""
    got, ref, absref = linear(nv, ws, M, N, K, seed=M * 11 + N + K, path="tensor_cores")
    check_close(got, ref, absref, f"decode tensor_cores {M}x{N}x{K}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 2])
def test_decode_residual(nv, ws, M, path):
    got, ref, absref = linear(nv, ws, M, 768, 2048, seed=40 + M, residual=True, path=path)
    check_close(got, ref, absref, f"decode {path} residual M={M}")


@pytest.mark.parametrize("path", PATHS)
def test_decode_residual_in_place(nv, ws, path):
    M, N, K = 2, 640, 1024
    rng = np.random.default_rng(44)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    r = synthetic.normal(rng, (M, N))
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    buf = dev(r)
    nv.nvfp4_gemm(A, W, buf, residual=buf, workspace=split_ws(nv, path))
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)
    check_close(f64(host(buf)), ref + f64(r), absref, "decode residual in place")


@pytest.mark.parametrize("path", PATHS)
def test_decode_pitched_weights(nv, ws, path):
    got, ref, absref = linear(nv, ws, 2, 320, 1088, seed=45, pitch=48, path=path)
    check_close(got, ref, absref, f"decode {path} pitched W")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,N,K", [(1, 7168, 5120), (2, 5120, 5120), (2, 5120, 17408), (1, 5120, 17408)])
def test_decode_full_size(nv, ws, M, N, K, path):
    """The QKV, O and down projection sizes (without the split workspace the
    down projection runs on the prefill kernels), every output compared."""
    got, ref, absref = linear(nv, ws, M, N, K, seed=M + N + K, path=path)
    check_close(got, ref, absref, f"decode {path} full {M}x{N}x{K}")


@pytest.mark.parametrize("path", PATHS)
def test_decode_deterministic(nv, ws, path):
    """Bit-identical repeats; on the tensor-core kernel also that each call
    leaves its tickets at zero for the next (a stale ticket would leave a
    block unfinished: NaN)."""
    rng = np.random.default_rng(46)
    A = quantize_gpu(synthetic.normal(rng, (1, 17408)), ws)
    W = quantize_gpu(synthetic.normal(rng, (3584, 17408), std=0.02), ws)   # 31 MB
    wsp = split_ws(nv, path)
    outs = []
    for _ in range(3):
        o = torch.full((1, 3584), float("nan"), dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_gemm(A, W, o, workspace=wsp)
        outs.append(o)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert not torch.isnan(outs[0]).any()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    if wsp is not None:
        assert int(wsp[:8192].count_nonzero()) == 0   # tickets back at zero


def sized_ws(nv, nbytes, path):
    """A call's workspace of nbytes (its public size, split slots included:
    tensor-core decode kernel) or without the split slots (CUDA cores)."""
    if path == "cuda_cores":
        nbytes -= nv.gemm_workspace_bytes() - 8192
    return nv.workspace(nbytes)


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


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T,K,I", [(1, 5120, 2048), (2, 1088, 1024), (2, 5120, 17408)])
def test_decode_swiglu_fused_equals_dynamic(nv, ws, T, K, I, path):
    """STATIC requant (in the epilogue) with the scale a DYNAMIC call computed
    reproduces that call's codes and scales (padding rows included) bit for
    bit; the two calls' bf16 SwiGLU outputs are identical."""
    _, (A, Wg, Wu) = swiglu_inputs(nv, ws, T, K, I, seed=50 + T + K, pitch_gate=32 if K == 1088 else 0,
                                   pitch_up=96 if K == 1088 else 0)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_dyn = nv.NVFP4Tensor.empty(T, I)
    s_dyn.sf.fill_(0xAB)
    s_bf_dyn = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = sized_ws(nv, nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC), path)
    nv.nvfp4_gemm_swiglu(A, Wg, Wu, nv.NVFP4_INTER_DYNAMIC, g, s_dyn, wsd, s_bf16=s_bf_dyn)
    s_st = nv.NVFP4Tensor.empty(T, I)
    s_st.sf.fill_(0xCD)   # padding rows must be rewritten as zeros
    s_bf_st = torch.empty_like(s_bf_dyn)
    wss = sized_ws(nv, nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_STATIC), path)
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


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T,K,I", [(1, 256, 256), (2, 5120, 2048), (2, 2112, 1024), (8, 1088, 1152)])
def test_decode_swiglu_values_vs_oracle(nv, ws, T, K, I, path):
    """The bf16 SwiGLU output against the oracle's, from the oracle's exact
    gate/up GEMMs; error bound propagated from the GEMM tolerance."""
    (a, wg, wu), (A, Wg, Wu) = swiglu_inputs(nv, ws, T, K, I, seed=60 + T + K + I)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    s_out = nv.NVFP4Tensor.empty(T, I)
    s_bf = torch.empty((T, I), dtype=torch.bfloat16, device="cuda")
    wsd = sized_ws(nv, nv.swiglu_workspace_bytes(T, I, nv.NVFP4_INTER_DYNAMIC), path)
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


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("mode", ["static", "dynamic"])
def test_decode_mlp(nv, ws, mode, path):
    """The whole MLP launch set at T=2 (both GEMMs on the decode kernels)."""
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
    mws = sized_ws(nv, nv.mlp_workspace_bytes(T, H, I, m), path)
    nv.nvfp4_mlp(dev(x), dev(nw), gpu["gate"], gpu["up"], gpu["down"], m, g_inter, out, mws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    if m == nv.NVFP4_INTER_DYNAMIC:
        assert abs(g_inter.item() - g_inter_val) <= 2 ** -7 * g_inter_val
    ref, absref, _ = oracle_mlp_rows(x, np.arange(T), nw, orc, g_inter_val)
    check_close(f64(host(out)), ref, absref, f"decode mlp {mode}")
