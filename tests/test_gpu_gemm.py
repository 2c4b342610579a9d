"""GPU parity of the tcgen05 block-scaled GEMM against the oracle's exact
(int64) dot products.  The GPU quantizes the operands itself; each test first
asserts those operands are bit-identical to the oracle's own quantization of
the same bf16 inputs, then compares the GEMM output within the tolerance
(rel. Frobenius <= 5e-3; |err| <= 2^-7 |ref| + 1e-3 sum|a w|)."""
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


@pytest.fixture()
def ws(nv):
    return nv.workspace(256)


def run_case(nv, ws, M, N, K, seed, residual=False, a_outliers=False, split=False):
    rng = np.random.default_rng(seed)
    if a_outliers:
        a = synthetic.student_t_outliers(rng, (M, K))
    else:
        a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(A, ac, asf, ga, "A")
    assert_same_quant(W, wc, wsf, gw, "W")
    res_bits = synthetic.normal(rng, (M, N)) if residual else None
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    gws = nv.workspace(nv.gemm_workspace_bytes()) if split else None
    nv.nvfp4_gemm(A, W, out, residual=None if res_bits is None else dev(res_bits), workspace=gws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ref, absref, out_bits = oracle.gemm(ac, asf, ga, wc, wsf, gw, residual=res_bits)
    got = f64(host(out))
    if residual:
        ref = ref + f64(res_bits)
    return got, ref, absref


def test_single_linear_16x512x256(nv, ws):
    """A 16x256 ~N(0,1), W 512x256 ~N(0,0.02), seed 0 (one stream)."""
    a, w = synthetic.single_linear(16, 512, 256, seed=0)
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(A, ac, asf, ga, "A")
    assert_same_quant(W, wc, wsf, gw, "W")
    out = torch.empty((16, 512), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(A, W, out)
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)
    check_close(f64(host(out)), ref, absref, "16x512x256")


@pytest.mark.parametrize("M,N,K", [
    (1, 256, 64), (3, 512, 192), (17, 384, 320), (128, 256, 256), (130, 512, 512),
    (16, 16, 256), (200, 1024, 1024), (777, 512, 5120), (64, 768, 17408 // 4),
])
def test_ragged_shapes(nv, ws, M, N, K):
    got, ref, absref = run_case(nv, ws, M, N, K, seed=M + N + K)
    check_close(got, ref, absref, f"{M}x{N}x{K}")


def test_residual_add(nv, ws):
    got, ref, absref = run_case(nv, ws, 33, 512, 256, seed=5, residual=True)
    check_close(got, ref, absref + np.abs(ref) * 0, "residual")


def test_residual_in_place(nv, ws):
    rng = np.random.default_rng(6)
    a = synthetic.normal(rng, (40, 256))
    w = synthetic.normal(rng, (256, 256), std=0.02)
    r = synthetic.normal(rng, (40, 256))
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    buf = dev(r)
    nv.nvfp4_gemm(A, W, buf, residual=buf)
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)
    check_close(f64(host(buf)), ref + f64(r), absref, "in-place residual")


def test_outlier_activations(nv, ws):
    got, ref, absref = run_case(nv, ws, 64, 512, 5120, seed=11, a_outliers=True)
    check_close(got, ref, absref, "outliers")


def test_deterministic(nv, ws):
    rng = np.random.default_rng(12)
    A = quantize_gpu(synthetic.normal(rng, (300, 1024)), ws)
    W = quantize_gpu(synthetic.normal(rng, (768, 1024), std=0.02), ws)
    o1 = torch.empty((300, 768), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    nv.nvfp4_gemm(A, W, o1)
    nv.nvfp4_gemm(A, W, o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("M,N,K", [(1024, 7168, 5120), (1024, 5120, 5120), (1024, 5120, 17408), (1, 5120, 17408)])
@pytest.mark.parametrize("split", [False, True])
def test_full_size_sampled(nv, ws, M, N, K, split):
    """Full projection sizes of the 27B-class model (QKV, O, down): quantized
    operands compared in full, GEMM outputs on 2048 sampled elements; with and
    without the workspace that lets the GEMM split tiles over all SMs."""
    rng = np.random.default_rng(M + N)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(A, W, out, workspace=nv.workspace(nv.gemm_workspace_bytes()) if split else None)
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(A, ac, asf, ga, "A")
    assert_same_quant(W, wc, wsf, gw, "W")
    m = rng.integers(0, M, 2048)
    n = rng.integers(0, N, 2048)
    # always include the last row / column tiles
    m[:8] = M - 1
    n[8:16] = N - 1
    dot, adot = oracle.dot_sampled(ac, asf, wc, wsf, m, n)
    alpha = float(np.float32(np.float32(ga) * np.float32(gw)))
    got = f64(host(out))[m, n]
    check_close(got, alpha * dot, alpha * adot, f"{M}x{N}x{K} sampled")


# Split schedule: the tiles' K ranges spread over the SMs, fp32 partials
# combined through the workspace.  Deep-K shapes whose tiles leave most SMs
# idle (so the split is taken), including a ragged M, a K with a partial
# last stage (K = 8384: 32 full stages of 256 + 192), and tiles with only a
# few valid rows (M = 1, 3, 131), whose finishers stage their contributors'
# partial slots in shared memory (up to 6 contributors per tile).  (M = 1
# with weights above 32 MiB: smaller ones go to the decode kernel.)
@pytest.mark.parametrize("M,N,K", [(777, 512, 8192), (300, 1024, 8192), (300, 768, 8384), (1, 5120, 16384),
                                   (3, 1024, 16384), (131, 1024, 8192)])
def test_split_schedule(nv, ws, M, N, K):
    got, ref, absref = run_case(nv, ws, M, N, K, seed=M + 7 * N + K, split=True)
    check_close(got, ref, absref, f"{M}x{N}x{K} split")


# Shallow-K shapes with a partial last wave, called with a split workspace
# (which the launcher leaves unused for them): residual epilogue, ragged M,
# a K that ends in a partial stage (K = 2112: 8 stages of 256 + 64), tiles
# with few valid rows.
@pytest.mark.parametrize("M,N,K", [(1024, 5120, 5120), (128, 7168, 5120), (300, 2560, 2048), (130, 1024, 2112),
                                   (3, 7168, 5120)])
def test_partial_wave_with_workspace(nv, ws, M, N, K):
    got, ref, absref = run_case(nv, ws, M, N, K, seed=M + 5 * N + K, residual=True, split=True)
    check_close(got, ref, absref, f"{M}x{N}x{K} partial wave")


def test_split_residual_and_repeat(nv, ws):
    """Residual add through the split schedule; two calls on one workspace
    (its ready flags return to zero) give identical outputs, and these agree
    with the unsplit schedule within the GEMM tolerance."""
    rng = np.random.default_rng(21)
    M, N, K = 300, 1024, 8192
    A = quantize_gpu(synthetic.normal(rng, (M, K)), ws)
    W = quantize_gpu(synthetic.normal(rng, (N, K), std=0.02), ws)
    r = dev(synthetic.normal(rng, (M, N)))
    gws = nv.workspace(nv.gemm_workspace_bytes())
    o1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    o2, o3 = torch.empty_like(o1), torch.empty_like(o1)
    nv.nvfp4_gemm(A, W, o1, residual=r, workspace=gws)
    nv.nvfp4_gemm(A, W, o2, residual=r, workspace=gws)
    nv.nvfp4_gemm(A, W, o3, residual=r)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert torch.equal(o1, o2)
    assert int(gws[:8192].count_nonzero()) == 0          # flags back to zero
    d = (o1.double() - o3.double()).abs()
    assert float(d.max()) <= 2 ** -7 * float(o3.double().abs().max()) + 1e-2


# SM-pair kernel (256 x 256 tiles on two SMs, taken when its tiles fill a
# wave of SM pairs): ragged M (the last pair tile partly or wholly past M in
# one CTA of the pair), K with a partial last stage, residual epilogue;
# outputs compared on 4096 sampled elements, always including the last rows
# and columns.
@pytest.mark.parametrize("M,N,K", [(777, 10240, 320), (300, 19456, 576), (1023, 9728, 1088)])
def test_pair_kernel_ragged_sampled(nv, ws, M, N, K):
    rng = np.random.default_rng(M * 3 + N + K)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    r = synthetic.normal(rng, (M, N))
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(A, W, out, residual=dev(r))
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    assert_same_quant(A, ac, asf, ga, "A")
    assert_same_quant(W, wc, wsf, gw, "W")
    m = rng.integers(0, M, 4096)
    n = rng.integers(0, N, 4096)
    m[:16] = M - 1
    n[16:32] = N - 1
    m[32:48] = M - 1 - np.arange(16)      # rows of the last 128-row half tile
    dot, adot = oracle.dot_sampled(ac, asf, wc, wsf, m, n)
    alpha = float(np.float32(np.float32(ga) * np.float32(gw)))
    got = f64(host(out))[m, n]
    check_close(got, alpha * dot + f64(r)[m, n], alpha * adot, f"{M}x{N}x{K} pair sampled")


# Split schedule on SM pairs: deep K (>= 32 stages) with a partial last wave
# of pair tiles, so the pairs share the (tile, K stage) units; ragged M, a K
# with a partial last stage (K = 8384: 32 full stages of 256 + 192), residual;
# two calls on one workspace agree bit for bit and leave its flags zero.
@pytest.mark.parametrize("M,N,K", [(777, 5120, 8384), (1024, 5120, 17408)])
def test_pair_split_sampled(nv, ws, M, N, K):
    rng = np.random.default_rng(M + 11 * N + K)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    r = synthetic.normal(rng, (M, N))
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    gws = nv.workspace(nv.gemm_workspace_bytes())
    o1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    nv.nvfp4_gemm(A, W, o1, residual=dev(r), workspace=gws)
    nv.nvfp4_gemm(A, W, o2, residual=dev(r), workspace=gws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    assert torch.equal(o1, o2)
    assert int(gws[:8192].count_nonzero()) == 0
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    m = rng.integers(0, M, 4096)
    n = rng.integers(0, N, 4096)
    m[:16] = M - 1
    n[16:32] = N - 1
    dot, adot = oracle.dot_sampled(ac, asf, wc, wsf, m, n)
    alpha = float(np.float32(np.float32(ga) * np.float32(gw)))
    got = f64(host(o1))[m, n]
    check_close(got, alpha * dot + f64(r)[m, n], alpha * adot, f"{M}x{N}x{K} pair split sampled")


# The residual epilogue, bit for bit: with a residual r the output is
# bf16_RNE(float(r) + float(y)), y the same GEMM's output without one
# (R8's residual step).  y comes from the kernel itself, so the check pins
# the epilogue's arithmetic exactly on every path that has one: the 1-SM
# kernel with whole tiles and with two tiles on some CTAs (its staged
# stores), the pair kernel's whole tiles (80 tiles on 76 pairs: staged
# stores on the four pairs with two tiles and on the last tiles), the split
# schedule on SM pairs and on single SMs (few rows: the finisher stages its
# contributors' partial rows in shared memory), and the decode kernels.
EPI_CASES = [(33, 512, 256, False), (100, 40960, 256, False), (1024, 5120, 5120, False),
             (1024, 5120, 17408, True), (17, 5120, 17408, True), (100, 5120, 17408, True),
             (4, 5120, 5120, True), (1, 5120, 5120, False)]


@pytest.mark.parametrize("M,N,K,with_ws", EPI_CASES)
def test_residual_epilogue_bit_exact(nv, ws, M, N, K, with_ws):
    g = torch.Generator(device="cuda")
    g.manual_seed(M + N + K)
    A = nv.quantize_new(torch.randn((M, K), generator=g, device="cuda").bfloat16(), ws)
    W = nv.quantize_new((0.02 * torch.randn((N, K), generator=g, device="cuda")).bfloat16(), ws)
    r = torch.randn((M, N), generator=g, device="cuda").bfloat16()
    gws = nv.workspace(nv.gemm_workspace_bytes()) if with_ws else None
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(y)
    nv.nvfp4_gemm(A, W, y, workspace=gws)
    nv.nvfp4_gemm(A, W, out, residual=r, workspace=gws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    want = (r.float().cpu() + y.float().cpu()).bfloat16()
    got = out.cpu()
    bad = (got.view(torch.int16) != want.view(torch.int16)).sum().item()
    assert bad == 0, f"{M}x{N}x{K}: {bad} outputs differ from bf16(r + y)"
