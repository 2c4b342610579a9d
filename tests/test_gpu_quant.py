"""GPU parity of the device global scale, the quantizer and the RMSNorm
prologue against the CPU oracle: codes, scales and global scales must be
bit-exact (inputs from the seeded generators, expected values from the
oracle only)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from _gpu import assert_same_quant, dev, host, oracle_quant, quantize_gpu

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


SHAPES = [(1, 64), (3, 128), (16, 256), (17, 320), (128, 512), (130, 1024), (777, 5120), (1, 17408)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_quantize_bit_exact(nv, ws, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    x = synthetic.normal(rng, (rows, cols))
    t = quantize_gpu(x, ws)
    c, s, g = oracle_quant(x)
    assert_same_quant(t, c, s, g, f"{rows}x{cols}")
    assert nv.device_status() == 0


@pytest.mark.parametrize("T", [1, 3, 17, 128, 777])
def test_quantize_outliers_and_zero_blocks(nv, ws, T):
    """Student-t(3) activations with 0.1% of channels x100 (E4M3 saturation,
    device global scale) and weights with 1% all-zero blocks."""
    x = synthetic.activations(T, seed=4, outliers=True)
    t = quantize_gpu(x, ws)
    c, s, g = oracle_quant(x)
    assert_same_quant(t, c, s, g, f"outliers T={T}")
    assert (s == 0x7E).any()
    w = synthetic.weight(40 + T, 256, 5120, zero_block_frac=0.01)
    tw = quantize_gpu(w, ws)
    c, s, g = oracle_quant(w)
    assert (s == 0).sum() >= int(0.01 * s.size)
    assert_same_quant(tw, c, s, g, "zero blocks")


def test_pitched_input_and_padded_codes(nv, ws):
    rng = np.random.default_rng(3)
    big = synthetic.normal(rng, (37, 704))
    x = big[:, :640]
    xd = dev(big)[:, :640]
    t = nv.NVFP4Tensor(codes=torch.empty((37, 352), dtype=torch.uint8, device="cuda")[:, :320],
                       sf=torch.full((nv.sf_bytes(37, 640),), 0xAB, dtype=torch.uint8, device="cuda"),
                       g=torch.zeros(1, dtype=torch.float32, device="cuda"), rows=37, cols=640)
    nv.nvfp4_amax_scale(xd, t.g, ws)
    nv.nvfp4_quantize(xd, t.g, t)
    c, s, g = oracle_quant(x)
    torch.cuda.synchronize()
    assert t.g.item() == g
    assert np.array_equal(t.codes.cpu().numpy(), c)
    assert np.array_equal(t.sf.cpu().numpy(), oracle.sf_swizzle(s))   # padding overwritten with 0


def test_global_scale_special_cases(nv, ws):
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    z = torch.zeros((5, 64), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_amax_scale(z, g, ws)
    assert g.item() == oracle.global_scale(host(z))          # the 1e-8 clamp
    x = synthetic.f32_to_bf16_bits(np.array([[1.0, -5376.0] + [0.5] * 62], np.float32))
    nv.nvfp4_amax_scale(dev(x), g, ws)
    assert g.item() == 2.0
    # the workspace is left zeroed: a second call on a smaller tensor is independent
    y = synthetic.f32_to_bf16_bits(np.full((2, 64), 2688.0, np.float32))
    nv.nvfp4_amax_scale(dev(y), g, ws)
    assert g.item() == 1.0


def test_exact_roundtrip_every_scale_and_code(nv):
    """g a power of two: blocks built from (scale, codes) must come back
    exactly, for every E4M3 scale 1..126 and every code."""
    rng = np.random.default_rng(8)
    e2m1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for g in (2.0 ** -3, 1.0, 2.0 ** 5):
        rows = []
        for sc in range(1, 0x7F):
            s = oracle.e4m3_value(sc)
            codes = rng.integers(0, 16, 64)
            codes[::16] = 7
            rows.append(np.where(codes & 8, -1.0, 1.0) * e2m1[codes & 7] * s * g)
        x = synthetic.f32_to_bf16_bits(np.array(rows))
        gd = torch.tensor([g], dtype=torch.float32, device="cuda")
        t = nv.NVFP4Tensor.empty(x.shape[0], 64)
        t.g.copy_(gd)
        nv.nvfp4_quantize(dev(x), gd, t)
        c, s = oracle.quantize(x, np.float32(g))
        torch.cuda.synchronize()
        assert np.array_equal(t.codes.cpu().numpy(), c)
        assert np.array_equal(t.sf.cpu().numpy(), oracle.sf_swizzle(s))
        assert list(s[:, 0]) == list(range(1, 0x7F))


def test_ties_signed_zero_and_saturation(nv):
    """Scale 1 and g = 1 make q = x: every E2M1 midpoint, +-1 ulp around it,
    negative values rounding to zero and values beyond 6."""
    vals = []
    for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
        vals += [np.nextafter(np.float32(m), np.float32(0)), m, np.nextafter(np.float32(m), np.float32(9))]
    vals += [-0.1, -0.2, -0.25, -0.0, 0.0, 1e-20, -1e-20, 5.9, -6.0, 0.3, -0.74, 2.9, -3.6,
             4.5, -5.5, 1.0, -1.0, 0.5, -0.5, 1.5, -1.5]
    # every 16-block leads with 6.0, so its scale is exactly 1 and q = x
    blocks = [[6.0] + vals[i:i + 15] for i in range(0, len(vals), 15)]
    blocks[-1] += [0.0] * (16 - len(blocks[-1]))
    # blocks whose amax rounds the scale down (6.1875 / 6 -> 1.0): saturation at 6
    blocks.append([6.1875, -6.1875, 6.0, 5.5] + [0.0] * 12)
    vals = [v for b in blocks for v in b]
    x = synthetic.f32_to_bf16_bits(np.array(vals, np.float32).reshape(-1, 64))
    g = np.float32(1.0)
    gd = torch.tensor([g], device="cuda")
    t = nv.NVFP4Tensor.empty(x.shape[0], 64)
    nv.nvfp4_quantize(dev(x), gd, t)
    c, s = oracle.quantize(x, g)
    torch.cuda.synchronize()
    gc = t.codes.cpu().numpy()
    bad = np.argwhere(gc != c)
    assert bad.size == 0, [(int(i), int(j), int(gc[i, j]), int(c[i, j])) for i, j in bad[:8]]
    assert np.array_equal(t.sf.cpu().numpy(), oracle.sf_swizzle(s))


@pytest.mark.parametrize("T", [1, 5, 128, 1024])
def test_rmsnorm_prologue_bit_exact(nv, ws, T):
    """Batched-row RMSNorm fused with the device scale and the quantizer:
    the normalised rows, the global scale, codes and scales all match the
    oracle bit for bit."""
    x = synthetic.activations(T, seed=2)
    w = synthetic.norm_weight(17)
    y = torch.empty((T, 5120), dtype=torch.bfloat16, device="cuda")
    t = nv.NVFP4Tensor.empty(T, 5120)
    xd, wd = dev(x), dev(w)
    nv.nvfp4_amax_scale(xd, t.g, ws, norm_w=wd, eps=1e-6)
    nv.nvfp4_quantize(xd, t.g, t, norm_w=wd, eps=1e-6, y_out=y)
    y_ref = oracle.rmsnorm(x, w, 1e-6)
    torch.cuda.synchronize()
    yg = host(y)
    bad = np.argwhere(yg != y_ref)
    assert bad.size == 0, f"{len(bad)} normalised values differ, first {bad[:3].tolist()}"
    c, s, g = oracle_quant(y_ref)
    assert_same_quant(t, c, s, g, f"norm T={T}")


def test_rmsnorm_outliers(nv, ws):
    x = synthetic.activations(777, seed=4, outliers=True)
    w = synthetic.norm_weight(17)
    t = nv.quantize_new(dev(x), ws, norm_w=dev(w))
    y_ref = oracle.rmsnorm(x, w, 1e-6)
    c, s, g = oracle_quant(y_ref)
    assert_same_quant(t, c, s, g, "norm outliers")


def test_deterministic(nv, ws):
    x = synthetic.activations(300, seed=9)
    a = quantize_gpu(x, ws)
    b = quantize_gpu(x, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and torch.equal(a.sf, b.sf) and torch.equal(a.g, b.g)


# One-launch scale + quantize (cooperative kernel with a grid barrier).  The
# shapes cover the resident variant (every row held in registers by one
# block), the streaming variant (more rows than resident blocks hold, rows
# staged in shared memory: 1300 to 16384 rows of up to 5120 columns; 70000
# rows of 64 leave more rows per group than the 1 / rms stash keeps) and the
# looping variant (rows wider than the streaming slots), with and without
# the RMSNorm, up to the 16384 x 5120 input that the row-kernel bandwidth
# figure is taken on.
FUSED = [(1, 64, False), (3, 128, True), (17, 320, False), (130, 1024, True), (777, 5120, True),
         (1024, 5120, True), (1024, 5120, False), (1300, 5120, True), (5, 17408, True), (2500, 256, False),
         (4000, 5120, True), (4000, 5120, False), (6000, 256, True), (6000, 256, False), (1000, 17408, True),
         (16384, 5120, True), (16384, 5120, False), (20, 28672, True), (20, 32768, False),
         (70000, 64, True), (70000, 64, False), (3000, 5312, True), (2000, 6144, False)]


@pytest.mark.parametrize("rows,cols,norm", FUSED)
def test_scale_quantize_bit_exact(nv, ws, rows, cols, norm):
    rng = np.random.default_rng(rows * 13 + cols)
    x = synthetic.normal(rng, (rows, cols))
    w = synthetic.norm_weight(cols + 1, cols) if norm else None
    t = nv.NVFP4Tensor.empty(rows, cols)
    nv.nvfp4_scale_quantize(dev(x), t, ws, None if w is None else dev(w), 1e-6)
    v = oracle.rmsnorm(x, w, 1e-6) if norm else x
    c, s, g = oracle_quant(v)
    assert_same_quant(t, c, s, g, f"fused {rows}x{cols} norm={norm}")
    assert nv.device_status() == 0
    assert int(ws[:256].count_nonzero()) == 0         # barrier words back to zero


@pytest.mark.parametrize("norm", [True, False])
def test_scale_quantize_streaming_outliers_zero_rows(nv, ws, norm):
    """The streaming variant (more rows than the resident blocks hold):
    outlier activations (the block holding the global amax saturates the
    E4M3 scale at 448) with every 7th row all zero (its RMSNorm is zero),
    then an all-zero matrix (the 1e-8 clamp of the global scale)."""
    T = 2100
    x = synthetic.activations(T, seed=12, outliers=True).copy()
    x[::7] = 0
    w = synthetic.norm_weight(23) if norm else None
    wd = None if w is None else dev(w)
    t = nv.NVFP4Tensor.empty(T, 5120)
    nv.nvfp4_scale_quantize(dev(x), t, ws, wd, 1e-6)
    c, s, g = oracle_quant(oracle.rmsnorm(x, w, 1e-6) if norm else x)
    assert_same_quant(t, c, s, g, f"streaming outliers, zero rows, norm={norm}")
    assert (s == 0x7E).any()
    z = np.zeros((T, 5120), np.uint16)
    nv.nvfp4_scale_quantize(dev(z), t, ws, wd, 1e-6)
    c, s, g = oracle_quant(oracle.rmsnorm(z, w, 1e-6) if norm else z)
    assert_same_quant(t, c, s, g, f"streaming all zero, norm={norm}")
    assert nv.device_status() == 0


@pytest.mark.parametrize("T,norm", [(777, True), (777, False), (3, True), (3000, True), (3000, False)])
def test_scale_quantize_outliers_pitched_repeat(nv, ws, T, norm):
    """Outlier activations read through a row pitch wider than the row;
    two calls on one workspace agree bit for bit with each other, with the
    two-launch path, and with the oracle."""
    x = synthetic.activations(T, seed=6, outliers=True)
    w = synthetic.norm_weight(19) if norm else None
    wide = np.zeros((T, 5120 + 64), np.uint16)
    wide[:, :5120] = x
    xd = dev(wide)[:, :5120]
    wd = None if w is None else dev(w)
    a = nv.NVFP4Tensor.empty(T, 5120)
    b = nv.NVFP4Tensor.empty(T, 5120)
    nv.nvfp4_scale_quantize(xd, a, ws, wd, 1e-6)
    nv.nvfp4_scale_quantize(xd, b, ws, wd, 1e-6)
    two = nv.quantize_new(xd, ws, norm_w=wd)
    torch.cuda.synchronize()
    for o in (b, two):
        assert torch.equal(a.codes, o.codes) and torch.equal(a.sf, o.sf) and torch.equal(a.g, o.g)
    v = oracle.rmsnorm(x, w, 1e-6) if norm else x
    c, s, g = oracle_quant(v)
    assert_same_quant(a, c, s, g, f"fused outliers T={T} norm={norm}")
    assert nv.device_status() == 0
