"""Pins of the oracle's quantizer, scale layout, GEMM, RMSNorm, SwiGLU and MLP
(CPU only).  References used: exact constructions, invariants, hand-worked
offsets, numpy/scipy binary64 routines and torch casts -- never the oracle
itself."""
import math

import numpy as np
import pytest
import scipy.special
import torch

import synthetic
from conftest import read_golden

from _decode import E2M1, dequant_independent, e4m3_torch  # noqa: F401  (decode shared by the pins)


def bf16(v):
    return synthetic.f32_to_bf16_bits(np.asarray(v, np.float32))


def f32(b):
    return synthetic.bf16_bits_to_f32(b).astype(np.float64)


# ------------------------------------------------------------- dequantize
def test_dequantize_matches_independent_decode(oracle_mod):
    """The oracle's element decode against the golden-table / torch-cast
    decode: every code at every finite scale byte, in both nibbles, with a
    non-trivial global scale."""
    sc = np.arange(0x7F, dtype=np.uint8)                # every non-NaN E4M3 byte
    rows = sc.size
    # codes: byte j of a 16-element block holds codes (2j, 2j+1); cover all
    # 16 codes in both nibbles across the row
    lo = np.arange(16, dtype=np.uint8)
    hi = (lo * 7 + 3) % 16
    block = (lo[:8] | (hi[:8] << 4)).astype(np.uint8)
    block2 = (lo[8:] | (hi[8:] << 4)).astype(np.uint8)
    codes = np.tile(np.concatenate([block, block2]), (rows, 1))     # 32 elements per row
    sf = np.stack([sc, sc[::-1]], axis=1)                           # two blocks per row
    g = float(np.float32(0.0123))
    got = oracle_mod.dequantize(codes, sf, g)
    want = dequant_independent(codes, sf, np.float32(g))
    assert np.array_equal(got, want)
    # a sign or nibble-order slip shows up: element 1 of row 1 is code hi[0]
    assert got[1, 1] == (-1.0 if hi[0] & 8 else 1.0) * E2M1[hi[0] & 7] * e4m3_torch([1])[0] * np.float32(g)


# --------------------------------------------------------------- quantize
@pytest.mark.parametrize("g", [2.0 ** -3, 1.0, 2.0 ** 5])
def test_quantize_exact_roundtrip_every_scale_and_code(oracle_mod, g):
    """With g a power of two every step is exact: a block made of
    code * scale * g values (one element = 6 * scale * g) must come back as
    exactly that scale and those codes."""
    rng = np.random.default_rng(8)
    rows = []
    want_sc, want_codes = [], []
    for sc in range(1, 0x7F):
        s = oracle_mod.e4m3_value(sc)
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = 7 | (8 * rng.integers(0, 2))
        vals = np.where(codes & 8, -1.0, 1.0) * E2M1[codes & 7] * s * g
        rows.append(vals)
        want_sc.append(sc)
        want_codes.append(codes)
    x = bf16(np.array(rows))
    assert np.array_equal(f32(x), np.array(rows))           # exactly representable
    codes, sf = oracle_mod.quantize(x, g)
    assert list(sf[:, 0]) == want_sc
    got = np.stack([codes & 15, codes >> 4], -1).reshape(len(rows), 16)
    want = np.array(want_codes)
    # a zero element of either sign decodes as zero; compare magnitudes there
    nz = (want & 7) != 0
    assert np.array_equal(got[nz], want[nz])
    assert np.all((got[~nz] & 7) == 0)


def test_quantize_ties_go_to_even_codes(oracle_mod):
    # scale 1.0 (0x38) and g = 1: den = 1, so q = x exactly; one element = 6
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    row = [6.0] + mids + [-m for m in mids] + [0.0]
    x = bf16(np.array([row]))
    codes, sf = oracle_mod.quantize(x, np.float32(1.0 / 1.0))
    # g = 1 -> d = 6, s_raw = 1, scale byte 0x38
    assert sf[0, 0] == 0x38
    got = np.stack([codes & 15, codes >> 4], -1).reshape(-1)
    assert list(got[1:8]) == [0, 2, 2, 4, 4, 6, 6]
    assert list(got[8:15]) == [8, 10, 10, 12, 12, 14, 14]


def test_quantize_invariants(oracle_mod):
    rng = np.random.default_rng(9)
    x = synthetic.normal(rng, (7, 256))
    g = oracle_mod.global_scale(x)
    c1, s1 = oracle_mod.quantize(x, g)
    # sign symmetry: negating x flips exactly the sign bit of every nibble
    c2, s2 = oracle_mod.quantize(x ^ np.uint16(0x8000), g)
    assert np.array_equal(s1, s2)
    assert np.array_equal(c2, c1 ^ np.uint8(0x88))
    # power-of-two scaling with g recomputed leaves codes and scales alone
    for k in (-6, 3):
        xs = bf16(f32(x) * 2.0 ** k)
        gs = oracle_mod.global_scale(xs)
        assert gs == np.float32(g * 2.0 ** k)
        c3, s3 = oracle_mod.quantize(xs, gs)
        assert np.array_equal(c3, c1) and np.array_equal(s3, s1)
    # the block holding the tensor amax gets the largest scale, 448
    r, c = np.unravel_index(np.argmax(np.abs(f32(x))), x.shape)
    assert s1[r, c // 16] == 0x7E
    assert np.all(s1 <= 0x7E)
    # an all-zero block: scale 0, codes 0
    xz = x.copy()
    xz[2, 32:48] = 0
    cz, sz = oracle_mod.quantize(xz, g)
    assert sz[2, 2] == 0 and np.all(cz[2, 16:24] == 0)


def test_quantize_error_bound(oracle_mod):
    """|x - dequant| is at most half an E2M1 step of the block scale (plus
    the scale's own rounding for the saturating top element)."""
    rng = np.random.default_rng(10)
    x = synthetic.normal(rng, (16, 512))
    g = oracle_mod.global_scale(x)
    codes, sf = oracle_mod.quantize(x, g)
    xd = dequant_independent(codes, sf, g)
    scale = np.repeat(e4m3_torch(sf), 16, axis=1) * float(g)
    err = np.abs(f32(x) - xd)
    # step of E2M1 is at most 2 (between 4 and 6); allow one full step at the top
    assert np.all(err <= 2.0 * scale * 1.07 + 1e-30)
    rel = np.linalg.norm(f32(x) - xd) / np.linalg.norm(f32(x))
    assert rel < 0.12


# ----------------------------------------------------------------- layout
def test_sf_layout_golden_offsets(oracle_mod):
    for kb, r, c, off in read_golden("sf_layout.txt"):
        assert oracle_mod.sf_offset(int(r), int(c), int(kb)) == int(off), (kb, r, c)


@pytest.mark.parametrize("rows,kb", [(1, 4), (130, 6), (256, 16), (17, 3)])
def test_sf_swizzle_bijection(oracle_mod, rows, kb):
    rng = np.random.default_rng(rows * 31 + kb)
    logical = rng.integers(1, 255, (rows, kb), dtype=np.uint8)
    swz = oracle_mod.sf_swizzle(logical)
    pr, pc = oracle_mod.sf_padded_shape(rows, kb)
    assert swz.size == pr * pc and pr % 128 == 0 and pc % 4 == 0
    offs = {oracle_mod.sf_offset(r, c, kb) for r in range(rows) for c in range(kb)}
    assert len(offs) == rows * kb                       # injective
    assert np.count_nonzero(swz) == rows * kb           # padding is zero
    assert np.array_equal(oracle_mod.sf_unswizzle(swz, rows, kb), logical)


# ------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (3, 5, 128), (17, 13, 256), (16, 17, 192)])
def test_gemm_exact_vs_numpy_fp64(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    a = synthetic.normal(rng, (M, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    ga, gw = oracle_mod.global_scale(a), oracle_mod.global_scale(w)
    ac, asf = oracle_mod.quantize(a, ga)
    wc, wsf = oracle_mod.quantize(w, gw)
    ref, absref, out = oracle_mod.gemm(ac, asf, ga, wc, wsf, gw)
    A = dequant_independent(ac, asf, 1.0)
    W = dequant_independent(wc, wsf, 1.0)
    alpha = float(np.float32(ga * gw))
    np.testing.assert_allclose(ref, alpha * (A @ W.T), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(absref, alpha * (np.abs(A) @ np.abs(W).T), rtol=1e-12, atol=1e-300)
    # bf16 output is the nearest bf16 of ref (torch's float32->bf16 cast of
    # a value exactly representable in float32 is a single rounding)
    ref32 = ref.astype(np.float32)
    exact = ref32.astype(np.float64) == ref
    want = synthetic.f32_to_bf16_bits(ref32)
    assert np.array_equal(out[exact], want[exact])


def test_gemm_sampled_matches_full(oracle_mod):
    rng = np.random.default_rng(3)
    a = synthetic.normal(rng, (9, 320))
    w = synthetic.normal(rng, (11, 320), std=0.02)
    ga, gw = oracle_mod.global_scale(a), oracle_mod.global_scale(w)
    ac, asf = oracle_mod.quantize(a, ga)
    wc, wsf = oracle_mod.quantize(w, gw)
    A = dequant_independent(ac, asf, 1.0)
    W = dequant_independent(wc, wsf, 1.0)
    m = rng.integers(0, 9, 20)
    n = rng.integers(0, 11, 20)
    dot, adot = oracle_mod.dot_sampled(ac, asf, wc, wsf, m, n)
    np.testing.assert_allclose(dot, np.einsum("ik,ik->i", A[m], W[n]), rtol=1e-12)
    np.testing.assert_allclose(adot, np.einsum("ik,ik->i", np.abs(A[m]), np.abs(W[n])), rtol=1e-12)


def test_gemm_residual_rounding(oracle_mod):
    rng = np.random.default_rng(4)
    a = synthetic.normal(rng, (4, 64))
    w = synthetic.normal(rng, (8, 64), std=0.02)
    res = synthetic.normal(rng, (4, 8))
    ga, gw = oracle_mod.global_scale(a), oracle_mod.global_scale(w)
    ac, asf = oracle_mod.quantize(a, ga)
    wc, wsf = oracle_mod.quantize(w, gw)
    ref, _, out0 = oracle_mod.gemm(ac, asf, ga, wc, wsf, gw)
    _, _, out1 = oracle_mod.gemm(ac, asf, ga, wc, wsf, gw, residual=res)
    # residual add of two bf16 values: sum exact in float32 here, one rounding
    s = (f32(res) + f32(out0)).astype(np.float32)
    assert np.array_equal(out1, synthetic.f32_to_bf16_bits(s))


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_vs_numpy(oracle_mod):
    rng = np.random.default_rng(12)
    x = synthetic.normal(rng, (6, 5120))
    w = synthetic.normal(rng, (5120,), mean=1.0, std=0.05)
    y = oracle_mod.rmsnorm(x, w, 1e-6)
    X = f32(x)
    ref = X / np.sqrt(np.mean(X * X, axis=1, keepdims=True) + 1e-6) * f32(w)
    ulp = np.abs(f32(y)) * 2.0 ** -7
    assert np.all(np.abs(f32(y) - ref) <= ulp * 1.01)


def test_rmsnorm_constant_row_closed_form(oracle_mod):
    # x = c everywhere: ms = c^2, y = w * c / sqrt(c^2 + eps) ~ w * sign(c)
    for c in (2.0, -0.5, 3.0):
        x = bf16(np.full((1, 64), c))
        w = bf16(np.linspace(0.5, 1.5, 64))
        y = oracle_mod.rmsnorm(x, w, 1e-6)
        ref = f32(w) * c / math.sqrt(c * c + 1e-6)
        assert np.all(np.abs(f32(y[0]) - ref) <= np.abs(ref) * 2.0 ** -8)
    # eps matters for a zero row: y = 0
    assert np.all(oracle_mod.rmsnorm(np.zeros((1, 64), np.uint16), bf16(np.ones(64)), 1e-6) == 0)


# ----------------------------------------------------------------- SwiGLU
def test_swiglu_vs_scipy(oracle_mod):
    rng = np.random.default_rng(13)
    gate = synthetic.normal(rng, (4000,), std=3.0)
    up = synthetic.normal(rng, (4000,))
    s = oracle_mod.swiglu(gate, up)
    G, U = f32(gate), f32(up)
    ref = G * scipy.special.expit(G) * U
    assert np.all(np.abs(f32(s) - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_swiglu_closed_forms(oracle_mod):
    one = bf16(1.0)[()]
    assert oracle_mod.swiglu(bf16([0.0]), bf16([5.0]))[0] == 0
    # silu(x) -> x for large x
    assert oracle_mod.swiglu(bf16([100.0]), bf16([2.0]))[0] == bf16(200.0)[()]
    # silu(x) -> 0 for very negative x
    assert f32(oracle_mod.swiglu(bf16([-100.0]), np.array([one])))[0] == pytest.approx(-100 * math.exp(-100), rel=1e-2)
    # gate and up are not interchangeable: silu(1)*2 != silu(2)*1
    a = f32(oracle_mod.swiglu(bf16([1.0]), bf16([2.0])))[0]
    b = f32(oracle_mod.swiglu(bf16([2.0]), bf16([1.0])))[0]
    assert a == pytest.approx(2 / (1 + math.exp(-1)), rel=2 ** -8)
    assert b == pytest.approx(2 / (1 + math.exp(-2)), rel=2 ** -8)


# -------------------------------------------------------------------- MLP
def test_mlp_tiny_against_float_reference(oracle_mod):
    """The oracle MLP, at T=5, H=64, I=128, against a binary64 float model of
    the same block (no quantization at all): they must agree to FP4
    accuracy; a dropped residual, swapped gate/up or transposed weight fails."""
    rng = np.random.default_rng(14)
    T, Hh, Ii = 5, 64, 128
    x = synthetic.normal(rng, (T, Hh))
    nw = synthetic.normal(rng, (Hh,), mean=1.0, std=0.05)
    Wg = synthetic.normal(rng, (Ii, Hh), std=0.2)
    Wu = synthetic.normal(rng, (Ii, Hh), std=0.2)
    Wd = synthetic.normal(rng, (Hh, Ii), std=0.1)
    qw = []
    for W in (Wg, Wu, Wd):
        g = oracle_mod.global_scale(W)
        c, s = oracle_mod.quantize(W, g)
        qw.append((c, s, g))
    res = oracle_mod.mlp(x, nw, *qw, g_inter=None, add_residual=True)
    X = f32(x)
    h = X / np.sqrt(np.mean(X * X, 1, keepdims=True) + 1e-6) * f32(nw)
    gate = h @ f32(Wg).T
    up = h @ f32(Wu).T
    s = gate * scipy.special.expit(gate) * up
    ref = X + s @ f32(Wd).T
    out = f32(res["out"])
    # loose: three FP4 roundings compound to ~20% at K=64; a dropped residual
    # or swapped gate/up lands far outside
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert rel < 0.35, rel
    # tight, staged: recompose the block in binary64 numpy from the oracle's
    # own quantization decisions (decoded independently)
    hq = dequant_independent(res["h_codes"], res["h_sf"], res["g_h"])
    assert np.linalg.norm(hq - h) / np.linalg.norm(h) < 0.12
    Wq = [dequant_independent(c, sf, g) for (c, sf, g) in qw]
    gate_q = hq @ Wq[0].T
    up_q = hq @ Wq[1].T
    s_q = gate_q * scipy.special.expit(gate_q) * up_q
    err_s = np.abs(f32(res["s"]) - s_q)
    bound_s = (np.abs(gate_q) + np.abs(up_q) + 1) * np.abs(s_q) * 2.0 ** -7 + 1e-6
    assert np.all(err_s <= bound_s)
    sq = dequant_independent(res["s_codes"], res["s_sf"], res["g_inter"])
    down_q = sq @ Wq[2].T
    err_o = np.abs(out - (X + down_q))
    assert np.all(err_o <= (np.abs(X) + np.abs(down_q)) * 2.0 ** -7 + 1e-3 * (np.abs(sq) @ np.abs(Wq[2]).T))
    # without the residual the output is the down projection alone
    res2 = oracle_mod.mlp(x, nw, *qw, g_inter=None, add_residual=False)
    assert np.all(np.abs(f32(res2["out"]) - down_q) <= np.abs(down_q) * 2.0 ** -7 + 1e-3 * (np.abs(sq) @ np.abs(Wq[2]).T))
    # a fixed intermediate scale equal to the per-call one gives the same result
    res3 = oracle_mod.mlp(x, nw, *qw, g_inter=res["g_inter"], add_residual=True)
    assert np.array_equal(res3["out"], res["out"])
    assert res["g_inter"] == oracle_mod.global_scale(res["s"])
