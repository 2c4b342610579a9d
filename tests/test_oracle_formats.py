"""Pins of the oracle's number formats and global scale (CPU only).

Each test ties the oracle to something other than itself: the value set of
the format, a closed form, torch's float8_e4m3fn cast, or an exhaustive
threshold formulation of round-to-nearest-even.
"""
import math
import struct

import numpy as np
import pytest
import torch

from conftest import read_golden


def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def f32_from_bits(b):
    return struct.unpack("<f", struct.pack("<I", int(b)))[0]


def neighbours(v):
    """v and its binary32 neighbours one ulp below and above."""
    b = f32_bits(v)
    return [f32_from_bits(b - 1) if v > 0 else -f32_from_bits(1), v, f32_from_bits(b + 1)]


# ------------------------------------------------------------------- E2M1
def test_e2m1_value_set_matches_golden(oracle_mod):
    table = {int(c): float(m) for c, m in read_golden("e2m1_values.txt")}
    assert sorted(table) == list(range(8))
    for c in range(8):
        assert oracle_mod.e2m1_value(c) == table[c]
        assert oracle_mod.e2m1_value(c | 8) == -table[c]
        assert math.copysign(1.0, oracle_mod.e2m1_value(c | 8)) == -1.0


def test_e2m1_minifloat_closed_form(oracle_mod):
    # OCP E2M1: exponent bias 1; e == 0 is subnormal (m * 0.5).
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        v = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert oracle_mod.e2m1_value(code) == (-v if s else v)


# thresholds of RNE onto {0,.5,1,1.5,2,3,4,6}: (midpoint, code taken AT the tie)
E2M1_MIDPOINTS = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]


def e2m1_by_thresholds(q):
    a = abs(q)
    code = 0
    for mid, at_tie in E2M1_MIDPOINTS:
        if a > mid or (a == mid and at_tie > code):
            code += 1
    return code | (8 if math.copysign(1.0, q) < 0 else 0)


def test_e2m1_encode_exhaustive_midpoints(oracle_mod):
    pts = [0.0, 1e-30, 0.1, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 6.5, 7.0, 100.0, 1e30]
    for mid, _ in E2M1_MIDPOINTS:
        pts += neighbours(mid)
    rng = np.random.default_rng(5)
    pts += list(rng.uniform(0, 8, 4000).astype(np.float32))
    for v in pts:
        for q in (float(np.float32(v)), -float(np.float32(v))):
            assert oracle_mod.e2m1_encode(q) == e2m1_by_thresholds(q), q


def test_e2m1_nearest_property(oracle_mod):
    # the chosen code's magnitude is at least as near as every other one
    mags = [oracle_mod.e2m1_value(c) for c in range(8)]
    for v in np.linspace(0, 7, 2801, dtype=np.float32):
        c = oracle_mod.e2m1_encode(float(v)) & 7
        assert all(abs(v - mags[c]) <= abs(v - m) for m in mags)


def test_e2m1_saturates_and_keeps_sign(oracle_mod):
    assert oracle_mod.e2m1_encode(6.0) == 7
    assert oracle_mod.e2m1_encode(1e9) == 7
    assert oracle_mod.e2m1_encode(-1e9) == 15
    assert oracle_mod.e2m1_encode(-0.1) == 8
    assert oracle_mod.e2m1_encode(-0.0) == 8
    assert oracle_mod.e2m1_encode(0.0) == 0


# ------------------------------------------------------------------- E4M3
def test_e4m3_decode_all_bytes_vs_torch(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        v = oracle_mod.e4m3_value(b)
        if math.isnan(ref[b]):
            assert math.isnan(v) and (b & 0x7F) == 0x7F
        else:
            assert v == ref[b], b


def test_e4m3_golden_points(oracle_mod):
    for v, hx, _ in read_golden("e4m3_points.txt"):
        assert oracle_mod.e4m3_encode(float(v)) == int(hx, 16), v
    assert oracle_mod.e4m3_value(0x7E) == 448.0


def test_e4m3_encode_vs_torch_cast(oracle_mod):
    # torch's float32 -> float8_e4m3fn cast rounds to nearest-even; it turns
    # values past the saturation midpoint (464) into NaN, so compare below it.
    vals = [oracle_mod.e4m3_value(b) for b in range(0x7F)]
    pts = []
    for a, b in zip(vals[:-1], vals[1:]):
        pts += neighbours((a + b) / 2)
        pts += neighbours(b)
    rng = np.random.default_rng(6)
    pts += list(np.exp(rng.uniform(math.log(1e-4), math.log(460), 20000)).astype(np.float32))
    pts = np.array([p for p in pts if 0 <= p < 464], np.float32)
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(p)) for p in pts])
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(pts[i], got[i], ref[i]) for i in bad[:5]]


def test_e4m3_saturates(oracle_mod):
    for v in [448.0, 460.0, 464.0, 480.0, 1e6, 3e38]:
        assert oracle_mod.e4m3_encode(v) == 0x7E


# ------------------------------------------------------------ global scale
def test_global_scale_golden(oracle_mod):
    for a, hx, *_ in read_golden("global_scale.txt"):
        g = oracle_mod.global_scale_from_amax(float(a))
        assert f32_bits(g) == int(hx, 16), (a, hex(f32_bits(g)))


def test_global_scale_power_of_two_closed_form(oracle_mod):
    for k in range(-20, 20):
        assert oracle_mod.global_scale_from_amax(2688.0 * 2.0 ** k) == np.float32(2.0 ** k)


def test_global_scale_of_tensor_uses_abs_max(oracle_mod):
    import synthetic
    x = synthetic.f32_to_bf16_bits(np.array([[0.5, -5376.0, 3.0, 0.0]], np.float32))
    assert oracle_mod.amax(x) == 5376.0
    assert oracle_mod.global_scale(x) == np.float32(2.0)
    z = np.zeros((3, 32), np.uint16)
    assert f32_bits(oracle_mod.global_scale(z)) == 0x2C82E4ED


# ------------------------------------------------------------------ bf16
def test_bf16_rounding_nearest_even(oracle_mod):
    # 1 + 2^-8 is the tie between 1 and 1 + 2^-7: even mantissa -> 1
    assert oracle_mod.bf16_from_double(1 + 2 ** -8) == 0x3F80
    assert oracle_mod.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82
    assert oracle_mod.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    rng = np.random.default_rng(7)
    v = rng.standard_normal(5000).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.bf16_from_double(float(t)) for t in v], np.uint16)
    assert np.array_equal(got, ref)
