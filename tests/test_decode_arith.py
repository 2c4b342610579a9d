"""CPU checks of the identities the decode-regime GEMM kernel rests on
(csrc/gemv.cu), each against the oracle's own format decoders or brute
force:

- the byte-permute split of four E2M1 codes into the magnitudes of the
  positive codes and of the negative codes (the PTX prmt default mode, as
  its definition reads: a selector nibble picks one of eight bytes, and with
  its bit 3 set yields that byte's sign replicated instead), whose bytewise
  difference is 2 x the code's value;
- the E4M3 scale byte read as the binary32 bit pattern byte << 20 is the
  scale times 2^-120 exactly (subnormal scales included), and the product
  of an activation scale times 2^119 with it is the exact sA * sW / 2;
- an exact int32 block sum times that product is exact in binary32;
- the work split: every (weight row, 1024-element unit) of a CTA belongs to
  exactly one warp, and a warp's range touches at most `slots` rows.
"""
import struct

import numpy as np
import pytest

MAG_LO, MAG_HI = 0x03020100, 0x0C080604


def prmt(a, b, sel):
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    r = 0
    for i in range(4):
        nib = (sel >> (4 * i)) & 0xF
        byte = src[nib & 7]
        if nib & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        r |= byte << (8 * i)
    return r


def f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def test_permute_split_gives_twice_the_code_value(oracle_mod):
    rng = np.random.default_rng(0)
    words = list(range(1 << 16)) + [int(x) for x in rng.integers(0, 1 << 32, 2000, dtype=np.uint64)]
    for w in words:
        pos = prmt(MAG_LO, MAG_HI, w)
        neg = prmt(MAG_LO, MAG_HI, w ^ 0x8888)
        for i in range(4):
            code = (w >> (4 * i)) & 0xF
            p, n = (pos >> (8 * i)) & 0xFF, (neg >> (8 * i)) & 0xFF
            assert p == 0 or n == 0
            assert p - n == 2 * oracle_mod.e2m1_value(code), (hex(w), i)


def test_scale_bit_pattern_and_product_are_exact(oracle_mod):
    vals = [oracle_mod.e4m3_value(b) for b in range(127)]   # 0x7F is NaN; scales stop at 0x7E = 448
    for b, v in enumerate(vals):
        assert f32(b << 20) == v * 2.0 ** -120, b
        assert v * 2.0 ** 119 < 2.0 ** 128
    a = np.array([v * 2.0 ** 119 for v in vals], np.float32)
    w = np.array([f32(b << 20) for b in range(127)], np.float32)
    prod = a[:, None] * w[None, :]                                # binary32 products
    exact = np.array(vals)[:, None] * np.array(vals)[None, :] / 2
    assert np.array_equal(prod.astype(np.float64), exact)
    # nonzero products are normal numbers with at most 8 significant bits, so
    # any |S| <= 16 * 144 (an int32 block sum of 2 x E2M1 products) times
    # them is exact in binary32
    nz = exact[exact > 0]
    assert nz.min() >= 2.0 ** -126
    m, _ = np.frexp(nz)
    assert np.all(np.ldexp(m, 8) == np.round(np.ldexp(m, 8)))
    S = np.arange(-16 * 144, 16 * 144 + 1, dtype=np.float64)
    sample = nz[np.random.default_rng(1).integers(0, nz.size, 64)]
    assert np.array_equal((S[:, None].astype(np.float32) * sample[None, :].astype(np.float32)).astype(np.float64),
                          S[:, None] * sample[None, :])


def decode_shape(N, K, swiglu, num_sms, warps=16, unit=1024):
    units = N // 16 if swiglu else N // 2        # 16-column blocks, or column pairs
    grid = min(units, num_sms)
    segs = (K + unit - 1) // unit
    per = (units + grid - 1) // grid
    rmax = 32 * per if swiglu else 2 * per
    umax = (rmax * segs + warps - 1) // warps
    slots = (umax + 2 * segs - 2) // segs
    return grid, segs, slots, rmax


@pytest.mark.parametrize("swiglu", [False, True])
def test_work_split_covers_each_unit_once(swiglu):
    rng = np.random.default_rng(2)
    cases = [(16, 64, 152), (48, 1088, 5), (5120, 17408, 152), (7168, 5120, 152), (17408, 5120, 152),
             (1040, 320, 152), (256, 2112, 7), (128, 65536, 3)]
    cases += [(16 * int(rng.integers(1, 3000)), 64 * int(rng.integers(1, 400)), int(rng.integers(1, 200)))
              for _ in range(60)]
    for N, K, sms in cases:
        grid, S, slots, rmax = decode_shape(N, K, swiglu, sms)
        cols = 0
        for c in range(grid):
            if swiglu:
                nb = N // 16
                C = 16 * ((c + 1) * nb // grid - c * nb // grid)
                R = 2 * C
            else:
                C = 2 * ((c + 1) * (N // 2) // grid - c * (N // 2) // grid)
                R = C
            assert 1 <= R <= rmax
            cols += C
            U = R * S
            seen = np.zeros(U, np.int32)
            for w in range(16):
                b, e = w * U // 16, (w + 1) * U // 16
                seen[b:e] += 1
                if e > b:
                    assert (e - 1) // S - b // S + 1 <= slots, (N, K, sms, c, w)
            assert np.all(seen == 1)
        assert cols == N
