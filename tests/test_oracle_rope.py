"""Pins of the oracle's rotary embedding (CPU only), the QKV-epilogue step
of "PERFORMANCE -- verified hot-path audit" P5: each test ties it to
something other than its own formula -- exact special angles, complex
multiplication in binary64, the inverse rotation, the untouched columns."""
import numpy as np
import pytest

import synthetic

HD, RD = 128, 64          # head_dim, rotated columns per head (the page's rope_dim)
QH, KH = 40, 8            # Q heads and K heads of the 7168-wide QKV output (V: 8 more)


def qkv_rows(rng, T):
    return synthetic.normal(rng, (T, synthetic.QKV))


def f32(bits):
    return synthetic.bf16_bits_to_f32(bits).astype(np.float64)


def const_tables(P, c, s):
    return np.full((P, RD // 2), c, np.float32), np.full((P, RD // 2), s, np.float32)


def test_zero_angle_is_identity(oracle_mod):
    rng = np.random.default_rng(0)
    y = qkv_rows(rng, 5)
    ct, st = const_tables(3, 1.0, 0.0)
    out = oracle_mod.rope(y, rng.integers(0, 3, 5), ct, st, 0, QH + KH, HD, RD)
    assert np.array_equal(out, y)


@pytest.mark.parametrize("inverse", [False, True])
def test_quarter_turn_swaps_pairs_exactly(oracle_mod, inverse):
    """c = 0, s = 1: (e, o) -> (-o, e) forward, (o, -e) inverse, bit for bit,
    on exactly the last RD columns of each rotated head."""
    rng = np.random.default_rng(1)
    T = 4
    y = qkv_rows(rng, T)
    ct, st = const_tables(2, 0.0, 1.0)
    out = oracle_mod.rope(y, np.zeros(T, np.int64), ct, st, 0, QH + KH, HD, RD, inverse=inverse)
    exp = y.copy()
    for h in range(QH + KH):
        base = h * HD + HD - RD
        e, o = y[:, base:base + RD:2], y[:, base + 1:base + RD:2]
        if inverse:
            exp[:, base:base + RD:2], exp[:, base + 1:base + RD:2] = o, e ^ np.uint16(0x8000)
        else:
            exp[:, base:base + RD:2], exp[:, base + 1:base + RD:2] = o ^ np.uint16(0x8000), e
    assert np.array_equal(out, exp)


def test_matches_complex_multiplication(oracle_mod):
    """(e + i o)(c + i s) in binary64, rounded to bf16: the oracle's two
    binary32 roundings can move a result by at most one bf16 ulp."""
    rng = np.random.default_rng(2)
    T, P = 16, 4096
    y = qkv_rows(rng, T)
    pos = rng.integers(0, P, T)
    ct, st = synthetic.rope_tables(P, RD)
    out = f32(oracle_mod.rope(y, pos, ct, st, 0, QH + KH, HD, RD))
    yy = f32(y)
    for h in range(QH + KH):
        base = h * HD + HD - RD
        z = (yy[:, base:base + RD:2] + 1j * yy[:, base + 1:base + RD:2]) * \
            (ct[pos].astype(np.float64) + 1j * st[pos].astype(np.float64))
        for got, ref in ((out[:, base:base + RD:2], z.real), (out[:, base + 1:base + RD:2], z.imag)):
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
            assert np.all(np.abs(got - ref) <= ulp * 1.01 + 1e-30), h


def test_inverse_undoes_forward(oracle_mod):
    rng = np.random.default_rng(3)
    T, P = 32, 1024
    y = qkv_rows(rng, T)
    pos = rng.integers(0, P, T)
    ct, st = synthetic.rope_tables(P, RD)
    back = f32(oracle_mod.rope(oracle_mod.rope(y, pos, ct, st, 0, QH + KH, HD, RD), pos, ct, st, 0, QH + KH, HD,
                               RD, inverse=True))
    yy = f32(y)
    # two bf16 roundings of a rotation: within ~3 ulps of the pair's norm
    for h in range(QH + KH):
        base = h * HD + HD - RD
        norm = np.hypot(yy[:, base:base + RD:2], yy[:, base + 1:base + RD:2])
        for k in (0, 1):
            d = np.abs(back[:, base + k:base + RD:2] - yy[:, base + k:base + RD:2])
            assert np.all(d <= 3 * 2.0 ** -8 * norm + 1e-30)


def test_unrotated_columns_untouched(oracle_mod):
    """The first HD - RD columns of each head, the V heads and the heads
    outside [col0, col0 + heads * HD) are copied bit for bit."""
    rng = np.random.default_rng(4)
    T, P = 6, 64
    y = qkv_rows(rng, T)
    ct, st = synthetic.rope_tables(P, RD)
    col0, heads = 3 * HD, 20
    out = oracle_mod.rope(y, rng.integers(0, P, T), ct, st, col0, heads, HD, RD)
    rotated = np.zeros(y.shape[1], bool)
    for h in range(heads):
        rotated[col0 + h * HD + HD - RD:col0 + (h + 1) * HD] = True
    assert np.array_equal(out[:, ~rotated], y[:, ~rotated])
    assert not np.array_equal(out[:, rotated], y[:, rotated])


def test_position_selects_the_table_row(oracle_mod):
    """Row t uses table row pos[t]: the same rows with the tables shifted by
    k and positions shifted by k give the same output."""
    rng = np.random.default_rng(5)
    T, P, k = 9, 200, 37
    y = qkv_rows(rng, T)
    pos = rng.integers(0, P - k, T)
    ct, st = synthetic.rope_tables(P, RD)
    a = oracle_mod.rope(y, pos, ct, st, 0, QH + KH, HD, RD)
    b = oracle_mod.rope(y, pos + k, np.roll(ct, k, axis=0), np.roll(st, k, axis=0), 0, QH + KH, HD, RD)
    assert np.array_equal(a, b)
    c = oracle_mod.rope(y, (pos + 1) % P, ct, st, 0, QH + KH, HD, RD)
    assert not np.array_equal(a, c)
