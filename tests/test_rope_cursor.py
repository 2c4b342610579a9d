"""CPU check of the index walk the GEMM epilogues use for the rotary
embedding (csrc/gemm_epilogue.cuh, rope_begin / rope_step): a thread walks
its output columns in pairs from an even column (128 columns from a
multiple of 128 in the tensor-core epilogues, one pair in the decode
kernel), keeping the rotated-head index and the column within the head.
The walk, written out here step by step with binary32 arithmetic, must give
the oracle's rotation bit for bit for every layout."""
import numpy as np
import pytest

import synthetic

F = np.float32


def walk(row_bits, n0, count, pos_row, ct, st, col0, heads, hd, rd, inverse):
    """Rotate `count` columns of one row from even column n0 as the epilogue
    does; returns the new bf16 bits of those columns."""
    y = synthetic.bf16_bits_to_f32(row_bits[n0:n0 + count]).copy()
    rel = n0 - col0
    head = rel // hd                      # floor division, as rope_begin
    within = rel - head * hd
    nope = hd - rd
    for q in range(count // 2):
        if 0 <= head < heads and within >= nope:
            i = (within - nope) >> 1
            c, s = ct[pos_row, i], st[pos_row, i]
            e, o = F(y[2 * q]), F(y[2 * q + 1])
            ec, os_, es, oc = F(e * c), F(o * s), F(e * s), F(o * c)
            if inverse:
                y[2 * q], y[2 * q + 1] = F(ec + os_), F(oc - es)
            else:
                y[2 * q], y[2 * q + 1] = F(ec - os_), F(es + oc)
        within += 2
        if within >= hd:
            within -= hd
            head += 1
    return synthetic.f32_to_bf16_bits(y)


@pytest.mark.parametrize("N,col0,heads,hd,rd", [(7168, 0, 48, 128, 64), (1024, 0, 8, 128, 128), (768, 64, 10, 64, 32),
                                                (2048, 256, 5, 256, 96), (640, 2, 3, 18, 6), (512, 130, 2, 190, 190)])
@pytest.mark.parametrize("inverse", [False, True])
def test_epilogue_walk_equals_oracle(oracle_mod, N, col0, heads, hd, rd, inverse):
    rng = np.random.default_rng(N + col0 + hd)
    T, P = 3, 97
    y = synthetic.normal(rng, (T, N))
    pos = rng.integers(0, P, T)
    ct, st = synthetic.rope_tables(P, rd)
    exp = oracle_mod.rope(y, pos, ct, st, col0, heads, hd, rd, inverse=inverse)
    for t in range(T):
        # tensor-core epilogue: 128-column chunks from multiples of 128
        got = np.concatenate([walk(y[t], n0, min(128, N - n0), pos[t], ct, st, col0, heads, hd, rd, inverse)
                              for n0 in range(0, N, 128)])
        assert np.array_equal(got, exp[t])
        # decode kernel: one pair per thread
        got = np.concatenate([walk(y[t], n0, 2, pos[t], ct, st, col0, heads, hd, rd, inverse)
                              for n0 in range(0, N, 2)])
        assert np.array_equal(got, exp[t])
