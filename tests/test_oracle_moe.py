"""Pins of the oracle's expert-indexed GEMM (CPU only), the routed
projection of a mixture-of-experts layer ("CUDA: NVFP4 prefill on Blackwell
leaves ~1.45x performance on the table", its MUL_MAT_ID tests; "PERFORMANCE
-- verified hot-path audit", the routed experts run from a device-side
routing table without a host sync).  Tied to an independent decode and
explicit fp64 sums, and to relabelling and routing invariants."""
import numpy as np

import synthetic
from _decode import dequant_independent


def quantized_experts(oracle_mod, rng, E, N, K):
    c, s, g = [], [], []
    for _ in range(E):
        w = synthetic.normal(rng, (N, K), std=0.02)
        ge = oracle_mod.global_scale(w)
        wc, wsf = oracle_mod.quantize(w, ge)
        c.append(wc), s.append(wsf), g.append(ge)
    return np.stack(c), np.stack(s), np.array(g, np.float32)


def quantized_tokens(oracle_mod, rng, T, K):
    a = synthetic.normal(rng, (T, K))
    ga = oracle_mod.global_scale(a)
    ac, asf = oracle_mod.quantize(a, ga)
    return ac, asf, ga


def test_matches_explicit_fp64_sums(oracle_mod):
    rng = np.random.default_rng(0)
    T, k, E, N, K = 5, 2, 4, 16, 128
    ac, asf, ga = quantized_tokens(oracle_mod, rng, T, K)
    wc, wsf, gw = quantized_experts(oracle_mod, rng, E, N, K)
    ids = rng.integers(0, E, (T, k))
    ref, absref, out = oracle_mod.gemm_id(ac, asf, ga, wc, wsf, gw, ids)
    A = dequant_independent(ac, asf, 1.0)                   # element values without g (not the oracle's decode)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            W = dequant_independent(wc[e], wsf[e], 1.0)
            alpha = float(np.float32(np.float32(ga) * gw[e]))
            exp = alpha * (W @ A[t])
            assert np.allclose(ref[t, j], exp, rtol=1e-12, atol=1e-300)
            assert np.allclose(absref[t, j], alpha * (np.abs(W) @ np.abs(A[t])), rtol=1e-12)
            for n in range(N):
                assert out[t, j, n] == oracle_mod.bf16_from_double(ref[t, j, n])


def test_single_expert_routing_is_the_plain_gemm(oracle_mod):
    rng = np.random.default_rng(1)
    T, E, N, K = 7, 3, 32, 256
    ac, asf, ga = quantized_tokens(oracle_mod, rng, T, K)
    wc, wsf, gw = quantized_experts(oracle_mod, rng, E, N, K)
    for e in range(E):
        _, _, out = oracle_mod.gemm_id(ac, asf, ga, wc, wsf, gw, np.full((T, 1), e))
        _, _, plain = oracle_mod.gemm(ac, asf, ga, wc[e], wsf[e], gw[e])
        assert np.array_equal(out[:, 0], plain)


def test_relabelling_experts_changes_nothing(oracle_mod):
    rng = np.random.default_rng(2)
    T, k, E, N, K = 9, 3, 5, 16, 192
    ac, asf, ga = quantized_tokens(oracle_mod, rng, T, K)
    wc, wsf, gw = quantized_experts(oracle_mod, rng, E, N, K)
    ids = rng.integers(0, E, (T, k))
    perm = rng.permutation(E)                    # new label of old expert e: perm[e]
    inv = np.argsort(perm)
    _, _, a = oracle_mod.gemm_id(ac, asf, ga, wc, wsf, gw, ids)
    _, _, b = oracle_mod.gemm_id(ac, asf, ga, wc[inv], wsf[inv], gw[inv], perm[ids])
    assert np.array_equal(a, b)
    # a token routed to two different experts gets two different rows
    t = int(np.nonzero(ids[:, 0] != ids[:, 1])[0][0])
    assert not np.array_equal(a[t, 0], a[t, 1])
