"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import torch

import nvfp4_block_scaled_device_gb300 as nv
import oracle

# Float tolerance of the GEMM and MLP outputs against the binary64 oracle on
# the same quantized operands: relative Frobenius error <= 5e-3 and, per
# element, |err| <= 2^-7 |ref| + 1e-3 * sum_k |a_k w_k| (alpha included).
REL_FROB = 5e-3
ELEM_REL = 2.0 ** -7
ELEM_ABS = 1e-3


def dev(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def host(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def quantize_gpu(bits, ws, norm_w=None):
    return nv.quantize_new(dev(bits), ws, None if norm_w is None else dev(norm_w))


def oracle_quant(bits):
    g = oracle.global_scale(bits)
    c, s = oracle.quantize(bits, g)
    return c, s, g


def assert_same_quant(t, codes, sf_logical, g, what=""):
    torch.cuda.synchronize()
    assert t.g.item() == np.float32(g), f"{what} global scale {t.g.item()!r} != {g!r}"
    gc = t.codes.cpu().numpy()
    bad = np.argwhere(gc != codes)
    assert bad.size == 0, f"{what} codes differ at {bad[:5].tolist()} ({len(bad)} bytes)"
    swz = oracle.sf_swizzle(sf_logical)
    gs = t.sf.cpu().numpy()
    assert gs.shape == swz.shape, f"{what} scale buffer size"
    bad = np.nonzero(gs != swz)[0]
    assert bad.size == 0, f"{what} scales differ at byte offsets {bad[:5].tolist()} ({bad.size})"


def check_close(got, ref, absref, what=""):
    """got: float64 array of the GPU output; ref/absref from the oracle."""
    err = np.abs(got - ref)
    bound = ELEM_REL * np.abs(ref) + ELEM_ABS * absref
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements outside the bound, first {bad[:3].tolist()}: "
                           f"got {got[tuple(bad[0])]!r} ref {ref[tuple(bad[0])]!r}")
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nrm if nrm > 0 else np.linalg.norm(got)
    assert rel <= REL_FROB, f"{what}: relative Frobenius error {rel:.3e}"
    return rel


def oracle_mlp_rows(x_bits, rows, norm_w, wq, g_inter, add_residual=True, eps=1e-6):
    """Oracle MLP output for a subset of token rows of x.  RMSNorm and the
    activation global scale cover ALL rows (the scale is per tensor); every
    later step is per row, so the sampled rows are exact.
    wq: dict with 'gate', 'up', 'down' -> (codes, logical sf, g) from the
    oracle.  g_inter: the intermediate global scale (given).
    Returns (ref fp64 [len(rows), H], absref fp64) of the down projection
    (+ residual in ref)."""
    y_all = oracle.rmsnorm(x_bits, norm_w, eps)
    g_h = oracle.global_scale(y_all)
    hc, hs = oracle.quantize(y_all[rows], g_h)
    gc, gs, gg = wq["gate"]
    uc, us, gu = wq["up"]
    dc, ds, gd = wq["down"]
    _, _, gate = oracle.gemm(hc, hs, g_h, gc, gs, gg)
    _, _, up = oracle.gemm(hc, hs, g_h, uc, us, gu)
    s = oracle.swiglu(gate, up)
    sc, ss = oracle.quantize(s, g_inter)
    ref, absref, _ = oracle.gemm(sc, ss, g_inter, dc, ds, gd)
    if add_residual:
        ref = ref + f64(x_bits[rows])
    return ref, absref, s
