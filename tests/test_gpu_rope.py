"""GPU parity of the GEMM with the rotary embedding in its epilogue
(nvfp4_gemm_rope) against the oracle: the rotated output must equal, bit
for bit, the oracle's rotation of the GPU's own unrotated GEMM output (the
same kernel and schedule, so the same accumulator and bf16 rounding), and
the GEMM output itself stays within the GEMM tolerance of the oracle.
Covers the decode kernel (T = 1, 2), the 1-SM and the SM-pair kernels, the
split schedule, both directions and several head layouts."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from _gpu import check_close, f64, host, oracle_quant, quantize_gpu

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


def run(nv, ws, T, N, K, col0, heads, hd, rd, inverse, seed, split=False, P=4096):
    rng = np.random.default_rng(seed)
    a = synthetic.normal(rng, (T, K))
    w = synthetic.normal(rng, (N, K), std=0.02)
    A, W = quantize_gpu(a, ws), quantize_gpu(w, ws)
    pos = rng.integers(0, P, T)
    ct, st = synthetic.rope_tables(P, rd)
    gws = nv.workspace(nv.gemm_workspace_bytes()) if split else None
    plain = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    rot = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(A, W, plain, workspace=gws)
    nv.nvfp4_gemm_rope(A, W, rot, torch.from_numpy(pos.astype(np.int32)).cuda(), torch.from_numpy(ct).cuda(),
                       torch.from_numpy(st).cuda(), col0, heads, hd, rd, inverse=inverse, workspace=gws)
    torch.cuda.synchronize()
    assert nv.device_status() == 0
    exp = oracle.rope(host(plain), pos, ct, st, col0, heads, hd, rd, inverse=inverse)
    got = host(rot)
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{len(bad)} outputs differ from the oracle's rotation, first {bad[:3].tolist()}"
    ac, asf, ga = oracle_quant(a)
    wc, wsf, gw = oracle_quant(w)
    if T * N <= 1 << 21:
        ref, absref, _ = oracle.gemm(ac, asf, ga, wc, wsf, gw)
        check_close(f64(host(plain)), ref, absref, f"gemm {T}x{N}x{K}")


# the QKV projection: 40 Q heads + 8 K heads of 128 rotated, 8 V heads not
@pytest.mark.parametrize("T", [1, 2, 5, 17, 300, 1024])
def test_rope_qkv(nv, ws, T):
    run(nv, ws, T, 7168, 5120, 0, 48, 128, 64, False, seed=T)


@pytest.mark.parametrize("T", [1, 130])
def test_rope_inverse(nv, ws, T):
    run(nv, ws, T, 7168, 5120, 0, 48, 128, 64, True, seed=10 + T)


# head layouts: the whole head rotated; 64-column heads; heads starting
# inside the output and stopping before its end
@pytest.mark.parametrize("T,N,K,col0,heads,hd,rd", [(1, 1024, 512, 0, 8, 128, 128), (33, 1024, 512, 0, 8, 128, 128),
                                                    (2, 768, 256, 64, 10, 64, 32), (77, 768, 256, 64, 10, 64, 32),
                                                    (200, 2048, 1024, 256, 5, 256, 96)])
def test_rope_layouts(nv, ws, T, N, K, col0, heads, hd, rd):
    run(nv, ws, T, N, K, col0, heads, hd, rd, False, seed=T + N + col0)


def test_rope_split_schedule(nv, ws):
    """A deep-K shape given the split workspace: at T=3 the tensor-core decode
    kernel, split along K over all SMs, its partials combined before the
    rotating epilogue."""
    run(nv, ws, 3, 1024, 16384, 0, 8, 128, 64, False, seed=99, split=True)


@pytest.mark.parametrize("T", [1, 8])
def test_rope_qkv_decode_tensor_cores(nv, ws, T):
    """The QKV projection at decode sizes with the split workspace (the
    tensor-core decode kernel's epilogue rotates)."""
    run(nv, ws, T, 7168, 5120, 0, 48, 128, 64, False, seed=40 + T, split=True)
