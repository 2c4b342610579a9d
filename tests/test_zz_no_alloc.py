"""nvfp4_mlp_noalloc: the MLP for callers that cannot allocate device memory
(for example a plugin holding only borrowed tensor pointers, or a caller that
cannot afford cudaMalloc's device-wide synchronisation).  Its intermediates
live in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against nvfp4_mlp (which takes a workspace) on the
same inputs, within the MLP tolerance of the other tests, on two calls in a
row (the array keeps the previous call's contents), in both intermediate-
scale modes; after the array's amax and flag words were left dirty, as a
call that stopped early may leave them, at full size with the GEMMs using
the array's split-schedule slots (T=1: the tensor-core decode GEMMs' tickets
and partials; T=512: the down projection's split schedule); and a request
larger than the array is refused without work.
This file sorts last so a stop-at-first-failure run has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from _gpu import ELEM_REL, REL_FROB, dev, quantize_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_device_gb300 as m
    return m


def close(a: torch.Tensor, b: torch.Tensor):
    """Within the tolerance the MLP tests use (elementwise 2^-7 relative plus
    a floor, and the relative Frobenius bound)."""
    x = a.double().cpu().numpy()
    y = b.double().cpu().numpy()
    err = np.abs(x - y)
    assert np.all(err <= ELEM_REL * np.abs(y) + 1e-3 * np.abs(y).mean()), err.max()
    assert np.linalg.norm(x - y) <= REL_FROB * np.linalg.norm(y)


@pytest.mark.parametrize("T,H,I,mode", [(33, 512, 1024, 0), (130, 1024, 2048, 1), (256, 5120, 17408, 0)])
def test_noalloc_matches_workspace_mlp(nv, T, H, I, mode):
    rng = np.random.default_rng(T + H)
    ws = nv.workspace(256)
    x = dev(synthetic.normal(rng, (T, H)))
    nw = dev(synthetic.normal(rng, (H,), mean=1.0, std=0.05))
    Wg = quantize_gpu(synthetic.normal(rng, (I, H), std=0.02), ws)
    Wu = quantize_gpu(synthetic.normal(rng, (I, H), std=0.02), ws)
    Wd = quantize_gpu(synthetic.normal(rng, (H, I), std=0.02), ws)
    g_ref = torch.full((1,), 0.004, dtype=torch.float32, device="cuda")
    ref = torch.empty_like(x)
    mws = nv.workspace(nv.mlp_workspace_bytes(T, H, I, mode))
    nv.nvfp4_mlp(x, nw, Wg, Wu, Wd, mode, g_ref, ref, mws)
    for call in range(2):           # the array keeps the previous call's contents
        g = torch.full((1,), 0.004, dtype=torch.float32, device="cuda")
        out = torch.full_like(x, float("nan"))
        nv.nvfp4_mlp_noalloc(x, nw, Wg, Wu, Wd, mode, g, out)
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        assert torch.isfinite(out.float()).all(), call
        close(out, ref)
        assert g.item() == g_ref.item()


class _DeviceBytes:
    """A torch view of device bytes at a raw address (CUDA array interface)."""

    def __init__(self, addr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (addr, False), "version": 3}


@pytest.mark.parametrize("T", [1, 512])
def test_noalloc_recovers_dirty_words_and_uses_split_slots(nv, T):
    H, I = 5120, 17408
    rng = np.random.default_rng(900 + T)
    ws = nv.workspace(256)
    x = dev(synthetic.normal(rng, (T, H)))
    nw = dev(synthetic.normal(rng, (H,), mean=1.0, std=0.05))
    Wg = quantize_gpu(synthetic.normal(rng, (I, H), std=0.02), ws)
    Wu = quantize_gpu(synthetic.normal(rng, (I, H), std=0.02), ws)
    Wd = quantize_gpu(synthetic.normal(rng, (H, I), std=0.02), ws)
    g_ref = torch.full((1,), 0.004, dtype=torch.float32, device="cuda")
    ref = torch.empty_like(x)
    mode = nv.NVFP4_INTER_STATIC
    nv.nvfp4_mlp(x, nw, Wg, Wu, Wd, mode, g_ref, ref, nv.workspace(nv.mlp_workspace_bytes(T, H, I, mode)))
    # the split slots fit in the array next to the intermediates
    addr, n = nv.noalloc_scratch()
    assert addr != 0 and n == 32 << 20
    base = nv.mlp_workspace_bytes(T, H, I, mode) - (nv.gemm_workspace_bytes() - 8192)
    assert base + (nv.gemm_workspace_bytes() - 8192) <= n
    words = torch.as_tensor(_DeviceBytes(addr, 256 + 8192), device="cuda")
    for call in range(2):
        words.fill_(0xA5)              # amax words, flags and tickets left dirty
        out = torch.full_like(x, float("nan"))
        g = torch.full((1,), 0.004, dtype=torch.float32, device="cuda")
        nv.nvfp4_mlp_noalloc(x, nw, Wg, Wu, Wd, mode, g, out)
        torch.cuda.synchronize()
        assert nv.device_status() == 0
        assert torch.isfinite(out.float()).all(), call
        close(out, ref)
        assert int(words[256:].count_nonzero()) == 0      # the call leaves its flag words zero


def test_noalloc_refuses_requests_beyond_the_array(nv):
    ws = nv.workspace(256)
    rng = np.random.default_rng(1)
    H, I = 256, 17408
    Wg = quantize_gpu(synthetic.normal(rng, (I, H), std=0.02), ws)
    Wd = quantize_gpu(synthetic.normal(rng, (H, I), std=0.02), ws)
    T = 2048                         # per-call bf16 SwiGLU output alone is 71 MB > 32 MiB
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(x, 7.0)
    g = torch.zeros(1, dtype=torch.float32, device="cuda")
    wg, wu, wd = Wg.c(), Wg.c(), Wd.c()
    st = nv.lib().nvfp4_mlp_noalloc(ctypes.c_void_p(x.data_ptr()), T, H, H, ctypes.c_void_p(x.data_ptr()),
                                    1e-6, ctypes.byref(wg), ctypes.byref(wu), ctypes.byref(wd),
                                    nv.NVFP4_INTER_DYNAMIC, ctypes.c_void_p(g.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()), H, 1, None)
    assert st == 5                   # NVFP4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)     # nothing was enqueued
