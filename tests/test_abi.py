"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every function include/nvfp4.h declares, its size helpers agree with
the documented layout, and invalid arguments are rejected before any CUDA
call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from nvfp4_block_scaled_device_gb300 import build
    build.build()
    import nvfp4_block_scaled_device_gb300 as nv
    return nv.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_four_path_entry_points():
    names = header_functions()
    for n in ("nvfp4_amax_scale", "nvfp4_quantize", "nvfp4_gemm", "nvfp4_mlp"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    names = header_functions()
    assert names
    for n in names:
        assert hasattr(L, n), n
    import nvfp4_block_scaled_device_gb300 as nv
    assert set(names) == set(nv.EXPORTED_FUNCTIONS)


def test_size_helpers(L):
    import nvfp4_block_scaled_device_gb300 as nv
    assert nv.codes_bytes(16, 256) == 16 * 128
    assert nv.sf_bytes(16, 256) == 128 * 16
    assert nv.sf_bytes(128, 64) == 128 * 4
    assert nv.sf_bytes(129, 5120) == 256 * 320
    assert nv.sf_bytes(1, 17408) == 128 * 1088
    assert nv.amax_workspace_bytes() >= 256
    assert nv.gemm_workspace_bytes() >= 8192            # ready flags (+ partial slots with a device)
    assert nv.swiglu_workspace_bytes(1024, 17408, nv.NVFP4_INTER_DYNAMIC) >= 1024 * 17408 * 2
    assert nv.mlp_workspace_bytes(1024, 5120, 17408, nv.NVFP4_INTER_STATIC) >= (
        1024 * 2560 + 1024 * 320 + 1024 * 8704 + 1024 * 1088)


def test_status_strings(L):
    for s in range(7):
        assert L.nvfp4_status_string(s)
    assert L.nvfp4_status_string(0) == b"ok"


def test_invalid_arguments_rejected_on_host(L):
    import nvfp4_block_scaled_device_gb300 as nv
    NULL = None
    # NULL tensors
    assert L.nvfp4_gemm(NULL, NULL, NULL, 0, NULL, 0, NULL, 0, NULL) == 1
    # bad shapes: cols not a multiple of 64
    a = nv._TensorC(16, 128 * 16, 4, 16, 100, 64)
    w = nv._TensorC(16, 128 * 16, 4, 512, 100, 64)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(w), 16, 512, NULL, 0, NULL, 0, NULL) == 1
    # misaligned codes pointer
    a = nv._TensorC(17, 128 * 16, 4, 16, 256, 128)
    w = nv._TensorC(16, 128 * 16, 4, 512, 256, 128)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(w), 16, 512, NULL, 0, NULL, 0, NULL) == 2
    # K mismatch
    a = nv._TensorC(16, 128 * 16, 4, 16, 256, 128)
    w = nv._TensorC(16, 128 * 16, 4, 512, 512, 256)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(w), 16, 512, NULL, 0, NULL, 0, NULL) == 1
    # quantize: cols % 64
    assert L.nvfp4_quantize(16, 4, 32, 32, NULL, 1e-6, 16, 16, 16, 128, NULL, NULL) == 1
    # amax: missing workspace
    assert L.nvfp4_amax_scale(16, 4, 64, 64, NULL, 1e-6, 16, NULL, 0, NULL) == 5
    # gemm_rope: no embedding, odd column, rotated heads past N, rope_dim > head_dim, misaligned table
    a = nv._TensorC(16, 128 * 16, 4, 16, 256, 128)
    w = nv._TensorC(16, 128 * 16, 4, 512, 256, 128)
    assert L.nvfp4_gemm_rope(ctypes.byref(a), ctypes.byref(w), 16, 512, NULL, NULL, 0, NULL) == 1
    for bad in (dict(col0=1), dict(heads=5), dict(rope_dim=256), dict(rope_dim=3), dict(table_ld=31)):
        f = dict(pos=16, cos_t=16, sin_t=16, table_ld=32, positions=8, col0=0, heads=4, head_dim=128, rope_dim=64,
                 inverse=0)
        f.update(bad)
        r = nv._RopeC(**f)
        assert L.nvfp4_gemm_rope(ctypes.byref(a), ctypes.byref(w), 16, 512, ctypes.byref(r), NULL, 0, NULL) == 1, bad
    r = nv._RopeC(pos=16, cos_t=18, sin_t=16, table_ld=32, positions=8, col0=0, heads=4, head_dim=128, rope_dim=64)
    assert L.nvfp4_gemm_rope(ctypes.byref(a), ctypes.byref(w), 16, 512, ctypes.byref(r), NULL, 0, NULL) == 2
    # mlp: bad inter mode
    t = nv._TensorC(16, 128, 4, 256, 256, 128)
    assert L.nvfp4_mlp(16, 4, 256, 256, 16, 1e-6, ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), 7, 16,
                       16, 256, 1, 256, 1 << 30, NULL) == 1


def test_python_binding_fails_loudly_without_library(tmp_path):
    import nvfp4_block_scaled_device_gb300 as nv
    with pytest.raises(RuntimeError):
        nv.lib(str(tmp_path / "missing.so"))


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "nvfp4_block_scaled_device_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), f
                assert "liboracle" not in src and "nvfp4_oracle" not in src, f


def test_experts_arguments_rejected_on_host(L):
    import nvfp4_block_scaled_device_gb300 as nv
    NULL = None
    a = nv._TensorC(16, 128 * 16, 4, 16, 256, 128)
    w = nv._TensorC(16, 128 * 16, 4, 4 * 256, 256, 128)
    ids = ctypes.c_void_p(256)
    # N = rows / E must be a multiple of 128; E >= 1; ids non-null
    assert L.nvfp4_gemm_experts(ctypes.byref(a), ctypes.byref(w), 16, ids, 2, 16, 128, NULL, 0, NULL) == 1
    assert L.nvfp4_gemm_experts(ctypes.byref(a), ctypes.byref(w), 0, ids, 2, 16, 128, NULL, 0, NULL) == 1
    assert L.nvfp4_gemm_experts(ctypes.byref(a), ctypes.byref(w), 4, NULL, 2, 16, 128, NULL, 0, NULL) == 1
    # no workspace
    assert L.nvfp4_gemm_experts(ctypes.byref(a), ctypes.byref(w), 4, ids, 2, 16, 256, NULL, 0, NULL) == 5
    # workspace size: routed rows padded per expert, codes + scales per row
    b = nv.experts_workspace_bytes(16, 2, 256, 4)
    assert b >= (32 + 127 * 4) // 128 * 128 * (128 + 16)
    assert nv.experts_workspace_bytes(0, 2, 256, 4) == 0


def test_noalloc_argument_errors_before_any_cuda_call(L):
    """nvfp4_mlp_noalloc returns nvfp4_mlp's argument statuses, and refuses an
    oversized request, before it looks up or clears its fixed array (no CUDA
    call: these run on a machine without a GPU)."""
    import nvfp4_block_scaled_device_gb300 as nv
    NULL = None
    H, I = 256, 512
    g = nv._TensorC(16, 256, 4, I, H, H // 2)      # gate / up [I x H]
    d = nv._TensorC(16, 256, 4, H, I, I // 2)      # down [H x I]
    call = lambda x, T, wg, wu, wd, mode, gi, out: L.nvfp4_mlp_noalloc(
        x, T, H, H, 16, 1e-6, ctypes.byref(wg), ctypes.byref(wu) if wu is not None else NULL, ctypes.byref(wd),
        mode, gi, out, H, 1, NULL)
    assert call(16, 4, g, None, d, 0, 16, 16) == 1           # missing W_up
    assert call(16, 4, g, g, d, 7, 16, 16) == 1              # bad intermediate-scale mode
    assert call(16, 4, g, g, d, 0, NULL, 16) == 1            # missing g_inter
    assert call(18, 4, g, g, d, 0, 16, 16) == 2              # misaligned x
    bad = nv._TensorC(16, 256, 4, I, H + 64, (H + 64) // 2)
    assert call(16, 4, bad, bad, d, 0, 16, 16) == 1          # gate cols != H
    # larger than the fixed array (valid arguments otherwise): NVFP4_ERR_WORKSPACE
    Hb, Ib = 5120, 17408
    gb = nv._TensorC(16, 256, 4, Ib, Hb, Hb // 2)
    db = nv._TensorC(16, 256, 4, Hb, Ib, Ib // 2)
    st = L.nvfp4_mlp_noalloc(16, 705, Hb, Hb, 16, 1e-6, ctypes.byref(gb), ctypes.byref(gb), ctypes.byref(db),
                             nv.NVFP4_INTER_DYNAMIC, 16, 16, Hb, 1, NULL)
    assert st == 5
    assert L.nvfp4_noalloc_scratch(NULL, NULL) == 1
