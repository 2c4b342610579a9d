"""Python binding of libnvfp4.so (include/nvfp4.h): the NVFP4 W4A4 linear
and MLP hot path on one sm_103a GPU.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  torch provides device memory and streams.  If the library has not
been built (``python -c "import __graft_entry__ as g; g.build()"``) every
call raises; there is no fallback.

Function names match the C ABI.  Tensors are CUDA torch tensors:
  bf16 matrices: torch.bfloat16, row-major (a row pitch is taken from
  ``stride(0)``); quantized matrices: :class:`NVFP4Tensor`.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4.so")

NVFP4_OK = 0
NVFP4_ERR_TIMEOUT = 6        # device-side: a bounded wait ran out (status word: 6 * 100 + site)
NVFP4_INTER_STATIC = 0
NVFP4_INTER_DYNAMIC = 1

_lock = threading.Lock()
_lib = None


class _TensorC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("g", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


class _RopeC(ctypes.Structure):
    _fields_ = [("pos", ctypes.c_void_p), ("cos_t", ctypes.c_void_p), ("sin_t", ctypes.c_void_p),
                ("table_ld", ctypes.c_int64), ("positions", ctypes.c_int64), ("col0", ctypes.c_int64),
                ("heads", ctypes.c_int64), ("head_dim", ctypes.c_int64), ("rope_dim", ctypes.c_int64),
                ("inverse", ctypes.c_int)]


_SIGS = {
    "nvfp4_codes_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "nvfp4_sf_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "nvfp4_amax_workspace_bytes": (ctypes.c_size_t, []),
    "nvfp4_gemm_workspace_bytes": (ctypes.c_size_t, []),
    "nvfp4_swiglu_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
    "nvfp4_mlp_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
    "nvfp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "nvfp4_mma_issue_rate": (ctypes.c_int, [ctypes.POINTER(ctypes.c_double)]),
    "nvfp4_noalloc_scratch": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_size_t)]),
    "nvfp4_experts_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                        ctypes.c_int64]),
    "nvfp4_gemm_experts": (ctypes.c_int, [ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC), ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nvfp4_amax_scale": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]),
    "nvfp4_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "nvfp4_scale_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                            ctypes.c_void_p]),
    "nvfp4_gemm": (ctypes.c_int, [ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC), ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                  ctypes.c_size_t, ctypes.c_void_p]),
    "nvfp4_gemm_rope": (ctypes.c_int, [ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC), ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.POINTER(_RopeC), ctypes.c_void_p, ctypes.c_size_t,
                                       ctypes.c_void_p]),
    "nvfp4_gemm_swiglu": (ctypes.c_int, [ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC),
                                         ctypes.POINTER(_TensorC), ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nvfp4_mlp": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(_TensorC),
                                 ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC), ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "nvfp4_mlp_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(_TensorC),
                                         ctypes.POINTER(_TensorC), ctypes.POINTER(_TensorC), ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_void_p]),
}

EXPORTED_FUNCTIONS = tuple(_SIGS)


def lib(path: str | None = None):
    """Load libnvfp4.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with nvfp4_block_scaled_device_gb300.build.build()")
            L = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return L
            _lib = L
    return _lib


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().nvfp4_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def _check(status: int, where: str):
    if status != NVFP4_OK:
        raise NVFP4Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16_2d(x: torch.Tensor, name: str):
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1 or not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA bf16 matrix with unit column stride")
    return x.shape[0], x.shape[1], x.stride(0)


# ------------------------------------------------------------ host helpers
def codes_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_codes_bytes(rows, cols))


def sf_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_sf_bytes(rows, cols))


def amax_workspace_bytes() -> int:
    return int(lib().nvfp4_amax_workspace_bytes())


def gemm_workspace_bytes() -> int:
    return int(lib().nvfp4_gemm_workspace_bytes())


def swiglu_workspace_bytes(T: int, I: int, inter_mode: int) -> int:
    return int(lib().nvfp4_swiglu_workspace_bytes(T, I, inter_mode))


def mlp_workspace_bytes(T: int, H: int, I: int, inter_mode: int) -> int:
    return int(lib().nvfp4_mlp_workspace_bytes(T, H, I, inter_mode))


def device_status(clear: bool = True) -> int:
    """Device-side status word (synchronous; diagnostics and tests)."""
    v = ctypes.c_int(0)
    _check(lib().nvfp4_device_status(ctypes.byref(v), int(clear)), "nvfp4_device_status")
    return v.value


def mma_issue_rate() -> float:
    """Multiply-adds per SM per clock of the GEMMs' block-scaled MMA form,
    measured on the current device (synchronous; a measurement diagnostic)."""
    v = ctypes.c_double(0.0)
    _check(lib().nvfp4_mma_issue_rate(ctypes.byref(v)), "nvfp4_mma_issue_rate")
    return v.value


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace buffer (torch's allocator aligns to >= 256 B)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


@dataclass
class NVFP4Tensor:
    """A quantized [rows x cols] matrix on the device: codes uint8 [rows, cols/2],
    swizzled scales uint8 [sf_bytes(rows, cols)], global scale float32 [1]."""
    codes: torch.Tensor
    sf: torch.Tensor
    g: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device=None) -> "NVFP4Tensor":
        device = device or "cuda"
        return NVFP4Tensor(
            codes=torch.empty((rows, cols // 2), dtype=torch.uint8, device=device),
            sf=torch.zeros((sf_bytes(rows, cols),), dtype=torch.uint8, device=device),
            g=torch.zeros((1,), dtype=torch.float32, device=device),
            rows=rows, cols=cols)

    def c(self) -> _TensorC:
        return _TensorC(self.codes.data_ptr(), self.sf.data_ptr(), self.g.data_ptr(),
                        self.rows, self.cols, self.codes.stride(0))


# -------------------------------------------------------------- the path
def nvfp4_amax_scale(x: torch.Tensor, g_out: torch.Tensor, ws: torch.Tensor, norm_w=None, eps=1e-6,
                     stream=None):
    rows, cols, ldx = _bf16_2d(x, "x")
    _check(lib().nvfp4_amax_scale(_ptr(x), rows, cols, ldx, _ptr(norm_w), eps, _ptr(g_out), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)), "nvfp4_amax_scale")


def nvfp4_quantize(x: torch.Tensor, g: torch.Tensor, out: NVFP4Tensor, norm_w=None, eps=1e-6, y_out=None,
                   stream=None):
    rows, cols, ldx = _bf16_2d(x, "x")
    _check(lib().nvfp4_quantize(_ptr(x), rows, cols, ldx, _ptr(norm_w), eps, _ptr(g), _ptr(out.codes),
                                out.codes.stride(0), _ptr(out.sf), _ptr(y_out), _stream(stream)),
           "nvfp4_quantize")


def nvfp4_scale_quantize(x: torch.Tensor, out: NVFP4Tensor, ws: torch.Tensor, norm_w=None, eps=1e-6, stream=None):
    """Global scale into out.g and quantization into out, in one launch."""
    rows, cols, ldx = _bf16_2d(x, "x")
    _check(lib().nvfp4_scale_quantize(_ptr(x), rows, cols, ldx, _ptr(norm_w), eps, _ptr(out.g), _ptr(out.codes),
                                      out.codes.stride(0), _ptr(out.sf), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "nvfp4_scale_quantize")


def quantize_new(x: torch.Tensor, ws: torch.Tensor, norm_w=None, eps=1e-6, stream=None) -> NVFP4Tensor:
    """Global scale + quantization of x into a newly allocated NVFP4Tensor."""
    t = NVFP4Tensor.empty(x.shape[0], x.shape[1], x.device)
    nvfp4_amax_scale(x, t.g, ws, norm_w, eps, stream)
    nvfp4_quantize(x, t.g, t, norm_w, eps, None, stream)
    return t


def nvfp4_gemm(A: NVFP4Tensor, W: NVFP4Tensor, out: torch.Tensor, residual=None, stream=None, workspace=None):
    """workspace: None, or a zero-filled uint8 tensor (see workspace()) of
    gemm_workspace_bytes() bytes that lets the GEMM split tiles over all SMs."""
    _, _, ldo = _bf16_2d(out, "out")
    ldr = _bf16_2d(residual, "residual")[2] if residual is not None else 0
    a, w = A.c(), W.c()
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().nvfp4_gemm(ctypes.byref(a), ctypes.byref(w), _ptr(out), ldo, _ptr(residual), ldr,
                            _ptr(workspace), nbytes, _stream(stream)), "nvfp4_gemm")


def nvfp4_gemm_rope(A: NVFP4Tensor, W: NVFP4Tensor, out: torch.Tensor, pos: torch.Tensor, cos_t: torch.Tensor,
                    sin_t: torch.Tensor, col0: int, heads: int, head_dim: int, rope_dim: int, inverse=False,
                    stream=None, workspace=None):
    """nvfp4_gemm with the rotary embedding in its epilogue.  pos: int32
    [M] on the device; cos_t, sin_t: float32 [positions, >= rope_dim/2] on
    the device (row-major, the same shape)."""
    _, _, ldo = _bf16_2d(out, "out")
    if pos.dtype != torch.int32 or cos_t.dtype != torch.float32 or sin_t.dtype != torch.float32:
        raise TypeError("pos must be int32, cos_t and sin_t float32")
    if cos_t.shape != sin_t.shape or cos_t.dim() != 2 or cos_t.stride(1) != 1 or sin_t.stride() != cos_t.stride():
        raise ValueError("cos_t and sin_t must be row-major 2-D tensors of one shape")
    r = _RopeC(pos.data_ptr(), cos_t.data_ptr(), sin_t.data_ptr(), cos_t.stride(0), cos_t.shape[0], col0, heads,
               head_dim, rope_dim, int(bool(inverse)))
    a, w = A.c(), W.c()
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().nvfp4_gemm_rope(ctypes.byref(a), ctypes.byref(w), _ptr(out), ldo, ctypes.byref(r),
                                 _ptr(workspace), nbytes, _stream(stream)), "nvfp4_gemm_rope")


def nvfp4_gemm_swiglu(A: NVFP4Tensor, W_gate: NVFP4Tensor, W_up: NVFP4Tensor, inter_mode: int,
                      g_inter: torch.Tensor, s_out: NVFP4Tensor, ws: torch.Tensor, s_bf16=None, stream=None):
    a, wg, wu = A.c(), W_gate.c(), W_up.c()
    _check(lib().nvfp4_gemm_swiglu(ctypes.byref(a), ctypes.byref(wg), ctypes.byref(wu), inter_mode,
                                   _ptr(g_inter), _ptr(s_out.codes), s_out.codes.stride(0), _ptr(s_out.sf),
                                   _ptr(s_bf16), _ptr(ws), ws.numel(), _stream(stream)), "nvfp4_gemm_swiglu")


def nvfp4_mlp_noalloc(x: torch.Tensor, norm_w: torch.Tensor, W_gate: NVFP4Tensor, W_up: NVFP4Tensor,
                      W_down: NVFP4Tensor, inter_mode: int, g_inter: torch.Tensor, out: torch.Tensor,
                      add_residual=True, eps=1e-6, stream=None):
    """nvfp4_mlp without a workspace (the library's fixed scratch array; for
    callers that cannot allocate device memory -- see include/nvfp4.h)."""
    T, H, ldx = _bf16_2d(x, "x")
    _, _, ldo = _bf16_2d(out, "out")
    wg, wu, wd = W_gate.c(), W_up.c(), W_down.c()
    _check(lib().nvfp4_mlp_noalloc(_ptr(x), T, H, ldx, _ptr(norm_w), eps, ctypes.byref(wg), ctypes.byref(wu),
                                   ctypes.byref(wd), inter_mode, _ptr(g_inter), _ptr(out), ldo,
                                   int(bool(add_residual)), _stream(stream)), "nvfp4_mlp_noalloc")


def noalloc_scratch():
    """(device address, bytes) of nvfp4_mlp_noalloc's fixed array on the
    current device (diagnostics and tests)."""
    p, n = ctypes.c_void_p(0), ctypes.c_size_t(0)
    _check(lib().nvfp4_noalloc_scratch(ctypes.byref(p), ctypes.byref(n)), "nvfp4_noalloc_scratch")
    return int(p.value or 0), int(n.value)


def nvfp4_mlp(x: torch.Tensor, norm_w: torch.Tensor, W_gate: NVFP4Tensor, W_up: NVFP4Tensor,
              W_down: NVFP4Tensor, inter_mode: int, g_inter: torch.Tensor, out: torch.Tensor,
              ws: torch.Tensor, add_residual=True, eps=1e-6, stream=None):
    T, H, ldx = _bf16_2d(x, "x")
    _, _, ldo = _bf16_2d(out, "out")
    wg, wu, wd = W_gate.c(), W_up.c(), W_down.c()
    _check(lib().nvfp4_mlp(_ptr(x), T, H, ldx, _ptr(norm_w), eps, ctypes.byref(wg), ctypes.byref(wu),
                           ctypes.byref(wd), inter_mode, _ptr(g_inter), _ptr(out), ldo, int(bool(add_residual)),
                           _ptr(ws), ws.numel(), _stream(stream)), "nvfp4_mlp")


def experts_workspace_bytes(T: int, topk: int, K: int, num_experts: int) -> int:
    return int(lib().nvfp4_experts_workspace_bytes(T, topk, K, num_experts))


def nvfp4_gemm_experts(A: NVFP4Tensor, W: NVFP4Tensor, num_experts: int, ids: torch.Tensor, out: torch.Tensor,
                       ws: torch.Tensor, stream=None):
    """Expert-indexed GEMM.  W: the experts' weights stacked (rows = E * N,
    W.g fp32[E]); ids: CUDA int32 [T, topk] (or [T * topk]); out: bf16
    [T * topk, N], row t * topk + j for token t, slot j."""
    if ids.dtype != torch.int32 or not ids.is_cuda or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous CUDA int32 tensor")
    topk = ids.shape[1] if ids.dim() == 2 else ids.numel() // A.rows
    _, _, ldo = _bf16_2d(out, "out")
    a, w = A.c(), W.c()
    _check(lib().nvfp4_gemm_experts(ctypes.byref(a), ctypes.byref(w), num_experts, _ptr(ids), topk, _ptr(out), ldo,
                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "nvfp4_gemm_experts")
