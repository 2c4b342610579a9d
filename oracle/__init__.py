"""CPU oracle for the NVFP4 W4A4 linear / MLP path.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only users.  The CUDA library never
imports, links or calls anything here, and this package imports nothing from
the CUDA library.  The arithmetic lives in ``nvfp4_oracle.c`` (plain C,
binary32/binary64, no FMA contraction); this module only builds it with gcc
and marshals numpy arrays through ctypes.

All arrays are numpy: bf16 tensors are passed as ``uint16`` bit patterns,
FP4 codes as packed ``uint8`` [rows, cols/2], scales as LOGICAL ``uint8``
[rows, cols/16] (use :func:`sf_swizzle` for the MMA layout).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
          "-shared", "-fPIC", "-Wall", "-Wno-unknown-pragmas"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (seconds) unless a library built from the
    same source on this machine architecture exists.  Returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    h = hashlib.sha256(platform.machine().encode() + " ".join(CFLAGS).encode())
    with open(_SRC, "rb") as f:
        h.update(f.read())
    stamp = _LIB_PATH + ".stamp"
    fp = h.hexdigest()
    if force or not os.path.exists(_LIB_PATH) or not os.path.exists(stamp) or open(stamp).read() != fp:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
        with open(stamp, "w") as f:
            f.write(fp)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, f32, f64, vp, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            sig = {
                "oracle_bf16_value": (f64, [ctypes.c_uint16]),
                "oracle_bf16_from_double": (ctypes.c_uint16, [f64]),
                "oracle_e2m1_value": (f64, [i32]),
                "oracle_e2m1_encode": (i32, [f32]),
                "oracle_e4m3_value": (f64, [i32]),
                "oracle_e4m3_encode": (i32, [f32]),
                "oracle_amax_bf16": (f32, [vp, i64, i64, i64]),
                "oracle_global_scale_from_amax": (f32, [f32]),
                "oracle_global_scale": (f32, [vp, i64, i64, i64]),
                "oracle_quantize": (None, [vp, i64, i64, i64, f32, vp, vp]),
                "oracle_dequant_element": (f64, [vp, vp, i64, f32, i64, i64]),
                "oracle_sf_padded_rows": (i64, [i64]),
                "oracle_sf_padded_cols": (i64, [i64]),
                "oracle_sf_offset": (i64, [i64, i64, i64]),
                "oracle_sf_swizzle": (None, [vp, i64, i64, vp]),
                "oracle_sf_unswizzle": (None, [vp, i64, i64, vp]),
                "oracle_dot_sampled": (None, [vp, vp, vp, vp, i64, vp, vp, i64, vp, vp]),
                "oracle_gemm": (None, [vp, vp, f32, vp, vp, f32, i64, i64, i64, vp, i64, vp, vp, vp, i64]),
                "oracle_rmsnorm": (None, [vp, i64, i64, i64, vp, f32, vp, i64]),
                "oracle_swiglu1": (ctypes.c_uint16, [ctypes.c_uint16, ctypes.c_uint16]),
                "oracle_swiglu": (None, [vp, vp, i64, vp]),
                "oracle_rope": (None, [vp, i64, i64, i64, vp, vp, vp, i64, i64, i64, i64, i64, i32, vp, i64]),
                "oracle_mlp": (None, [vp, i64, i64, i64, i64, vp, f32,
                                      vp, vp, f32, vp, vp, f32, vp, vp, f32,
                                      f32, i32, vp, i64,
                                      vp, vp, vp, vp, vp, vp, vp]),
                "oracle_num_threads": (i32, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(int(bits))


def bf16_from_double(v: float) -> int:
    return int(lib().oracle_bf16_from_double(float(v)))


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e2m1_encode(q: float) -> int:
    return int(lib().oracle_e2m1_encode(float(q)))


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(int(byte))


def e4m3_encode(s: float) -> int:
    return int(lib().oracle_e4m3_encode(float(s)))


# ------------------------------------------------------------ global scale
def amax(x_bits: np.ndarray) -> float:
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    return float(np.float32(lib().oracle_amax_bf16(_p(x), rows, cols, cols)))


def global_scale_from_amax(a: float) -> np.float32:
    return np.float32(lib().oracle_global_scale_from_amax(float(a)))


def global_scale(x_bits: np.ndarray) -> np.float32:
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    return np.float32(lib().oracle_global_scale(_p(x), rows, cols, cols))


# ---------------------------------------------------------------- quantize
def quantize(x_bits: np.ndarray, g: float):
    """bf16 [R, K] -> (codes uint8 [R, K/2], logical scales uint8 [R, K/16])."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.empty((rows, cols // 2), np.uint8)
    sf = np.empty((rows, cols // 16), np.uint8)
    lib().oracle_quantize(_p(x), rows, cols, cols, float(np.float32(g)), _p(codes), _p(sf))
    return codes, sf


def dequantize(codes: np.ndarray, sf: np.ndarray, g: float) -> np.ndarray:
    """Exact binary64 decode of a whole quantized matrix (small sizes)."""
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2
    L = lib()
    out = np.empty((rows, cols), np.float64)
    for r in range(rows):
        for k in range(cols):
            out[r, k] = L.oracle_dequant_element(_p(codes), _p(sf), cols, float(np.float32(g)), r, k)
    return out


# ----------------------------------------------------------------- layout
def sf_padded_shape(rows: int, kb: int):
    L = lib()
    return int(L.oracle_sf_padded_rows(rows)), int(L.oracle_sf_padded_cols(kb))


def sf_offset(r: int, c: int, kb: int) -> int:
    return int(lib().oracle_sf_offset(r, c, kb))


def sf_swizzle(logical: np.ndarray) -> np.ndarray:
    logical = _c(logical, np.uint8)
    rows, kb = logical.shape
    pr, pc = sf_padded_shape(rows, kb)
    out = np.empty(pr * pc, np.uint8)
    lib().oracle_sf_swizzle(_p(logical), rows, kb, _p(out))
    return out


def sf_unswizzle(swz: np.ndarray, rows: int, kb: int) -> np.ndarray:
    swz = _c(swz, np.uint8).reshape(-1)
    out = np.empty((rows, kb), np.uint8)
    lib().oracle_sf_unswizzle(_p(swz), rows, kb, _p(out))
    return out


# ------------------------------------------------------------------- GEMM
def dot_sampled(a_codes, a_sf, w_codes, w_sf, m_idx, n_idx):
    """Exact sum_k a[m,k] w[n,k] (no global scales) and sum_k |a w| at pairs."""
    a_codes, a_sf = _c(a_codes, np.uint8), _c(a_sf, np.uint8)
    w_codes, w_sf = _c(w_codes, np.uint8), _c(w_sf, np.uint8)
    m_idx, n_idx = _c(m_idx, np.int64), _c(n_idx, np.int64)
    K = a_codes.shape[1] * 2
    assert w_codes.shape[1] * 2 == K
    n = m_idx.size
    dot = np.empty(n, np.float64)
    adot = np.empty(n, np.float64)
    lib().oracle_dot_sampled(_p(a_codes), _p(a_sf), _p(w_codes), _p(w_sf), K,
                             _p(m_idx), _p(n_idx), n, _p(dot), _p(adot))
    return dot, adot


def gemm(a_codes, a_sf, g_a, w_codes, w_sf, g_w, residual=None):
    """Returns (ref fp64 [M,N], absref fp64 [M,N], out bf16 bits [M,N])."""
    a_codes, a_sf = _c(a_codes, np.uint8), _c(a_sf, np.uint8)
    w_codes, w_sf = _c(w_codes, np.uint8), _c(w_sf, np.uint8)
    M, N, K = a_codes.shape[0], w_codes.shape[0], a_codes.shape[1] * 2
    ref = np.empty((M, N), np.float64)
    absref = np.empty((M, N), np.float64)
    out = np.empty((M, N), np.uint16)
    res = _c(residual, np.uint16) if residual is not None else None
    lib().oracle_gemm(_p(a_codes), _p(a_sf), float(np.float32(g_a)), _p(w_codes), _p(w_sf),
                      float(np.float32(g_w)), M, N, K, _p(res), N if res is not None else 0,
                      _p(ref), _p(absref), _p(out), N)
    return ref, absref, out


def gemm_id(a_codes, a_sf, g_a, w_codes, w_sf, g_w, ids):
    """Expert-indexed GEMM (a mixture-of-experts layer's routed projection):
    for token t and routing slot j, row [t, j] is the GEMM row of A[t] with
    the weights of expert ids[t, j], with that expert's global scale:
      out[t, j, n] = bf16( fp32(g_a * g_w[e]) * sum_k A[t, k] W_e[n, k] ),  e = ids[t, j].
    w_codes uint8 [E, N, K/2], w_sf logical uint8 [E, N, K/16], g_w [E],
    ids int [T, k] in [0, E).  Each expert's rows go through `gemm`.
    Returns (ref fp64 [T, k, N], absref fp64 [T, k, N], out bf16 bits [T, k, N])."""
    ids = np.asarray(ids)
    T, kk = ids.shape
    E, N = w_codes.shape[0], w_codes.shape[1]
    assert ids.min() >= 0 and ids.max() < E and a_codes.shape[0] == T
    ref = np.zeros((T, kk, N), np.float64)
    absref = np.zeros((T, kk, N), np.float64)
    out = np.zeros((T, kk, N), np.uint16)
    for e in range(E):
        t_idx, j_idx = np.nonzero(ids == e)
        if t_idx.size == 0:
            continue
        r, ar, o = gemm(a_codes[t_idx], a_sf[t_idx], g_a, w_codes[e], w_sf[e], g_w[e])
        ref[t_idx, j_idx] = r
        absref[t_idx, j_idx] = ar
        out[t_idx, j_idx] = o
    return ref, absref, out


# --------------------------------------------------------- norm / SwiGLU
def rmsnorm(x_bits, w_bits, eps=1e-6):
    x = _c(x_bits, np.uint16)
    w = _c(w_bits, np.uint16)
    rows, cols = x.shape
    y = np.empty_like(x)
    lib().oracle_rmsnorm(_p(x), rows, cols, cols, _p(w), float(np.float32(eps)), _p(y), cols)
    return y


def swiglu(gate_bits, up_bits):
    g = _c(gate_bits, np.uint16)
    u = _c(up_bits, np.uint16)
    s = np.empty_like(g)
    lib().oracle_swiglu(_p(g), _p(u), g.size, _p(s))
    return s


def rope(y_bits, pos, cos_t, sin_t, col0, heads, head_dim, rope_dim, inverse=False):
    """Rotary embedding of bf16 rows y [rows, cols] (see oracle_rope): the
    `heads` heads of head_dim columns from column col0 get their last
    rope_dim columns rotated as (even, odd) pairs by the angles of table row
    pos[t] (cos_t, sin_t: float32 [positions, >= rope_dim/2])."""
    y = _c(y_bits, np.uint16)
    p = _c(pos, np.int32)
    ct = _c(cos_t, np.float32)
    st = _c(sin_t, np.float32)
    rows, cols = y.shape
    assert p.shape == (rows,) and ct.shape == st.shape and ct.shape[1] * 2 >= rope_dim
    assert rope_dim % 2 == 0 and 0 < rope_dim <= head_dim and col0 + heads * head_dim <= cols
    assert p.min() >= 0 and p.max() < ct.shape[0]
    out = np.empty_like(y)
    lib().oracle_rope(_p(y), rows, cols, cols, _p(p), _p(ct), _p(st), ct.shape[1], col0, heads, head_dim, rope_dim,
                      int(bool(inverse)), _p(out), cols)
    return out


def mlp(x_bits, norm_w_bits, wg, wu, wd, g_inter=None, add_residual=True, eps=1e-6):
    """Whole MLP block.  wg/wu/wd are (codes, logical_sf, g) triples.
    g_inter None -> per-call intermediate scale from this call's SwiGLU output.
    Returns dict with out and every stage."""
    x = _c(x_bits, np.uint16)
    nw = _c(norm_w_bits, np.uint16)
    T, H = x.shape
    I = wg[0].shape[0]
    out = np.empty((T, H), np.uint16)
    g_h = np.zeros(1, np.float32)
    hc = np.empty((T, H // 2), np.uint8)
    hs = np.empty((T, H // 16), np.uint8)
    s = np.empty((T, I), np.uint16)
    gi = np.zeros(1, np.float32)
    sc = np.empty((T, I // 2), np.uint8)
    ss = np.empty((T, I // 16), np.uint8)
    W = [(_c(c, np.uint8), _c(f, np.uint8), float(np.float32(g))) for (c, f, g) in (wg, wu, wd)]
    lib().oracle_mlp(_p(x), T, H, I, H, _p(nw), float(np.float32(eps)),
                     _p(W[0][0]), _p(W[0][1]), W[0][2],
                     _p(W[1][0]), _p(W[1][1]), W[1][2],
                     _p(W[2][0]), _p(W[2][1]), W[2][2],
                     -1.0 if g_inter is None else float(np.float32(g_inter)), int(bool(add_residual)),
                     _p(out), H, _p(g_h), _p(hc), _p(hs), _p(s), _p(gi), _p(sc), _p(ss))
    return dict(out=out, g_h=np.float32(g_h[0]), h_codes=hc, h_sf=hs, s=s,
                g_inter=np.float32(gi[0]), s_codes=sc, s_sf=ss)


def num_threads() -> int:
    return int(lib().oracle_num_threads())
