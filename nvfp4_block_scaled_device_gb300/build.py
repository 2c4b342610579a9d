"""Build libnvfp4.so in-tree with nvcc for sm_103a (compute capability 10.3).

Each translation unit compiles in parallel to an object file under
``_build/``; the objects link into ``libnvfp4.so`` next to this file.  The
CUDA runtime is linked statically, so the library needs only the driver.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnvfp4.so")
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "gemm2.cu", "gemv.cu", "gemm_decode.cu", "noalloc.cu", "probe.cu", "experts.cu"]
HEADERS = ["common.cuh", "internal.h", "gemm_epilogue.cuh", "decode_epilogue.cuh", "gemv.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def flags(extra=()):
    return ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-O2",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _fingerprint(files, extra):
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(extra).encode())
    for f in files:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, extra_flags=(), out: str | None = None, verbose: bool = False) -> str:
    """Compile unless a library built from identical sources on this machine
    architecture exists; return the path of the library."""
    out = out or LIB
    build_dir = BUILD if out == LIB else out + ".objs"
    os.makedirs(build_dir, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "nvfp4.h"),
                                                                   os.path.abspath(__file__)]
    fp = _fingerprint(deps, [*flags(extra_flags), *ARCH])
    stamp = out + ".stamp"
    if not force and os.path.exists(out) and os.path.exists(stamp) and open(stamp).read() == fp:
        return out
    objs, jobs = [], []
    for src in SOURCES:
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        jobs.append([nvcc(), *flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", o])
    with cf.ThreadPoolExecutor(len(jobs)) as ex:
        for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            if verbose or res.returncode != 0:
                sys.stderr.write(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], check=True)
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(fp)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else ()))
