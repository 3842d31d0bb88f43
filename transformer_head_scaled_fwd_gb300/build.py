"""Build the CUDA library ``libmha.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc to an object in parallel, then the
objects are linked into ``transformer_head_scaled_fwd_gb300/libmha.so``
(static CUDA runtime, no libcuda link: the tensor-map encoder is fetched from
the driver at run time). Rebuilds only when a source or header is newer than
the library.

``build(debug=True)`` builds ``libmha_debug.so`` instead: the same sources with
MHA_DEVICE_CHECKS defined, so the kernels check their block and tile indices at
entry and record a status code (mha_check_device_status) instead of touching
memory when one falls outside the problem.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmha.so")
LIB_DEBUG = os.path.join(PKG, "libmha_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libmha.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(CSRC, "*.inc")) + [os.path.join(ROOT, "include", "mha.h"), __file__])


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not needs_build(lib):
        return lib
    out_dir = BUILD + ("_debug" if debug else "")
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = list(extra_flags) + (["-DMHA_DEVICE_CHECKS"] if debug else [])
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include"), *flags]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    flags = ["-Xptxas", "-v"] if v else []
    print(build(force=True, verbose=v, extra_flags=flags))
