"""Build the CUDA library ``libgemm_rs.so`` in-tree for sm_103a.

    python -m tensor_gemm_reduce_tcgen05_gb300.build [--force] [--verbose-ptxas] [--checked]

``--checked`` builds ``libgemm_rs_checked.so`` instead: the same code compiled
with ``GEMM_RS_CHECKED``, whose kernels test every global access of the
epilogue and the folds against its buffer and report an access outside it
through the status word (a stand-in for a memory checker, for tests).

Each ``csrc/*.cu`` file is compiled to an object in parallel.  The objects are
then linked into a shared library next to this file.  The C ABI is declared
in ``include/gemm_rs.h``.  The library links the CUDA runtime dynamically, and
its rpath points at the toolkit's lib64.  If a process has already loaded
libcudart.so.13 (PyTorch does), the library uses that copy.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgemm_rs.so")
LIB_CHECKED = os.path.join(PKG, "libgemm_rs_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.isdir(home):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(_cuda_home(), "bin", "nvcc")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _up_to_date(lib: str) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose_ptxas: bool, checked: bool = False) -> str:
    out = os.path.join(BUILD, "checked") if checked else BUILD
    obj = os.path.join(out, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           "--expt-relaxed-constexpr", "-DGEMM_RS_BUILD", "-c", src, "-o", obj]
    if checked:
        cmd.insert(1, "-DGEMM_RS_CHECKED")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Compile (if needed) and return the path of libgemm_rs.so (or, with
    checked=True, of libgemm_rs_checked.so)."""
    lib = LIB_CHECKED if checked else LIB
    if not force and not verbose_ptxas and _up_to_date(lib):
        return lib
    os.makedirs(os.path.join(BUILD, "checked") if checked else BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, checked), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cuda_lib = os.path.join(_cuda_home(), "lib64")
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--checked", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, checked=args.checked))
