"""Build the in-tree shared library ``libmoe_gb300.so`` with nvcc for sm_103a.

Each translation unit compiles in parallel; the library links the CUDA
runtime statically so that loading it needs no GPU. A rebuild happens only
when a source or header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = PKG / "libmoe_gb300.so"

SOURCES = ["api.cu", "route.cu", "route_dispatch.cu", "route_grouped.cu", "dispatch.cu", "combine.cu", "experts_simt.cu", "experts_tc.cu",
           "train_router.cu", "train_experts.cu", "experts_bwd_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-I", str(INCLUDE), "-I", str(CSRC)]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_gb300.so")
    return path


def _inputs() -> list[Path]:
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(CSRC.glob("*.h")) + \
        list(INCLUDE.glob("*.h")) + [Path(__file__)]


def needs_build() -> bool:
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    return any(p.stat().st_mtime > t for p in _inputs())


def _run(cmd: list[str]) -> str:
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    """Compile every CUDA source for sm_103a and link the shared library."""
    if not force and not needs_build():
        return LIB
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> tuple[str, str]:
        obj = BUILD / (Path(src).stem + ".o")
        out = _run([cc, *ARCH, *CFLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)])
        return str(obj), out

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    tmp = LIB.with_suffix(".so.tmp")
    _run([cc, *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *objs, "-lpthread", "-ldl", "-lrt"])
    os.replace(tmp, LIB)
    if verbose or ptxas_info:
        for _, out in results:
            if out.strip():
                print(out)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv))
