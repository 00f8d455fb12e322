"""Build libkvl.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

One translation unit per .cu file under csrc/, compiled in parallel, then linked
into ``layer_wise_paged_gb300/_build/libkvl.so`` against the shared CUDA runtime (the
one PyTorch also loads).  No cmake, no torch extension machinery.
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
LIB = BUILD / "libkvl.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = Path(cuda) / "bin" / "nvcc"
    return str(cand) if cand.exists() else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(CSRC.glob("*.cu"))


def _stale() -> bool:
    if not LIB.exists():
        return True
    newest = max(p.stat().st_mtime for p in list(CSRC.glob("*")) + list(INCLUDE.glob("*.h")))
    return LIB.stat().st_mtime < newest


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile every csrc/*.cu for sm_103a and link libkvl.so (skipped when fresh)."""
    if not force and not _stale():
        return LIB
    BUILD.mkdir(exist_ok=True)
    nvcc = _nvcc()
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", str(INCLUDE), "-I", str(CSRC)]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: Path) -> Path:
        obj = BUILD / (src.stem + ".o")
        subprocess.run([*common, "-c", str(src), "-o", str(obj)], check=True)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB.with_suffix(f".so.{os.getpid()}")
    cuda_lib = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda")) / "lib64"
    subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", *map(str, objs), "-o", str(tmp),
                    "-Xlinker", f"-rpath,{cuda_lib}"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
