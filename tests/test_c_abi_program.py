"""The C ABI from plain C: tests/c_abi/kvl_c_check.c drives libkvl.so with cudaMalloc'd
buffers and compares every result with the oracle compiled into the same program.
Compiling it needs no GPU; running it does."""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _compile(out_dir: Path) -> Path:
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    lib_dir = kvl.LIB.parent
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = out_dir / "kvl_c_check"
    cmd = [cc, "-O1", "-Wall", "-Wextra", "-Werror", "-I", str(ROOT / "include"),
           "-I", str(CUDA / "include"), str(ROOT / "tests" / "c_abi" / "kvl_c_check.c"),
           str(ROOT / "oracle" / "kvl_oracle.c"), "-L", str(lib_dir), "-lkvl",
           "-L", str(CUDA / "lib64"), "-lcudart", f"-Wl,-rpath,{lib_dir}",
           f"-Wl,-rpath,{CUDA / 'lib64'}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_against_the_header(tmp_path):
    assert _compile(tmp_path).exists()


@pytest.mark.gpu
def test_c_program_matches_the_oracle(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c-abi: ok" in r.stdout
