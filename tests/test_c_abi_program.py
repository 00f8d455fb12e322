"""The C ABI from plain C.

tests/c_abi/kvl_c_check.c drives libkvl.so with cudaMalloc'd buffers and compares every
result with the oracle compiled into the same program.
tests/c_abi/kvl_static_scratch_reset.c checks the static-scratch plan builder across a
cudaDeviceReset and under stream capture (a process of its own: the reset ends the
context, which no torch process could survive).
Compiling them needs no GPU; running them does."""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _compile(out_dir: Path, name: str = "kvl_c_check", with_oracle: bool = True) -> Path:
    import layer_wise_paged_gb300 as kvl
    kvl.build()
    lib_dir = kvl.LIB.parent
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = out_dir / name
    srcs = [str(ROOT / "tests" / "c_abi" / f"{name}.c")]
    if with_oracle:
        srcs.append(str(ROOT / "oracle" / "kvl_oracle.c"))
    cmd = [cc, "-O1", "-Wall", "-Wextra", "-Werror", "-I", str(ROOT / "include"),
           "-I", str(CUDA / "include"), *srcs, "-L", str(lib_dir), "-lkvl",
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


def test_static_scratch_reset_program_compiles(tmp_path):
    assert _compile(tmp_path, "kvl_static_scratch_reset", with_oracle=False).exists()


@pytest.mark.gpu
def test_static_scratch_plan_survives_a_device_reset_and_capture(tmp_path):
    """Two calls before a cudaDeviceReset and two after it (and one captured into a
    graph on each side) each give kvl_batch_plan's plan; a captured call that would use
    the address remembered from the old context is refused."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path, "kvl_static_scratch_reset", with_oracle=False)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "static-scratch-reset: ok" in r.stdout
