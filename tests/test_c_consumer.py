"""The C ABI from a plain C99 program (tests/c/ra_consumer.c): the header
compiles as C, the shared library links into a C program, and (on a GPU) a
bf16 ring forward called from C matches the fp64 oracle's ring."""
import os
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
LIBDIR = ROOT / "long_context_ra_gb300" / "_lib"
SRC = ROOT / "tests" / "c" / "ra_consumer.c"
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _lib():
    from long_context_ra_gb300.build import build
    build()
    return LIBDIR / "libra_gb300.so"


def _compile(out: Path, gpu: bool) -> None:
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", f"-I{ROOT / 'include'}",
           str(SRC), "-o", str(out), f"-L{LIBDIR}", "-lra_gb300", f"-Wl,-rpath,{LIBDIR}", "-lm"]
    if gpu:
        import __graft_entry__
        __graft_entry__._build_oracle()
        cmd[1:1] = ["-DRA_CONSUMER_GPU", f"-I{CUDA / 'include'}"]
        cmd += [f"-L{CUDA / 'lib64'}", "-lcudart", f"-L{ROOT / 'oracle'}", "-lra_oracle",
                f"-Wl,-rpath,{ROOT / 'oracle'}", f"-Wl,-rpath,{CUDA / 'lib64'}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not found")
def test_c_program_validates_without_a_device(tmp_path):
    _lib()
    exe = tmp_path / "ra_consumer"
    _compile(exe, gpu=False)
    r = subprocess.run([str(exe), "cpu"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("ok")


@pytest.mark.gpu
def test_c_program_forward_matches_the_oracle(tmp_path):
    _lib()
    exe = tmp_path / "ra_consumer_gpu"
    _compile(exe, gpu=True)
    r = subprocess.run([str(exe), "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
