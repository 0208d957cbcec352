"""Build the CUDA library ``_lib/libra_gb300.so`` in-tree with nvcc.

Each ``csrc/*.cu`` translation unit is compiled for sm_103a only, in
parallel, then linked into one shared library with a static CUDA runtime.
A rebuild happens only when a source, a header or the flags changed.

    python -m long_context_ra_gb300.build          # build if stale
    python -m long_context_ra_gb300.build --force  # rebuild
    python -m long_context_ra_gb300.build --ptxas  # print -Xptxas -v usage
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
LIBDIR = PKG / "_lib"
LIB = LIBDIR / "libra_gb300.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
          "-fvisibility=hidden", "-Xcompiler", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _fingerprint(extra: list[str]) -> str:
    h = hashlib.sha256()
    for f in sorted(list(CSRC.glob("*")) + list(INCLUDE.glob("*.h"))):
        if f.is_file():
            h.update(f.name.encode())
            h.update(f.read_bytes())
    h.update(" ".join(ARCH + CFLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, ptxas_verbose: bool = False, extra: list[str] | None = None) -> Path:
    extra = list(extra or [])
    if ptxas_verbose:
        extra += ["-Xptxas", "-v"]
    stamp = LIBDIR / ".fingerprint"
    fp = _fingerprint(extra)
    if not force and LIB.exists() and stamp.exists() and stamp.read_text() == fp:
        return LIB
    BUILD.mkdir(exist_ok=True)
    LIBDIR.mkdir(exist_ok=True)
    cc = nvcc()

    def compile_one(src: Path) -> tuple[Path, str]:
        obj = BUILD / (src.stem + ".o")
        cmd = [cc, *ARCH, *CFLAGS, *extra, "-c", str(src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    if ptxas_verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [str(o) for o, _ in results]
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    stamp.write_text(fp)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="show register/spill usage")
    args = ap.parse_args()
    print(build(force=args.force or args.ptxas, ptxas_verbose=args.ptxas))


if __name__ == "__main__":
    main()
