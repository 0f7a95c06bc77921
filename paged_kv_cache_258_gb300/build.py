"""Builds libpkv.so in-tree: CUDA sources for sm_103a plus the host C block manager.

Translation units compile in parallel (nvcc / gcc), then nvcc links one shared library with a
static CUDA runtime. A stamp of the sources and flags skips work when nothing changed.
Set PKV_PTXAS_VERBOSE=1 to record ptxas register / shared-memory reports in _build/ptxas.txt.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
BUILD = PKG / "_build"
LIB = PKG / "libpkv.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", str(INCLUDE), "-I", str(CSRC)]
CC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-Wall", "-I", str(INCLUDE)]


def _nvcc() -> str:
    return shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


def _sources():
    cu = sorted(CSRC.glob("*.cu"))
    c = sorted(CSRC.glob("*.c"))
    headers = sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))
    return cu, c, headers


def _stamp(verbose: bool) -> str:
    cu, c, headers = _sources()
    h = hashlib.sha256()
    for p in cu + c + headers:
        h.update(p.name.encode())
        h.update(p.read_bytes())
    h.update(" ".join(NVCC_FLAGS + CC_FLAGS).encode())
    h.update(b"v" if verbose else b"q")
    return h.hexdigest()


def build(force: bool = False) -> Path:
    """Compile and link libpkv.so if sources changed; returns its path."""
    verbose = os.environ.get("PKV_PTXAS_VERBOSE") == "1"
    stamp = _stamp(verbose)
    stamp_file = BUILD / "stamp"
    if not force and LIB.exists() and stamp_file.exists() and stamp_file.read_text() == stamp:
        return LIB
    BUILD.mkdir(parents=True, exist_ok=True)
    cu, c, _ = _sources()
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_cu(src: Path):
        obj = BUILD / (src.stem + ".o")
        r = subprocess.run([nvcc, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)],
                           capture_output=True, text=True)
        return src, obj, r

    def compile_c(src: Path):
        obj = BUILD / (src.stem + ".c.o")
        r = subprocess.run(["gcc", *CC_FLAGS, "-c", str(src), "-o", str(obj)], capture_output=True, text=True)
        return src, obj, r

    objs, reports = [], []
    with cf.ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as ex:
        futs = [ex.submit(compile_cu, s) for s in cu] + [ex.submit(compile_c, s) for s in c]
        for f in futs:
            src, obj, r = f.result()
            if r.returncode != 0:
                raise RuntimeError(f"compiling {src.name} failed:\n{r.stdout}\n{r.stderr}")
            objs.append(obj)
            reports.append(f"== {src.name}\n{r.stderr}")
    if verbose:
        (BUILD / "ptxas.txt").write_text("\n".join(reports))
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp.so")
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking libpkv.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    stamp_file.write_text(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
