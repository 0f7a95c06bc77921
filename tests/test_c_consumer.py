"""The C ABI used from plain C (tests/c/pkv_c_consumer.c): the host block manager, pkv_kv_append
and the fused decode step called from a C program linked against libpkv.so and the CUDA runtime,
checked against the fp64 oracle (oracle/oracle.c) on host copies of the same rows.

Compiling it needs no GPU (it catches drift between include/pkv.h, the exported symbols and a C
caller); running it does.
"""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
SRC = ROOT / "tests" / "c" / "pkv_c_consumer.c"
PKG = ROOT / "paged_kv_cache_258_gb300"


def _cuda_root() -> Path:
    nvcc = shutil.which("nvcc")
    return Path(nvcc).resolve().parent.parent if nvcc else Path("/usr/local/cuda")


def _compile(out: Path) -> None:
    cuda = _cuda_root()
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", str(ROOT / "include"), "-I", str(cuda / "include"),
           str(SRC), str(ROOT / "oracle" / "oracle.c"), "-fopenmp", "-L", str(PKG), "-lpkv",
           "-L", str(cuda / "lib64"), "-lcudart", "-lm", f"-Wl,-rpath,{PKG}", "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_c_consumer_compiles_and_links(tmp_path):
    _compile(tmp_path / "pkv_c_consumer")


@pytest.mark.gpu
def test_c_consumer_matches_oracle(tmp_path):
    exe = tmp_path / "pkv_c_consumer"
    _compile(exe)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c consumer ok" in r.stdout
