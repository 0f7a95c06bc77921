"""Oracle package -- TEST INFRASTRUCTURE, not part of the product.

Plain, slow, obviously correct CPU statements of the paged KV cache hot path:
  * ``oracle.c`` (fp64 C): paged decode attention, paged (chunked) prefill attention, KV
    append, copy-on-write block copy, KV bytes per token, and its own fp16 / bf16 decoders;
  * ``manager.py`` (Python): the block manager (free list, block tables, refcounts,
    prefix sharing, copy-on-write, admission in blocks).

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline / reference leg may
import this package. The product library never loads it, and it never loads the product.
Nothing here is shared with the CUDA path except the seeded input generators, which live in
a module of their own and contain none of the method's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

from .manager import BlockManagerOracle  # noqa: F401

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "_build" / "liboracle.so"

F32, F16, BF16 = 0, 1, 2  # the oracle's own dtype codes
_DTYPE_NAMES = {"f32": F32, "f16": F16, "bf16": BF16}

_lib = None


def build(force: bool = False) -> Path:
    """Compile oracle.c into _build/liboracle.so with gcc (OpenMP when available)."""
    if not force and _LIB.exists() and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    _LIB.parent.mkdir(parents=True, exist_ok=True)
    tmp = _LIB.with_suffix(f".{os.getpid()}.tmp")
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", str(_SRC), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        # PKV_ORACLE_LIB names another build of oracle.c to load instead (the mutation tests point
        # it at copies with a planted mistake, to show that the pins reject them)
        override = os.environ.get("PKV_ORACLE_LIB")
        path = Path(override) if override else build()
        L = ctypes.CDLL(str(path))
        vp, i32p, i64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
        L.oracle_paged_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            vp, vp, vp, i32p, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_double,
            ctypes.POINTER(ctypes.c_double), ctypes.c_int]
        L.oracle_paged_decode.restype = ctypes.c_int
        L.oracle_paged_prefill.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            vp, vp, vp, i32p, ctypes.c_int, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.POINTER(ctypes.c_double), ctypes.c_int]
        L.oracle_paged_prefill.restype = ctypes.c_int
        L.oracle_kv_append.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            vp, vp, i64p, ctypes.c_int, vp, vp]
        L.oracle_kv_append.restype = ctypes.c_int
        L.oracle_copy_blocks.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            vp, vp, i32p, ctypes.c_int]
        L.oracle_copy_blocks.restype = ctypes.c_int
        L.oracle_kv_bytes_per_token.argtypes = [ctypes.c_int] * 4
        L.oracle_kv_bytes_per_token.restype = ctypes.c_uint64
        L.oracle_elem_to_double.argtypes = [ctypes.c_int, vp, ctypes.c_size_t]
        L.oracle_elem_to_double.restype = ctypes.c_double
        L.oracle_elems_to_double.argtypes = [ctypes.c_int, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_double)]
        L.oracle_elems_to_double.restype = None
        L.oracle_max_threads.argtypes = []
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _code(dtype) -> int:
    return _DTYPE_NAMES[dtype] if isinstance(dtype, str) else int(dtype)


def _raw(a: np.ndarray, elem_bytes: int) -> np.ndarray:
    """A C-contiguous view whose buffer holds the elements' raw bytes."""
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize != elem_bytes:
        raise TypeError(f"expected {elem_bytes}-byte elements, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def elem_bytes(dtype) -> int:
    return 4 if _code(dtype) == F32 else 2


def paged_decode(dtype, q, k_pool, v_pool, tables, lens, scale, n_threads: int = 1) -> np.ndarray:
    """fp64 paged decode attention for one layer.

    q [n_seqs, n_q, d]; k_pool, v_pool [num_blocks, n_kv, block_size, d] (float32 for "f32",
    float16 for "f16", uint16 bit patterns for "bf16"); tables [n_seqs, max_blocks] int;
    lens [n_seqs] int. Returns float64 [n_seqs, n_q, d].
    """
    code = _code(dtype)
    eb = elem_bytes(code)
    q, k_pool, v_pool = _raw(q, eb), _raw(k_pool, eb), _raw(v_pool, eb)
    tables, lens = _i32(tables), _i32(lens)
    n_seqs, n_q, d = q.shape
    num_blocks, n_kv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    if tables.ndim != 2 or tables.shape[0] != n_seqs or lens.shape != (n_seqs,):
        raise ValueError("tables / lens shape mismatch")
    out = np.zeros((n_seqs, n_q, d), dtype=np.float64)
    rc = lib().oracle_paged_decode(
        code, n_q, n_kv, d, bs, num_blocks, _ptr(q), _ptr(k_pool), _ptr(v_pool),
        tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), tables.shape[1],
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n_seqs, float(scale),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_paged_decode refused its arguments")
    return out


def paged_prefill(dtype, q, k_pool, v_pool, tables, lens, query_start, scale, n_threads: int = 1) -> np.ndarray:
    """fp64 paged prefill attention for one layer (causal chunk of new tokens per sequence).

    q [n_tokens, n_q, d]; pools, tables and lens as paged_decode; query_start [n_seqs + 1]:
    the tokens of sequence s are q rows query_start[s] .. query_start[s+1]-1, at positions
    lens[s] - n_s .. lens[s] - 1. Returns float64 [n_tokens, n_q, d] (rows of no sequence: 0).
    """
    code = _code(dtype)
    eb = elem_bytes(code)
    q, k_pool, v_pool = _raw(q, eb), _raw(k_pool, eb), _raw(v_pool, eb)
    tables, lens, query_start = _i32(tables), _i32(lens), _i32(query_start)
    n_tokens, n_q, d = q.shape
    num_blocks, n_kv, bs, d2 = k_pool.shape
    n_seqs = lens.shape[0]
    assert d2 == d and v_pool.shape == k_pool.shape
    if tables.ndim != 2 or tables.shape[0] != n_seqs or query_start.shape != (n_seqs + 1,):
        raise ValueError("tables / lens / query_start shape mismatch")
    out = np.zeros((n_tokens, n_q, d), dtype=np.float64)
    rc = lib().oracle_paged_prefill(
        code, n_q, n_kv, d, bs, num_blocks, _ptr(q), _ptr(k_pool), _ptr(v_pool),
        tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), tables.shape[1],
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        query_start.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n_seqs, n_tokens, float(scale),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_paged_prefill refused its arguments")
    return out


def kv_append(k, v, slots, k_pool, v_pool) -> None:
    """In-place byte copy of k, v [n_tok, n_kv, d] into one layer's host pools."""
    eb = k.dtype.itemsize
    k, v = _raw(k, eb), _raw(v, eb)
    slots = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    if not (k_pool.flags.c_contiguous and v_pool.flags.c_contiguous):
        raise ValueError("pools must be C-contiguous")
    num_blocks, n_kv, bs, d = k_pool.shape
    rc = lib().oracle_kv_append(eb, n_kv, d, bs, num_blocks, _ptr(k), _ptr(v),
                                slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(slots),
                                _ptr(k_pool), _ptr(v_pool))
    if rc != 0:
        raise ValueError("oracle_kv_append refused its arguments")


def copy_blocks(k_pool, v_pool, pairs) -> None:
    """In-place copy-on-write block copy over all layers. pools [L, num_blocks, n_kv, bs, d]."""
    pairs = _i32(pairs).reshape(-1, 2)
    if not (k_pool.flags.c_contiguous and v_pool.flags.c_contiguous):
        raise ValueError("pools must be C-contiguous")
    n_layers, num_blocks, n_kv, bs, d = k_pool.shape
    rc = lib().oracle_copy_blocks(k_pool.dtype.itemsize, n_layers, n_kv, d, bs, num_blocks,
                                  _ptr(k_pool), _ptr(v_pool),
                                  pairs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(pairs))
    if rc != 0:
        raise ValueError("oracle_copy_blocks refused its arguments")


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes_: int) -> int:
    return int(lib().oracle_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, elem_bytes_))


def elem_to_double(dtype, raw: np.ndarray, i: int) -> float:
    raw = np.ascontiguousarray(raw)
    return float(lib().oracle_elem_to_double(_code(dtype), _ptr(raw), i))


def elems_to_double(dtype, raw: np.ndarray) -> np.ndarray:
    """Decode every element of a raw array (float32 / float16 / uint16 bf16 bits) to float64."""
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, dtype=np.float64)
    lib().oracle_elems_to_double(_code(dtype), _ptr(raw), raw.size,
                                 out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out.reshape(raw.shape)


def max_threads() -> int:
    return int(lib().oracle_max_threads())
