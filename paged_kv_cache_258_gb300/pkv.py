"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every compute step runs in the library's CUDA kernels; this module checks tensor placement,
dtype, contiguity and shape, passes ``data_ptr()`` and the current CUDA stream, and turns
status codes into exceptions. It never computes on the CPU and has no fallback: if
libpkv.so is missing it raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libpkv.so"

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_NO_BLOCKS, PKV_ERR_BAD_STATE, PKV_ERR_CUDA = range(6)
STATUS_NAMES = {0: "ok", 1: "invalid", 2: "unsupported", 3: "no_blocks", 4: "bad_state", 5: "cuda"}
PKV_DEV_BAD_BLOCK_ID, PKV_DEV_BAD_CONTEXT_LEN, PKV_DEV_BAD_SLOT, PKV_DEV_BAD_PAIR, PKV_DEV_WAIT_TIMEOUT = 1, 2, 4, 8, 16
PKV_DEV_BAD_QUERY_RANGE = 32
PKV_DECODE_OVERLAP_PREVIOUS = 1
PKV_PREFILL_OVERLAP_PREVIOUS = 1
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
BLOCK = 16


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


class CacheDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32)]

    @property
    def dtype_name(self) -> str:
        return {v: k for k, v in DTYPE_CODES.items()}[self.dtype]


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("free_blocks", "used_blocks", "n_seqs", "alloc_failures",
                                              "tail_waste_rows", "prefix_hits", "cow_copies", "append_oom")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None


def lib():
    """Load libpkv.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() (needs nvcc)")
    L = ctypes.CDLL(str(LIB_PATH))
    c_i32, c_i64, c_u32, c_u64, c_sz, vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64,
                                            ctypes.c_size_t, ctypes.c_void_p)
    dp = ctypes.POINTER(CacheDesc)
    sigs = {
        "pkv_status_str": (ctypes.c_char_p, [ctypes.c_int]),
        "pkv_validate_desc": (ctypes.c_int, [dp]),
        "pkv_bytes_per_token": (c_u64, [dp]),
        "pkv_pool_bytes": (c_u64, [dp]),
        "pkv_decode_workspace_bytes": (c_sz, [dp, c_i32, c_i32]),
        "pkv_decode_split_geometry": (ctypes.c_int, [dp, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_i32),
                                                     ctypes.POINTER(c_i32), ctypes.POINTER(c_sz)]),
        "pkv_decode_ctas_per_sm": (ctypes.c_int, [dp, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32)]),
        "pkv_prefill_wave_tokens": (ctypes.c_int, [dp, ctypes.POINTER(c_i32)]),
        "pkv_kv_append": (ctypes.c_int, [dp, c_i32, vp, vp, vp, c_i32, vp, vp, vp]),
        "pkv_paged_decode_attention": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, c_i32, vp, c_i32, ctypes.c_float,
                                                      vp, vp, c_sz, vp]),
        "pkv_paged_decode_append_attention": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, vp, vp, c_i32, vp, c_i32,
                                                             ctypes.c_float, vp, vp, c_sz, vp]),
        "pkv_paged_decode_append_attention_ex": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, vp, vp, c_i32, vp, c_i32,
                                                                ctypes.c_float, vp, vp, c_sz, c_u32, vp]),
        "pkv_paged_decode_attention_static": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, c_i32, vp, c_i32,
                                                             ctypes.c_float, vp, vp]),
        "pkv_dense_decode_attention": (ctypes.c_int, [dp, c_i32, vp, vp, vp, c_i32, vp, c_i32, ctypes.c_float,
                                                      vp, vp, c_sz, c_u32, vp]),
        "pkv_paged_prefill_attention": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, c_i32, vp, vp, c_i32, c_i32,
                                                       c_i32, ctypes.c_float, vp, vp]),
        "pkv_paged_prefill_attention_ex": (ctypes.c_int, [dp, c_i32, vp, vp, vp, vp, c_i32, vp, vp, c_i32, c_i32,
                                                          c_i32, ctypes.c_float, vp, c_u32, vp]),
        "pkv_copy_blocks": (ctypes.c_int, [dp, vp, vp, vp, c_i32, vp]),
        "pkv_upload_metadata": (ctypes.c_int, [vp, vp, c_sz, vp]),
        "pkv_get_device_status": (ctypes.c_int, [vp, ctypes.POINTER(c_u32)]),
        "pkv_launch_count": (c_u64, []),
        "pkv_hbm_read_probe": (ctypes.c_int, [vp, c_sz, vp, vp]),
        "pkv_selftest_wait_timeout": (ctypes.c_int, [vp]),
        "pkv_mgr_create": (vp, [c_i32, c_i32, vp]),
        "pkv_mgr_clone": (vp, [vp]),
        "pkv_mgr_destroy": (None, [vp]),
        "pkv_mgr_add_seq": (ctypes.c_int, [vp, c_i64, c_i32, c_i32, vp]),
        "pkv_mgr_fork": (ctypes.c_int, [vp, c_i64, c_i64]),
        "pkv_mgr_append_slot": (ctypes.c_int, [vp, c_i64, vp, vp, vp]),
        "pkv_mgr_append_batch": (ctypes.c_int, [vp, vp, c_i32, vp, vp, vp, vp]),
        "pkv_mgr_extend": (ctypes.c_int, [vp, c_i64, c_i32, vp, vp, vp]),
        "pkv_mgr_free_seq": (ctypes.c_int, [vp, c_i64]),
        "pkv_mgr_block_table": (ctypes.c_int, [vp, c_i64, vp, c_i32, vp, vp]),
        "pkv_mgr_pack_tables": (ctypes.c_int, [vp, vp, c_i32, c_i32, vp, vp]),
        "pkv_mgr_stats": (ctypes.c_int, [vp, ctypes.POINTER(Stats)]),
        "pkv_mgr_refcount": (c_i32, [vp, c_i32]),
        "pkv_mgr_free_list": (c_i32, [vp, vp, c_i32]),
        "pkv_mgr_inject_alloc_failure": (ctypes.c_int, [vp, c_i32]),
        "pkv_mgr_save_bytes": (c_sz, [vp]),
        "pkv_mgr_save": (ctypes.c_int, [vp, vp, c_sz, ctypes.POINTER(c_sz)]),
        "pkv_mgr_load": (vp, [vp, c_sz]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_str(status: int) -> str:
    return lib().pkv_status_str(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != PKV_OK:
        raise PkvError(rc, what)


def make_desc(dtype: str, n_layers: int, num_blocks: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
              block_size: int = BLOCK) -> CacheDesc:
    return CacheDesc(DTYPE_CODES[dtype], n_layers, num_blocks, n_q_heads, n_kv_heads, head_dim, block_size)


# ---- torch marshalling --------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def torch_dtype(name: str):
    t = _torch()
    return {"f32": t.float32, "f16": t.float16, "bf16": t.bfloat16}[name]


def _stream_handle(stream):
    t = _torch()
    if stream is None:
        return ctypes.c_void_p(t.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _current_device() -> int:
    """Index of the current CUDA device, or -1 where CUDA cannot be initialised (every tensor check
    then fails on its own, with a ValueError, before any launch)."""
    try:
        return _torch().cuda.current_device()
    except (RuntimeError, AssertionError):
        return -1


def _on_current_device(x, name, cur=None):
    """The library runs on the current device: a tensor elsewhere is refused. `cur` (the current
    device's index) is read once per call by callers that check several tensors."""
    if cur is None:
        cur = _torch().cuda.current_device()
    if x.get_device() != cur:
        raise ValueError(f"{name} is on {x.device}; the calls run on the current device, cuda:{cur}")


def _dev(x, name, dtype=None, shape=None, cur=None):
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    _on_current_device(x, name, cur)
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(x.shape)}")
    return ctypes.c_void_p(x.data_ptr())


def pool_shape(desc: CacheDesc):
    return (desc.n_layers, desc.num_blocks, desc.n_kv_heads, desc.block_size, desc.head_dim)


def pkv_validate_desc(desc: CacheDesc) -> int:
    return int(lib().pkv_validate_desc(ctypes.byref(desc)))


def pkv_bytes_per_token(desc: CacheDesc) -> int:
    return int(lib().pkv_bytes_per_token(ctypes.byref(desc)))


def pkv_pool_bytes(desc: CacheDesc) -> int:
    return int(lib().pkv_pool_bytes(ctypes.byref(desc)))


def pkv_decode_workspace_bytes(desc: CacheDesc, n_seqs: int, max_blocks_per_seq: int) -> int:
    return int(lib().pkv_decode_workspace_bytes(ctypes.byref(desc), int(n_seqs), int(max_blocks_per_seq)))


def pkv_decode_split_geometry(desc: CacheDesc, n_seqs: int, max_blocks_per_seq: int, sm_count: int,
                              ctas_per_sm: int):
    """(blocks per partition, partitions, workspace bytes) of decode on a part with sm_count SMs that
    each hold ctas_per_sm decode CTAs."""
    bpp, nparts, nbytes = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_size_t(0)
    _check(lib().pkv_decode_split_geometry(ctypes.byref(desc), int(n_seqs), int(max_blocks_per_seq), int(sm_count),
                                           int(ctas_per_sm), ctypes.byref(bpp), ctypes.byref(nparts),
                                           ctypes.byref(nbytes)),
           "pkv_decode_split_geometry")
    return int(bpp.value), int(nparts.value), int(nbytes.value)


def pkv_prefill_wave_tokens(desc: CacheDesc) -> int:
    """Tokens of one sequence's chunk that fill one wave of the prefill grid on the current device."""
    t = ctypes.c_int32(0)
    _check(lib().pkv_prefill_wave_tokens(ctypes.byref(desc), ctypes.byref(t)), "pkv_prefill_wave_tokens")
    return int(t.value)


def wave_aligned_chunk(desc: CacheDesc, target: int) -> int:
    """The whole number of prefill waves (at least one) closest to `target` tokens per chunk."""
    w = pkv_prefill_wave_tokens(desc)
    return w * max(1, int(round(target / w)))


def pkv_decode_ctas_per_sm(desc: CacheDesc):
    """(decode CTAs per SM for this descriptor, SM count) on the current device."""
    per_sm, sms = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib().pkv_decode_ctas_per_sm(ctypes.byref(desc), ctypes.byref(per_sm), ctypes.byref(sms)),
           "pkv_decode_ctas_per_sm")
    return int(per_sm.value), int(sms.value)


def pkv_kv_append(desc: CacheDesc, layer: int, k, v, slot_mapping, k_pool, v_pool, stream=None) -> None:
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_tok = int(k.shape[0])
    row = (n_tok, desc.n_kv_heads, desc.head_dim)
    rc = lib().pkv_kv_append(
        ctypes.byref(desc), int(layer), _dev(k, "k", dt, row, cur=cur), _dev(v, "v", dt, row, cur=cur),
        _dev(slot_mapping, "slot_mapping", t.int64, (n_tok,), cur=cur), n_tok,
        _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur), _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _stream_handle(stream))
    _check(rc, "pkv_kv_append")


def pkv_paged_decode_attention(desc: CacheDesc, layer: int, q, k_pool, v_pool, block_tables, context_lens,
                               scale: float, out, workspace=None, stream=None) -> None:
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_seqs = int(q.shape[0])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    max_blocks = int(block_tables.shape[1])
    qshape = (n_seqs, desc.n_q_heads, desc.head_dim)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace", cur=cur)
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pkv_paged_decode_attention(
        ctypes.byref(desc), int(layer), _dev(q, "q", dt, qshape, cur=cur),
        _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur), _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _dev(block_tables, "block_tables", t.int32, (n_seqs, max_blocks), cur=cur), max_blocks,
        _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur), n_seqs, float(scale),
        _dev(out, "out", dt, qshape, cur=cur), ws_ptr, ws_bytes, _stream_handle(stream))
    _check(rc, "pkv_paged_decode_attention")


def dense_cache_shape(desc: CacheDesc, n_seqs: int, max_seq_len: int):
    """[n_layers, n_seqs, n_kv, max_seq_len, d]: the dense (batch, heads, length, head_dim) cache."""
    return (desc.n_layers, n_seqs, desc.n_kv_heads, max_seq_len, desc.head_dim)


def pkv_dense_decode_attention(desc: CacheDesc, layer: int, q, k_cache, v_cache, context_lens, scale: float, out,
                               workspace=None, stream=None, overlap_previous: bool = False) -> None:
    """Decode attention over a dense cache [L, n_seqs, n_kv, S, d] (identity walk, no block table)."""
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_seqs = int(q.shape[0])
    if k_cache.dim() != 5:
        raise ValueError("k_cache must be [n_layers, n_seqs, n_kv, max_seq_len, head_dim]")
    s_max = int(k_cache.shape[3])
    shape = dense_cache_shape(desc, n_seqs, s_max)
    qshape = (n_seqs, desc.n_q_heads, desc.head_dim)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace", cur=cur)
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pkv_dense_decode_attention(
        ctypes.byref(desc), int(layer), _dev(q, "q", dt, qshape, cur=cur), _dev(k_cache, "k_cache", dt, shape, cur=cur),
        _dev(v_cache, "v_cache", dt, shape, cur=cur), s_max, _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur), n_seqs,
        float(scale), _dev(out, "out", dt, qshape, cur=cur), ws_ptr, ws_bytes,
        PKV_DECODE_OVERLAP_PREVIOUS if overlap_previous else 0, _stream_handle(stream))
    _check(rc, "pkv_dense_decode_attention")


def pkv_paged_decode_append_attention(desc: CacheDesc, layer: int, q, k_new, v_new, k_pool, v_pool, block_tables,
                                      context_lens, scale: float, out, workspace=None, stream=None,
                                      overlap_previous: bool = False) -> None:
    """One decode step of one layer: append each sequence's new K/V row at position len-1, then attend.

    overlap_previous: launch with PKV_DECODE_OVERLAP_PREVIOUS (only when the previous kernel on the
    stream is this call for the previous layer of the same step).
    """
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_seqs = int(q.shape[0])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    max_blocks = int(block_tables.shape[1])
    qshape = (n_seqs, desc.n_q_heads, desc.head_dim)
    kvshape = (n_seqs, desc.n_kv_heads, desc.head_dim)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, "workspace", cur=cur)
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib().pkv_paged_decode_append_attention_ex(
        ctypes.byref(desc), int(layer), _dev(q, "q", dt, qshape, cur=cur), _dev(k_new, "k_new", dt, kvshape, cur=cur),
        _dev(v_new, "v_new", dt, kvshape, cur=cur), _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur),
        _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _dev(block_tables, "block_tables", t.int32, (n_seqs, max_blocks), cur=cur), max_blocks,
        _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur), n_seqs, float(scale),
        _dev(out, "out", dt, qshape, cur=cur), ws_ptr, ws_bytes,
        PKV_DECODE_OVERLAP_PREVIOUS if overlap_previous else 0, _stream_handle(stream))
    _check(rc, "pkv_paged_decode_append_attention")


def pkv_paged_decode_attention_static(desc: CacheDesc, layer: int, q, k_pool, v_pool, block_tables, context_lens,
                                      scale: float, out, stream=None) -> None:
    """pkv_paged_decode_attention with the library's fixed scratch instead of a workspace.

    For callers that cannot allocate device memory when attention runs; see include/pkv.h
    for the scratch limit and the rule that overlapping calls must be serialised.
    """
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_seqs = int(q.shape[0])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    max_blocks = int(block_tables.shape[1])
    qshape = (n_seqs, desc.n_q_heads, desc.head_dim)
    rc = lib().pkv_paged_decode_attention_static(
        ctypes.byref(desc), int(layer), _dev(q, "q", dt, qshape, cur=cur),
        _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur), _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _dev(block_tables, "block_tables", t.int32, (n_seqs, max_blocks), cur=cur), max_blocks,
        _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur), n_seqs, float(scale),
        _dev(out, "out", dt, qshape, cur=cur), _stream_handle(stream))
    _check(rc, "pkv_paged_decode_attention_static")


def pkv_paged_prefill_attention(desc: CacheDesc, layer: int, q, k_pool, v_pool, block_tables, context_lens,
                                query_start, max_query_len: int, scale: float, out, stream=None,
                                overlap_previous: bool = False) -> None:
    """Causal attention of each sequence's chunk of new tokens over its paged cache (one layer).

    q, out [n_tokens, n_q, d]; query_start int32 [n_seqs + 1] (device); max_query_len is the
    largest chunk, known to the caller from its own planning (no device read here).
    overlap_previous: launch with PKV_PREFILL_OVERLAP_PREVIOUS (only when the previous kernel on the
    stream is this call for the previous layer and every layer's rows were appended before).
    """
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_tokens = int(q.shape[0])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    n_seqs, max_blocks = int(block_tables.shape[0]), int(block_tables.shape[1])
    qshape = (n_tokens, desc.n_q_heads, desc.head_dim)
    rc = lib().pkv_paged_prefill_attention_ex(
        ctypes.byref(desc), int(layer), _dev(q, "q", dt, qshape, cur=cur),
        _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur), _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _dev(block_tables, "block_tables", t.int32, (n_seqs, max_blocks), cur=cur), max_blocks,
        _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur),
        _dev(query_start, "query_start", t.int32, (n_seqs + 1,), cur=cur), n_seqs, n_tokens, int(max_query_len),
        float(scale), _dev(out, "out", dt, qshape, cur=cur), PKV_PREFILL_OVERLAP_PREVIOUS if overlap_previous else 0,
        _stream_handle(stream))
    _check(rc, "pkv_paged_prefill_attention")


def pkv_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self-test (a wait nobody completes; it gives up and flags the status)."""
    _check(lib().pkv_selftest_wait_timeout(_stream_handle(stream)), "pkv_selftest_wait_timeout")


def pkv_copy_blocks(desc: CacheDesc, k_pool, v_pool, pairs, stream=None) -> None:
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    n_pairs = int(pairs.shape[0])
    rc = lib().pkv_copy_blocks(
        ctypes.byref(desc), _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur), _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur),
        _dev(pairs, "pairs", t.int32, (n_pairs, 2), cur=cur), n_pairs, _stream_handle(stream))
    _check(rc, "pkv_copy_blocks")


def pkv_upload_metadata(dst, src, stream=None) -> None:
    """dst (device) <- src (pinned host), same byte size, through a kernel rather than a copy engine."""
    if not dst.is_cuda or not dst.is_contiguous():
        raise ValueError("dst must be a contiguous CUDA tensor")
    if src.is_cuda or not src.is_contiguous() or not src.is_pinned():
        raise ValueError("src must be a contiguous pinned host tensor")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must have the same byte size")
    rc = lib().pkv_upload_metadata(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                   _stream_handle(stream))
    _check(rc, "pkv_upload_metadata")


def upload_metadata_ptr(dst_ptr: int, src_ptr: int, nbytes: int, stream_handle: int) -> None:
    """pkv_upload_metadata on raw pointers (the engine keeps its pinned and device images' addresses)."""
    _check(lib().pkv_upload_metadata(dst_ptr, src_ptr, nbytes, stream_handle), "pkv_upload_metadata")


# ---- per-step launchers: a step's tensors validated once, one C call per layer ---------------------
#
# A step launches the same call for every layer with the same [L, ...] tensors. The launchers below
# check them once (device, dtype, shape, each layer's slice contiguous -- views of larger buffers are
# fine) and keep raw addresses, so a layer's launch is a single call into the C ABI with the same
# arguments the per-call bindings above would pass.

def _layered(x, name, dtype, n_layers: int, row_shape, cur=None):
    """(address of layer 0, bytes between layers) of a [n_layers, *row_shape] tensor."""
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    _on_current_device(x, name, cur)
    if x.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {x.dtype}")
    if tuple(x.shape) != (n_layers, *row_shape):
        raise ValueError(f"{name} must have shape {(n_layers, *row_shape)}, got {tuple(x.shape)}")
    if not x[0].is_contiguous():
        raise ValueError(f"{name}: each layer's slice must be contiguous")
    return x.data_ptr(), x.stride(0) * x.element_size()


def _raw_stream(stream) -> int:
    return _stream_handle(stream).value or 0


def decode_append_launcher(desc: CacheDesc, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens,
                           scale: float, out, workspace=None, stream=None):
    """launch(layer, overlap_previous=False): pkv_paged_decode_append_attention_ex of one layer, with
    q/out [L, n, n_q, d] and k_new/v_new [L, n, n_kv, d] validated here once."""
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    L, n = desc.n_layers, int(q.shape[1])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    mb = int(block_tables.shape[1])
    q0, qs = _layered(q, "q", dt, L, (n, desc.n_q_heads, desc.head_dim), cur=cur)
    o0, os_ = _layered(out, "out", dt, L, (n, desc.n_q_heads, desc.head_dim), cur=cur)
    k0, ks = _layered(k_new, "k_new", dt, L, (n, desc.n_kv_heads, desc.head_dim), cur=cur)
    v0, vs = _layered(v_new, "v_new", dt, L, (n, desc.n_kv_heads, desc.head_dim), cur=cur)
    kp = _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur).value
    vp = _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur).value
    tb = _dev(block_tables, "block_tables", t.int32, (n, mb), cur=cur).value
    ln = _dev(context_lens, "context_lens", t.int32, (n,), cur=cur).value
    wsp, wsb = (None, 0) if workspace is None else (_dev(workspace, "workspace", cur=cur).value,
                                                    workspace.numel() * workspace.element_size())
    fn, dref, sc, sh = lib().pkv_paged_decode_append_attention_ex, ctypes.byref(desc), float(scale), _raw_stream(stream)

    def launch(layer: int, overlap_previous: bool = False) -> None:
        rc = fn(dref, layer, q0 + layer * qs, k0 + layer * ks, v0 + layer * vs, kp, vp, tb, mb, ln, n, sc,
                o0 + layer * os_, wsp, wsb, PKV_DECODE_OVERLAP_PREVIOUS if overlap_previous else 0, sh)
        if rc:
            raise PkvError(rc, "pkv_paged_decode_append_attention")
    return launch


def prefill_launcher(desc: CacheDesc, q, k_pool, v_pool, block_tables, context_lens, query_start,
                     max_query_len: int, scale: float, out, stream=None):
    """launch(layer, overlap_previous=False): pkv_paged_prefill_attention_ex of one layer, with
    q/out [L, n_tokens, n_q, d] validated here once."""
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    L, n_tok = desc.n_layers, int(q.shape[1])
    if block_tables.dim() != 2:
        raise ValueError("block_tables must be [n_seqs, max_blocks]")
    n_seqs, mb = int(block_tables.shape[0]), int(block_tables.shape[1])
    q0, qs = _layered(q, "q", dt, L, (n_tok, desc.n_q_heads, desc.head_dim), cur=cur)
    o0, os_ = _layered(out, "out", dt, L, (n_tok, desc.n_q_heads, desc.head_dim), cur=cur)
    kp = _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur).value
    vp = _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur).value
    tb = _dev(block_tables, "block_tables", t.int32, (n_seqs, mb), cur=cur).value
    ln = _dev(context_lens, "context_lens", t.int32, (n_seqs,), cur=cur).value
    qsd = _dev(query_start, "query_start", t.int32, (n_seqs + 1,), cur=cur).value
    fn, dref, sc, sh = lib().pkv_paged_prefill_attention_ex, ctypes.byref(desc), float(scale), _raw_stream(stream)
    mq = int(max_query_len)

    def launch(layer: int, overlap_previous: bool = False) -> None:
        rc = fn(dref, layer, q0 + layer * qs, kp, vp, tb, mb, ln, qsd, n_seqs, n_tok, mq, sc, o0 + layer * os_,
                PKV_PREFILL_OVERLAP_PREVIOUS if overlap_previous else 0, sh)
        if rc:
            raise PkvError(rc, "pkv_paged_prefill_attention")
    return launch


def append_launcher(desc: CacheDesc, k, v, slot_mapping, k_pool, v_pool, stream=None):
    """launch(layer): pkv_kv_append of one layer, with k/v [L, n_tokens, n_kv, d] validated here once."""
    t = _torch()
    dt = torch_dtype(desc.dtype_name)
    cur = _current_device()
    L, n_tok = desc.n_layers, int(k.shape[1])
    k0, ks = _layered(k, "k", dt, L, (n_tok, desc.n_kv_heads, desc.head_dim), cur=cur)
    v0, vs = _layered(v, "v", dt, L, (n_tok, desc.n_kv_heads, desc.head_dim), cur=cur)
    sl = _dev(slot_mapping, "slot_mapping", t.int64, (n_tok,), cur=cur).value
    kp = _dev(k_pool, "k_pool", dt, pool_shape(desc), cur=cur).value
    vp = _dev(v_pool, "v_pool", dt, pool_shape(desc), cur=cur).value
    fn, dref, sh = lib().pkv_kv_append, ctypes.byref(desc), _raw_stream(stream)

    def launch(layer: int) -> None:
        rc = fn(dref, layer, k0 + layer * ks, v0 + layer * vs, sl, n_tok, kp, vp, sh)
        if rc:
            raise PkvError(rc, "pkv_kv_append")
    return launch


def pkv_get_device_status(stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib().pkv_get_device_status(_stream_handle(stream), ctypes.byref(flags)), "pkv_get_device_status")
    return int(flags.value)


def pkv_hbm_read_probe(buf, fold, stream=None) -> None:
    """Stream every byte of the device tensor buf once; XOR-fold its 32-bit words into fold (a
    device int32 tensor of one element)."""
    if not buf.is_contiguous():
        raise ValueError("buf must be contiguous")
    _on_current_device(buf, "buf")
    _check(lib().pkv_hbm_read_probe(ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(),
                                    _dev(fold, "fold", _torch().int32, (1,)), _stream_handle(stream)),
           "pkv_hbm_read_probe")


def pkv_launch_count() -> int:
    return int(lib().pkv_launch_count())


def alloc_workspace(desc: CacheDesc, n_seqs: int, max_blocks_per_seq: int, device="cuda"):
    """A device buffer of pkv_decode_workspace_bytes (allocated by torch; None when 0)."""
    t = _torch()
    n = pkv_decode_workspace_bytes(desc, n_seqs, max_blocks_per_seq)
    return t.zeros(max(n, 16) // 4 + 4, dtype=t.float32, device=device) if n else None


# ---- host block manager -------------------------------------------------------------------------

# The manager's array arguments are declared void* and take the array's address: building a
# typed ctypes pointer per argument cost more than the manager call itself. The arrays are
# contiguous int64 / int32 numpy arrays that the caller keeps alive through the call.
def _i64p(a):
    return a.ctypes.data


def _i32p(a):
    return a.ctypes.data


class BlockManager:
    """Owner of one pkv_mgr handle; methods return the C status code (and outputs)."""

    def __init__(self, num_blocks: int, block_size: int = BLOCK, free_order=None, _handle=None):
        L = lib()
        if _handle is not None:
            self._h = _handle
        else:
            order = None
            if free_order is not None:
                order = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
                if order.shape != (num_blocks,):
                    raise ValueError("free_order must list every block once")
            self._h = L.pkv_mgr_create(int(num_blocks), int(block_size), _i32p(order) if order is not None else None)
        if not self._h:
            raise PkvError(PKV_ERR_INVALID_ARG, "pkv_mgr_create")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.pkv_mgr_destroy(h)
            self._h = None

    def clone(self) -> "BlockManager":
        h = lib().pkv_mgr_clone(self._h)
        if not h:
            raise PkvError(PKV_ERR_BAD_STATE, "pkv_mgr_clone")
        return BlockManager(self.num_blocks, self.block_size, _handle=h)

    def save(self) -> bytes:
        """The manager's state as a pkv_mgr_save image (checkpoint)."""
        L = lib()
        n = int(L.pkv_mgr_save_bytes(self._h))
        buf = ctypes.create_string_buffer(n)
        written = ctypes.c_size_t(0)
        _check(L.pkv_mgr_save(self._h, buf, n, ctypes.byref(written)), "pkv_mgr_save")
        return buf.raw[: written.value]

    @classmethod
    def load(cls, image: bytes) -> "BlockManager":
        """A manager resumed from a save() image; raises PkvError if the image is malformed."""
        data = bytes(image)
        h = lib().pkv_mgr_load(data, len(data))
        if not h:
            raise PkvError(PKV_ERR_INVALID_ARG, "pkv_mgr_load (malformed image)")
        num_blocks = int.from_bytes(data[8:12], "little")
        block_size = int.from_bytes(data[12:16], "little")
        return cls(num_blocks, block_size, _handle=h)

    def add_seq(self, seq_id: int, n_prompt: int, reserve_tokens: int = 0):
        slots = np.zeros(max(int(n_prompt), 1), dtype=np.int64)
        rc = lib().pkv_mgr_add_seq(self._h, int(seq_id), int(n_prompt), int(reserve_tokens), _i64p(slots))
        return rc, (slots[:n_prompt] if rc == PKV_OK else slots[:0])

    def fork(self, parent: int, child: int) -> int:
        return lib().pkv_mgr_fork(self._h, int(parent), int(child))

    def extend(self, seq_id: int, n_tokens: int, slots_out=None):
        """Slots of n_tokens new positions at once (all or nothing); returns (rc, slots, src, dst)."""
        n = int(n_tokens)
        slots = slots_out if slots_out is not None else np.zeros(max(n, 1), dtype=np.int64)
        src, dst = ctypes.c_int32(-1), ctypes.c_int32(-1)
        rc = lib().pkv_mgr_extend(self._h, int(seq_id), n, _i64p(slots), ctypes.byref(src), ctypes.byref(dst))
        return rc, (slots[:n] if rc == PKV_OK else slots[:0]), int(src.value), int(dst.value)

    def append_slot(self, seq_id: int):
        slot, src, dst = ctypes.c_int64(-1), ctypes.c_int32(-1), ctypes.c_int32(-1)
        rc = lib().pkv_mgr_append_slot(self._h, int(seq_id), ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst))
        return rc, int(slot.value), int(src.value), int(dst.value)

    def append_batch(self, seq_ids):
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = len(ids)
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros(max(2 * n, 2), dtype=np.int32)
        n_cow, n_done = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = lib().pkv_mgr_append_batch(self._h, _i64p(ids), n, _i64p(slots), _i32p(pairs),
                                        ctypes.byref(n_cow), ctypes.byref(n_done))
        return rc, slots[:n_done.value], pairs[:2 * n_cow.value].reshape(-1, 2), int(n_done.value)

    def free_seq(self, seq_id: int) -> int:
        return lib().pkv_mgr_free_seq(self._h, int(seq_id))

    def block_table(self, seq_id: int):
        nb, ctx = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = lib().pkv_mgr_block_table(self._h, int(seq_id), None, 0, ctypes.byref(nb), ctypes.byref(ctx))
        if rc != PKV_OK and nb.value == 0 and ctx.value == 0:
            return rc, [], 0
        buf = np.zeros(max(nb.value, 1), dtype=np.int32)
        rc = lib().pkv_mgr_block_table(self._h, int(seq_id), _i32p(buf), nb.value, ctypes.byref(nb), ctypes.byref(ctx))
        return rc, buf[:nb.value].tolist(), int(ctx.value)

    def pack_tables(self, seq_ids, max_blocks: int, tables_out=None, lens_out=None):
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        n = len(ids)
        tables = tables_out if tables_out is not None else np.empty((n, max_blocks), dtype=np.int32)
        lens = lens_out if lens_out is not None else np.empty(n, dtype=np.int32)
        rc = lib().pkv_mgr_pack_tables(self._h, _i64p(ids), n, int(max_blocks), _i32p(tables), _i32p(lens))
        return rc, tables, lens

    def stats(self) -> dict:
        st = Stats()
        _check(lib().pkv_mgr_stats(self._h, ctypes.byref(st)), "pkv_mgr_stats")
        return st.as_dict()

    def refcount(self, block: int) -> int:
        return int(lib().pkv_mgr_refcount(self._h, int(block)))

    def refcounts(self):
        return [self.refcount(b) for b in range(self.num_blocks)]

    def free_list(self):
        buf = np.zeros(max(self.num_blocks, 1), dtype=np.int32)
        n = lib().pkv_mgr_free_list(self._h, _i32p(buf), self.num_blocks)
        return buf[:n].tolist()

    def inject_alloc_failure(self, after_n_allocs: int) -> int:
        return lib().pkv_mgr_inject_alloc_failure(self._h, int(after_n_allocs))
