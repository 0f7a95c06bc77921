"""The C ABI library loads and exports every symbol include/pkv.h declares; host-only calls.

No compute call here: device entry points are only checked for their host-side argument
validation paths that return before any CUDA call.
"""
import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_cache_258_gb300 import pkv

HEADERS = sorted((Path(__file__).resolve().parent.parent / "include").glob("*.h"))


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    L = pkv.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # the binding declares a signature for exactly the functions the header declares
    import inspect
    src = inspect.getsource(pkv.lib)
    bound = set(re.findall(r'"(pkv_\w+)":', src))
    assert bound == set(names)


def test_bytes_per_token_matches_pages(golden):
    g = golden["kv_bytes_per_token_gpt"]
    d = pkv.make_desc("f16", g["n_layers"], 100, 32, g["n_kv_heads"], g["head_dim"])
    assert pkv.pkv_bytes_per_token(d) == g["value"]
    d = pkv.make_desc("bf16", 16, 100, 16, 4, 256)
    assert pkv.pkv_bytes_per_token(d) * 16 == golden["longdoc_block_bytes"]["value"]
    assert pkv.pkv_pool_bytes(d) == 16 * 100 * 4 * 16 * 256 * 2


@pytest.mark.parametrize("kw,want", [
    (dict(dtype="f16", n_layers=1, num_blocks=8, n_q_heads=8, n_kv_heads=2, head_dim=128), pkv.PKV_OK),
    (dict(dtype="f32", n_layers=1, num_blocks=8, n_q_heads=16, n_kv_heads=2, head_dim=64), pkv.PKV_OK),
    (dict(dtype="bf16", n_layers=1, num_blocks=8, n_q_heads=6, n_kv_heads=2, head_dim=128), pkv.PKV_ERR_UNSUPPORTED),
    (dict(dtype="f16", n_layers=1, num_blocks=8, n_q_heads=32, n_kv_heads=2, head_dim=128), pkv.PKV_ERR_UNSUPPORTED),
    (dict(dtype="f16", n_layers=1, num_blocks=8, n_q_heads=2, n_kv_heads=2, head_dim=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(dtype="f16", n_layers=0, num_blocks=8, n_q_heads=2, n_kv_heads=2, head_dim=64), pkv.PKV_ERR_INVALID_ARG),
    (dict(dtype="f16", n_layers=1, num_blocks=8, n_q_heads=2, n_kv_heads=2, head_dim=64, block_size=32),
     pkv.PKV_ERR_UNSUPPORTED),
])
def test_validate_desc(kw, want):
    assert pkv.pkv_validate_desc(pkv.make_desc(**kw)) == want


def _ws(desc, n_seqs, max_blocks, sms=152, per_sm=3):
    return pkv.pkv_decode_split_geometry(desc, n_seqs, max_blocks, sms, per_sm)[2]


def test_workspace_only_when_split():
    d = pkv.make_desc("f16", 1, 4096, 32, 32, 128)
    assert _ws(d, 64, 64) == 0                                      # one partition per sequence
    n = _ws(d, 64, 129)
    assert n == 64 * 32 * 3 * (128 + 2) * 4 + 64 * 32 * 8          # 129 blocks -> 3 partitions of 64
    d4 = pkv.make_desc("bf16", 16, 30000, 16, 4, 256)
    # 40 (sequence, KV head) pairs over 456 slots: one wave of 11 partitions of 187 blocks each
    assert _ws(d4, 10, 2048) == 10 * 16 * 11 * (256 + 2) * 4 + 10 * 4 * 8
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_split_geometry(d, 0, 10, 152, 3)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_split_geometry(d, 4, 10, 0, 3)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_decode_split_geometry(d, 4, 10, 152, 0)
    assert pkv.pkv_decode_workspace_bytes(d, 0, 10) == 0


@pytest.mark.parametrize("sms,per_sm,bpp,n_parts", [
    (152, 3, 187, 11),     # 440 of 456 slots: one wave of equal CTAs
    (76, 3, 410, 5),       # 200 of 228
    (152, 2, 293, 7),      # 280 of 304
    (20, 1, 64, 32),       # more pairs than slots: several waves of 64-block partitions
    (1000, 3, 16, 128),    # the one-wave partitions would be short (28 blocks): ~4 CTAs per SM instead
])
def test_split_geometry_follows_the_device(sms, per_sm, bpp, n_parts):
    """10 sequences x 4 KV heads x 2,048 blocks (the long-document shape) on parts of other sizes."""
    d4 = pkv.make_desc("bf16", 16, 30000, 16, 4, 256)
    got_bpp, got_parts, nbytes = pkv.pkv_decode_split_geometry(d4, 10, 2048, sms, per_sm)
    assert (got_bpp, got_parts) == (bpp, n_parts)
    assert got_parts == -(-2048 // got_bpp)
    assert nbytes == 10 * 16 * n_parts * (256 + 2) * 4 + 10 * 4 * 8


def test_split_geometry_rules():
    # fp32 pools run the CUDA-core kernel, whose partitions stop at 64 entries: no one-wave split
    d32 = pkv.make_desc("f32", 16, 30000, 16, 4, 256)
    assert pkv.pkv_decode_split_geometry(d32, 10, 2048, 152, 3)[:2] == (64, 32)
    # as many pairs as slots or more: 64-entry partitions (the GPT-style batch: 64 x 32 pairs)
    d = pkv.make_desc("f16", 1, 4096, 32, 32, 128)
    assert pkv.pkv_decode_split_geometry(d, 64, 129, 152, 3)[:2] == (64, 3)
    # one wave would leave over a quarter of the slots empty (256 pairs, 1 CTA each): 64 entries
    d_gqa = pkv.make_desc("f16", 1, 4096, 32, 4, 128)
    assert pkv.pkv_decode_split_geometry(d_gqa, 64, 140, 152, 3)[:2] == (64, 3)
    # a single sequence and head is spread as far as 4-block partitions allow
    one = pkv.make_desc("f16", 1, 4096, 1, 1, 128)
    assert pkv.pkv_decode_split_geometry(one, 1, 128, 8, 3)[:2] == (4, 32)
    # a growing slot count never shrinks a one-wave partition below 64 entries
    for sms in range(100, 400, 7):
        b, n, _ = pkv.pkv_decode_split_geometry(pkv.make_desc("bf16", 1, 30000, 16, 4, 256), 10, 2048, sms, 3)
        assert b >= 4 and n == -(-2048 // b) and (b >= 64 or 40 * n >= 4 * sms)


def test_device_calls_reject_bad_arguments_before_launch():
    L = pkv.lib()
    d = pkv.make_desc("f16", 2, 16, 4, 4, 64)
    bad = pkv.make_desc("f16", 2, 16, 4, 3, 64)
    null = ctypes.c_void_p(0)
    assert L.pkv_kv_append(ctypes.byref(bad), 0, null, null, null, 1, null, null, null) == pkv.PKV_ERR_UNSUPPORTED
    assert L.pkv_kv_append(ctypes.byref(d), 2, null, null, null, 1, null, null, null) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_kv_append(ctypes.byref(d), 0, null, null, null, 0, null, null, null) == pkv.PKV_OK
    assert L.pkv_kv_append(ctypes.byref(d), 0, null, null, null, 3, null, null, null) == pkv.PKV_ERR_INVALID_ARG
    mis = ctypes.c_void_p(0x1008)
    assert L.pkv_kv_append(ctypes.byref(d), 0, mis, mis, mis, 3, mis, mis, null) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_paged_decode_attention(ctypes.byref(d), 0, null, null, null, null, 4, null, 0, 1.0, null, null, 0,
                                        null) == pkv.PKV_OK
    assert L.pkv_paged_decode_attention(ctypes.byref(d), 0, null, null, null, null, 4, null, 3, 1.0, null, null, 0,
                                        null) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_copy_blocks(ctypes.byref(d), null, null, null, 0, null) == pkv.PKV_OK
    assert L.pkv_copy_blocks(ctypes.byref(d), null, null, null, -1, null) == pkv.PKV_ERR_INVALID_ARG
    assert pkv.status_str(pkv.PKV_ERR_NO_BLOCKS).startswith("PKV_ERR_NO_BLOCKS")


def test_manager_create_rejects_non_permutation():
    L = pkv.lib()
    import numpy as np
    bad = np.array([0, 1, 1], dtype=np.int32)
    assert not L.pkv_mgr_create(3, 16, bad.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    assert not L.pkv_mgr_create(0, 16, None)


def test_overlap_flags_are_validated_before_anything_runs():
    """The *_ex calls refuse unknown launch-flag bits before looking at anything else, and accept
    PKV_*_OVERLAP_PREVIOUS (an empty call launches nothing). No GPU is needed."""
    import ctypes
    desc = pkv.make_desc("f16", 1, 4, 2, 2, 64)
    L = pkv.lib()
    for flags, want in ((2, pkv.PKV_ERR_INVALID_ARG), (pkv.PKV_DECODE_OVERLAP_PREVIOUS, pkv.PKV_OK)):
        rc = L.pkv_paged_decode_append_attention_ex(ctypes.byref(desc), 0, None, None, None, None, None, None, 4,
                                                    None, 0, 1.0, None, None, 0, flags, None)
        assert rc == want
    for flags, want in ((6, pkv.PKV_ERR_INVALID_ARG), (pkv.PKV_PREFILL_OVERLAP_PREVIOUS, pkv.PKV_OK)):
        rc = L.pkv_paged_prefill_attention_ex(ctypes.byref(desc), 0, None, None, None, None, 4, None, None, 0, 0,
                                              0, 1.0, None, flags, None)
        assert rc == want


def test_upload_metadata_rejects_bad_arguments_before_any_cuda_call():
    """Sizes and alignment are checked on the host first; an empty upload is a no-op. No GPU."""
    L = pkv.lib()
    null, a, mis = ctypes.c_void_p(0), ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10004)
    assert L.pkv_upload_metadata(null, null, 0, null) == pkv.PKV_OK
    assert L.pkv_upload_metadata(null, a, 16, null) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_upload_metadata(a, null, 16, null) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_upload_metadata(a, a, 6, null) == pkv.PKV_ERR_INVALID_ARG      # not whole words
    assert L.pkv_upload_metadata(mis, a, 16, null) == pkv.PKV_ERR_INVALID_ARG    # dst not 16-byte aligned
    assert L.pkv_upload_metadata(a, mis, 16, null) == pkv.PKV_ERR_INVALID_ARG    # src not 16-byte aligned
    assert L.pkv_upload_metadata(a, a, (1 << 30) + 4, null) == pkv.PKV_ERR_INVALID_ARG


def test_launchers_refuse_host_tensors_before_any_cuda_call():
    """The per-step launchers check their tensors on the host first: CPU tensors are refused
    with ValueError before the library is asked to launch anything. No GPU is needed."""
    import torch
    desc = pkv.make_desc("f16", 2, 8, 4, 2, 64)
    q = torch.zeros((2, 3, 4, 64), dtype=torch.float16)
    k = torch.zeros((2, 3, 2, 64), dtype=torch.float16)
    pool = torch.zeros(pkv.pool_shape(desc), dtype=torch.float16)
    tables = torch.zeros((3, 4), dtype=torch.int32)
    lens = torch.ones(3, dtype=torch.int32)
    with pytest.raises(ValueError):
        pkv.decode_append_launcher(desc, q, k, k, pool, pool, tables, lens, 0.1, q)
    with pytest.raises(ValueError):
        pkv.prefill_launcher(desc, q, pool, pool, tables, lens, torch.zeros(4, dtype=torch.int32), 1, 0.1, q)
    with pytest.raises(ValueError):
        pkv.append_launcher(desc, k, k, torch.zeros(3, dtype=torch.int64), pool, pool)


def test_wave_aligned_chunk_rounds_to_whole_waves(monkeypatch):
    """The chunk helper keeps a whole number (at least one) of prefill waves, the one closest to the
    target: 2,048 tokens over waves of 1,216 -> 2,432; over waves of 3,000 -> one wave."""
    d = pkv.make_desc("bf16", 1, 64, 16, 4, 256)
    for wave, target, want in [(1216, 2048, 2432), (1216, 1000, 1216), (3000, 2048, 3000), (512, 2048, 2048),
                               (600, 2048, 1800)]:
        monkeypatch.setattr(pkv, "pkv_prefill_wave_tokens", lambda desc, w=wave: w)
        assert pkv.wave_aligned_chunk(d, target) == want, (wave, target)
