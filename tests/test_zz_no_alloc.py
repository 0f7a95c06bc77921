"""The allocation-free decode entry point against the ordinary one (GPU, through the C ABI).

pkv_paged_decode_attention_static serves callers that cannot allocate device memory when they
run attention (inside a stream capture, in a loop that forbids allocation, under a fixed
memory budget): its split-K scratch is an array compiled into the library instead of a
caller-provided workspace. Two calls in a row, on different inputs, must each match what
pkv_paged_decode_attention (with a torch-allocated workspace) returns for the same inputs, bit for
bit, so the shared scratch's leftover contents from the first call cannot leak into the second.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL, as_f64, paged_case, to_torch
from paged_kv_cache_258_gb300 import pkv

pytestmark = pytest.mark.gpu


def _inputs(dtype, lens, n_q, n_kv, d, seed):
    q, kp, vp, tables, lens, nb = paged_case(dtype, lens, n_q, n_kv, d, seed)
    desc = pkv.make_desc(dtype, 1, nb, n_q, n_kv, d)
    return (desc, to_torch(q, dtype), to_torch(kp, dtype), to_torch(vp, dtype),
            torch.from_numpy(np.ascontiguousarray(tables)).cuda(), torch.from_numpy(lens).cuda())


@pytest.mark.parametrize("dtype,n_q,n_kv,n_kv2,d", [("f16", 8, 2, 4, 128), ("bf16", 16, 4, 2, 256),
                                                    ("f32", 2, 1, 2, 64)])
def test_static_scratch_matches_workspace_version_twice(dtype, n_q, n_kv, n_kv2, d):
    # The second call has another geometry (sequences, table width, KV heads) and needs less than
    # half the scratch of the first, so its arrival counters sit where the first call left float
    # partials: leftovers of an earlier call must read as zero arrivals, whatever they hold.
    cases = [_inputs(dtype, [1, 17, 600, 1500, 2100, 3000, 777], n_q, n_kv, d, seed=31),
             _inputs(dtype, [900, 5, 333], n_q, n_kv2, d, seed=32)]
    need = [pkv.pkv_decode_workspace_bytes(c[0], c[1].shape[0], c[4].shape[1]) for c in cases]
    assert need[0] > 0 and need[1] > 0                      # split-K is in use in both calls
    assert 2 * need[1] <= need[0]
    for desc, q, kp, vp, tables, lens in cases:
        max_blocks = tables.shape[1]
        ref = torch.full_like(q, float("nan"))
        ws = pkv.alloc_workspace(desc, q.shape[0], max_blocks)
        pkv.pkv_paged_decode_attention(desc, 0, q, kp, vp, tables, lens, 0.1, ref, ws)
        got = torch.full_like(q, float("nan"))
        pkv.pkv_paged_decode_attention_static(desc, 0, q, kp, vp, tables, lens, 0.1, got)
        assert pkv.pkv_get_device_status() == 0
        a, b = as_f64(got), as_f64(ref)
        assert np.all(np.isfinite(a))
        assert np.max(np.abs(a - b)) <= TOL[dtype]
        # same kernels, same partitions, same merge order: the results agree bit for bit
        assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))


def test_static_scratch_rejects_oversized_calls_before_launching():
    desc, q, kp, vp, tables, lens = _inputs("f16", [40, 70], 4, 4, 64, seed=33)
    # 4,096 sequences (more (sequence, KV head) pairs than any GPU holds CTAs) with tables 2^20 blocks
    # wide would need far more than 16 MiB of partials; the call is refused before anything is read
    n_seqs, big = 4096, 1 << 20
    need = pkv.pkv_decode_workspace_bytes(desc, n_seqs, big)
    assert need > 16 << 20
    before = pkv.pkv_launch_count()
    L = pkv.lib()
    rc = L.pkv_paged_decode_attention_static(
        ctypes.byref(desc), 0, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), ctypes.c_void_p(tables.data_ptr()), big, ctypes.c_void_p(lens.data_ptr()),
        n_seqs, ctypes.c_float(0.1), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(0))
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    assert pkv.pkv_launch_count() == before
