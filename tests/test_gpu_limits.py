"""The boundary's size limits on the GPU: the largest batch a launch takes (65,535 sequences, the
grid's z extent) runs and matches the fp64 oracle, and one sequence more, or a table row longer
than 2^24 entries, is refused with a status code before anything is launched.

Unused pool rows are NaN-poisoned (vectorised here: the batches are too large for per-token loops).
"""
import ctypes

import numpy as np
import pytest

import oracle
from helpers import TOL, as_f64, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu
MAX_SEQS = 65535


def big_case(dtype, lens, n_q, n_kv, d, seed):
    """Pools [1, num_blocks, n_kv, 16, d] with shuffled tables; every row that is not a valid row of
    some sequence is NaN."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nb = -(-lens.astype(np.int64) // W.BLOCK)
    num_blocks = int(nb.sum()) + 3
    tables = W.shuffled_tables(lens, num_blocks, seed)
    kp = W.normal_values(rng, (1, num_blocks, n_kv, W.BLOCK, d), dtype)
    vp = W.normal_values(rng, (1, num_blocks, n_kv, W.BLOCK, d), dtype)
    # valid (block, offset) pairs: token j of sequence s is row j % 16 of block tables[s, j // 16]
    seq = np.repeat(np.arange(len(lens)), lens)
    j = np.arange(int(lens.sum())) - np.repeat(np.cumsum(lens) - lens, lens)
    valid = np.zeros((num_blocks, W.BLOCK), dtype=bool)
    valid[tables[seq, j // W.BLOCK], j % W.BLOCK] = True
    nanv = W.nan_value(dtype)
    for pool in (kp, vp):
        pool[0].transpose(0, 2, 1, 3)[~valid] = nanv
    return kp, vp, tables, lens, num_blocks


def test_decode_largest_batch_matches_oracle():
    import torch
    dtype, n_q, n_kv, d = "f16", 2, 1, 64
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 40, size=MAX_SEQS)
    kp, vp, tables, lens, num_blocks = big_case(dtype, lens, n_q, n_kv, d, seed=11)
    q = W.normal_values(rng, (MAX_SEQS, n_q, d), dtype)
    scale = 1.0 / np.sqrt(d)
    desc = pkv.make_desc(dtype, 1, num_blocks, n_q, n_kv, d)
    q_t = to_torch(q, dtype)
    out = torch.full_like(q_t, float("nan"))
    t_t = torch.from_numpy(np.ascontiguousarray(tables)).cuda()
    l_t = torch.from_numpy(lens).cuda()
    ws = pkv.alloc_workspace(desc, MAX_SEQS, tables.shape[1])
    pkv.pkv_paged_decode_attention(desc, 0, q_t, to_torch(kp, dtype), to_torch(vp, dtype), t_t, l_t, scale, out, ws)
    assert pkv.pkv_get_device_status() == 0
    got = as_f64(out)
    want = oracle.paged_decode(dtype, q, kp[0], vp[0], tables, lens, scale)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) <= TOL[dtype]


def test_prefill_largest_batch_matches_oracle():
    import torch
    dtype, n_q, n_kv, d = "f16", 4, 2, 64
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 40, size=MAX_SEQS)
    n_new = np.minimum(lens, rng.integers(1, 6, size=MAX_SEQS)).astype(np.int32)
    kp, vp, tables, lens, num_blocks = big_case(dtype, lens, n_q, n_kv, d, seed=12)
    qs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    q = W.normal_values(rng, (int(qs[-1]), n_q, d), dtype)
    scale = 1.0 / np.sqrt(d)
    desc = pkv.make_desc(dtype, 1, num_blocks, n_q, n_kv, d)
    q_t = to_torch(q, dtype)
    out = torch.full_like(q_t, float("nan"))
    pkv.pkv_paged_prefill_attention(
        desc, 0, q_t, to_torch(kp, dtype), to_torch(vp, dtype), torch.from_numpy(np.ascontiguousarray(tables)).cuda(),
        torch.from_numpy(lens).cuda(), torch.from_numpy(qs).cuda(), int(n_new.max()), scale, out)
    assert pkv.pkv_get_device_status() == 0
    got = as_f64(out)
    want = oracle.paged_prefill(dtype, q, kp[0], vp[0], tables, lens, qs, scale)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) <= TOL[dtype]


def test_one_sequence_past_the_limit_is_refused():
    """65,536 sequences: PKV_ERR_UNSUPPORTED from decode and prefill, nothing launched. (A launch
    would need a grid z extent of 65,536, which CUDA rejects; its reads would stay in block 0: every
    table entry is 0, decode lengths 0, prefill one token at position 0.)"""
    import torch
    n = MAX_SEQS + 1
    desc = pkv.make_desc("f16", 1, 4, 2, 1, 64)
    pool = torch.zeros(pkv.pool_shape(desc), dtype=torch.float16, device="cuda")
    q = torch.zeros((n, 2, 64), dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    tables = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    lens = torch.zeros((n,), dtype=torch.int32, device="cuda")
    ws = torch.zeros((1 << 20,), dtype=torch.uint8, device="cuda")
    before = pkv.pkv_launch_count()
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_decode_attention(desc, 0, q, pool, pool, tables, lens, 0.125, out, ws)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    qs = torch.arange(n + 1, dtype=torch.int32, device="cuda").clamp_(max=n)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_paged_prefill_attention(desc, 0, q, pool, pool, tables, torch.ones_like(lens), qs, 1, 0.125, out)
    assert e.value.status == pkv.PKV_ERR_UNSUPPORTED
    assert pkv.pkv_launch_count() == before
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0


def test_table_rows_past_2_24_entries_are_refused():
    """max_blocks_per_seq above 2^24: PKV_ERR_INVALID_ARG from decode and prefill before any read of
    the tables (the row claimed here is longer than the buffer behind it; the one sequence has
    length 1, so a launch would read entry 0 only)."""
    import torch
    desc = pkv.make_desc("bf16", 1, 4, 2, 2, 64)
    pool = torch.zeros(pkv.pool_shape(desc), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((1, 2, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    tables = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    lens = torch.ones((1,), dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ws = torch.zeros((1 << 20,), dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    L = pkv.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    too_long = (1 << 24) + 1
    before = pkv.pkv_launch_count()
    rc = L.pkv_paged_decode_attention(ctypes.byref(desc), 0, p(q), p(pool), p(pool), p(tables), too_long, p(lens), 1,
                                      ctypes.c_float(0.125), p(out), p(ws), ctypes.c_size_t(ws.numel()), stream)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    rc = L.pkv_paged_prefill_attention(ctypes.byref(desc), 0, p(q), p(pool), p(pool), p(tables), too_long, p(lens),
                                       p(qs), 1, 1, 1, ctypes.c_float(0.125), p(out), stream)
    assert rc == pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_launch_count() == before
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_empty_batches_are_no_ops(dtype):
    """Zero sequences, tokens or pairs: every device call returns PKV_OK, launches nothing and leaves
    the pools and outputs as they were."""
    import torch
    desc = pkv.make_desc(dtype, 2, 8, 4, 2, 64)
    dt = pkv.torch_dtype(dtype)
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    kp = torch.randn(pkv.pool_shape(desc), device="cuda", generator=g).to(dt)
    vp = torch.randn(pkv.pool_shape(desc), device="cuda", generator=g).to(dt)
    k0, v0 = kp.clone(), vp.clone()
    q = torch.zeros((0, 4, 64), dtype=dt, device="cuda")
    out = torch.zeros((0, 4, 64), dtype=dt, device="cuda")
    rows = torch.zeros((0, 2, 64), dtype=dt, device="cuda")
    tables = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    lens = torch.zeros((0,), dtype=torch.int32, device="cuda")
    slots = torch.zeros((0,), dtype=torch.int64, device="cuda")
    pairs = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    qs = torch.zeros((1,), dtype=torch.int32, device="cuda")
    dense = torch.zeros((2, 0, 2, 16, 64), dtype=dt, device="cuda")
    before = pkv.pkv_launch_count()
    pkv.pkv_kv_append(desc, 1, rows, rows, slots, kp, vp)
    pkv.pkv_copy_blocks(desc, kp, vp, pairs)
    pkv.pkv_paged_decode_attention(desc, 1, q, kp, vp, tables, lens, 0.125, out)
    pkv.pkv_paged_decode_append_attention(desc, 1, q, rows, rows, kp, vp, tables, lens, 0.125, out)
    pkv.pkv_paged_decode_attention_static(desc, 1, q, kp, vp, tables, lens, 0.125, out)
    pkv.pkv_dense_decode_attention(desc, 1, q, dense, dense, lens, 0.125, out)
    pkv.pkv_paged_prefill_attention(desc, 1, q, kp, vp, tables, lens, qs, 0, 0.125, out)
    assert pkv.pkv_launch_count() == before
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0
    assert torch.equal(kp.view(torch.uint8), k0.view(torch.uint8))
    assert torch.equal(vp.view(torch.uint8), v0.view(torch.uint8))
