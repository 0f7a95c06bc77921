"""Paged (chunked) prefill attention on the GPU against the fp64 oracle, element by element.

Chunk token i of sequence s sits at position lens[s] - n_s + i and attends causally to keys
0 .. that position through the block table ("PagedAttention e continuous batching", "01 -
Conceito", paragraph 5; "La idea de PagedAttention", step 5). Tolerance (max abs error): 1e-5
for fp32 storage, 2e-2 for fp16 / bf16 (fp32 accumulation, output rounded to the storage type).
Unreferenced pool rows and block tails are NaN-poisoned, so a stray read turns a row to NaN.
"""
import os

import numpy as np
import pytest

import oracle
from helpers import TOL, as_f64, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


def prefill_case(dtype, lens, n_new, n_q, n_kv, d, seed, n_layers=1, slack=3, max_blocks=None):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    n_new = np.asarray(n_new, dtype=np.int32)
    nb = -(-lens.astype(np.int64) // W.BLOCK)
    num_blocks = int(nb.sum()) + slack
    if max_blocks is None:
        max_blocks = max(1, int(nb.max()))
    tables = W.shuffled_tables(lens, num_blocks, seed, max_blocks=max_blocks)
    kp = W.normal_values(rng, (n_layers, num_blocks, n_kv, W.BLOCK, d), dtype)
    vp = W.normal_values(rng, (n_layers, num_blocks, n_kv, W.BLOCK, d), dtype)
    for layer in range(n_layers):
        W.poison_unreferenced(kp[layer], tables, lens, dtype)
        W.poison_unreferenced(vp[layer], tables, lens, dtype)
    qs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    q = W.normal_values(rng, (int(qs[-1]), n_q, d), dtype)
    return q, kp, vp, tables, lens, qs


def run_prefill(dtype, q, kp, vp, tables, lens, qs, scale, n_q, n_kv, d, layer=0, n_tokens=None,
                max_query_len=None):
    import torch
    desc = pkv.make_desc(dtype, kp.shape[0], kp.shape[1], n_q, n_kv, d)
    n_tok = q.shape[0] if n_tokens is None else n_tokens
    q_full = np.zeros((n_tok, n_q, d), dtype=q.dtype)
    q_full[: q.shape[0]] = q
    q_t = to_torch(q_full, dtype)
    out = torch.full_like(q_t, float("nan"))
    mql = int(np.max(np.diff(qs))) if max_query_len is None else max_query_len
    pkv.pkv_paged_prefill_attention(
        desc, layer, q_t, to_torch(kp, dtype), to_torch(vp, dtype),
        torch.from_numpy(np.ascontiguousarray(tables, np.int32)).cuda(),
        torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda(),
        torch.from_numpy(np.ascontiguousarray(qs, np.int32)).cuda(), mql, scale, out)
    flags = pkv.pkv_get_device_status()
    return as_f64(out), flags


def check(dtype, lens, n_new, n_q, n_kv, d, seed, **kw):
    q, kp, vp, tables, lens, qs = prefill_case(dtype, lens, n_new, n_q, n_kv, d, seed, **kw)
    scale = 1.0 / np.sqrt(d)
    got, flags = run_prefill(dtype, q, kp, vp, tables, lens, qs, scale, n_q, n_kv, d)
    want = oracle.paged_prefill(dtype, q, kp[0], vp[0], tables, lens, qs, scale, n_threads=THREADS)
    assert flags == 0
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - want))
    assert err <= TOL[dtype], f"max abs error {err:.3e}"
    return got, want


# whole prompts, chunks ending mid-block, single tokens, an empty chunk, chunks spanning several
# query tiles (128 rows per CTA) and several 128-key tiles with ragged tails
LENS = [300, 77, 1, 16, 17, 640, 129, 33]
NEW = [300, 45, 1, 0, 17, 200, 64, 1]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_shapes(dtype, d, group):
    check(dtype, LENS, NEW, 2 * group, 2, d, seed=300 + d + group)


@pytest.mark.parametrize("dtype,d,group", [("f16", 128, 1), ("bf16", 256, 4), ("f32", 64, 2)])
def test_chunked_equals_whole_prompt(dtype, d, group):
    """A prompt prefilled in chunks (cache growing chunk by chunk) equals one whole prefill."""
    c = 700
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [c], [c], 2 * group, 2, d, seed=41)
    scale = 1.0 / np.sqrt(d)
    whole, flags = run_prefill(dtype, q, kp, vp, tables, lens, qs, scale, 2 * group, 2, d)
    assert flags == 0
    want = oracle.paged_prefill(dtype, q, kp[0], vp[0], tables, lens, qs, scale, n_threads=THREADS)
    assert np.max(np.abs(whole - want)) <= TOL[dtype]
    start = 0
    for chunk in (256, 256, 129, 59):
        part, flags = run_prefill(dtype, q[start:start + chunk], kp, vp, tables, [start + chunk], [0, chunk],
                                  scale, 2 * group, 2, d)
        assert flags == 0
        err = np.max(np.abs(part - want[start:start + chunk]))
        assert err <= TOL[dtype], f"chunk at {start}: {err:.3e}"
        start += chunk


def test_single_token_chunks_equal_decode():
    """A chunk of one token per sequence gives the decode kernel's result (same rows, same rule)."""
    import torch
    dtype, n_q, n_kv, d = "bf16", 8, 2, 128
    lens = [1, 16, 17, 300, 1025]
    q, kp, vp, tables, lens_a, qs = prefill_case(dtype, lens, [1] * len(lens), n_q, n_kv, d, seed=9)
    scale = 1.0 / np.sqrt(d)
    got, flags = run_prefill(dtype, q, kp, vp, tables, lens_a, qs, scale, n_q, n_kv, d)
    assert flags == 0
    desc = pkv.make_desc(dtype, 1, kp.shape[1], n_q, n_kv, d)
    q_t = to_torch(q, dtype)
    out = torch.full_like(q_t, float("nan"))
    t_t = torch.from_numpy(np.ascontiguousarray(tables, np.int32)).cuda()
    l_t = torch.from_numpy(np.ascontiguousarray(lens_a, np.int32)).cuda()
    pkv.pkv_paged_decode_attention(desc, 0, q_t, to_torch(kp, dtype), to_torch(vp, dtype), t_t, l_t, scale, out,
                                   pkv.alloc_workspace(desc, len(lens), tables.shape[1]))
    assert np.max(np.abs(got - as_f64(out))) <= TOL[dtype]


def test_layer_offset_and_unowned_rows():
    """Layer 2 of a 3-layer pool; rows after query_start[n_seqs] keep their contents."""
    dtype, n_q, n_kv, d = "f16", 4, 4, 64
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [90, 40], [50, 40], n_q, n_kv, d, seed=12, n_layers=3)
    scale = 0.125
    got, flags = run_prefill(dtype, q, kp, vp, tables, lens, qs, scale, n_q, n_kv, d, layer=2, n_tokens=100)
    assert flags == 0
    want = oracle.paged_prefill(dtype, q, kp[2], vp[2], tables, lens, qs, scale)
    assert np.max(np.abs(got[:90] - want)) <= TOL[dtype]
    assert np.all(np.isnan(got[90:]))


def test_causality_on_device():
    """Changing the key/value of position 100 leaves rows < 100 bit-identical and moves the rest."""
    dtype, n_q, n_kv, d = "bf16", 8, 2, 128
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [260], [260], n_q, n_kv, d, seed=13)
    a, _ = run_prefill(dtype, q, kp, vp, tables, lens, qs, 0.1, n_q, n_kv, d)
    blk, off = tables[0, 100 // 16], 100 % 16
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[0, blk, :, off, :] = kp[0, tables[0, 0], :, 0, :]
    vp2[0, blk, :, off, :] = vp[0, tables[0, 0], :, 1, :]
    b, _ = run_prefill(dtype, q, kp2, vp2, tables, lens, qs, 0.1, n_q, n_kv, d)
    np.testing.assert_array_equal(a[:100], b[:100])
    assert np.all(np.abs(a[100:] - b[100:]).max(axis=(1, 2)) > 0)


def test_physical_permutation_is_bit_identical():
    dtype, n_q, n_kv, d = "f16", 8, 8, 128
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [500, 130], [200, 130], n_q, n_kv, d, seed=14)
    a, _ = run_prefill(dtype, q, kp, vp, tables, lens, qs, 0.1, n_q, n_kv, d)
    perm = np.random.default_rng(3).permutation(kp.shape[1])
    inv = np.argsort(perm)
    t2 = tables.copy()
    for s in range(len(lens)):
        nb = -(-int(lens[s]) // 16)
        t2[s, :nb] = inv[tables[s, :nb]]
    b, _ = run_prefill(dtype, q, kp[:, perm], vp[:, perm], t2, lens, qs, 0.1, n_q, n_kv, d)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_bad_values_are_flagged_not_read(dtype):
    """A table entry out of range is skipped (masked) and flagged; a chunk longer than its
    context or than max_query_len leaves that sequence's rows unwritten and is flagged."""
    n_q, n_kv, d = 4, 2, 64
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [100, 64], [100, 64], n_q, n_kv, d, seed=15)
    bad = tables.copy()
    bad[0, 3] = kp.shape[1] + 7        # keys 48..63 of sequence 0 are skipped
    got, flags = run_prefill(dtype, q, kp, vp, bad, lens, qs, 0.125, n_q, n_kv, d)
    assert flags & pkv.PKV_DEV_BAD_BLOCK_ID
    assert np.all(np.isfinite(got))
    ok = oracle.paged_prefill(dtype, q, kp[0], vp[0], tables, lens, qs, 0.125)
    assert np.max(np.abs(got[:48] - ok[:48])) <= TOL[dtype]   # rows before the skipped block agree
    assert np.max(np.abs(got[100:] - ok[100:])) <= TOL[dtype]  # the other sequence is untouched
    # chunk of sequence 1 longer than its context: its rows stay NaN, sequence 0 is computed
    got, flags = run_prefill(dtype, q, kp, vp, tables, [100, 60], qs, 0.125, n_q, n_kv, d)
    assert flags & pkv.PKV_DEV_BAD_QUERY_RANGE
    assert np.all(np.isnan(got[100:])) and np.max(np.abs(got[:100] - ok[:100])) <= TOL[dtype]
    # max_query_len smaller than a chunk: flagged, no row of that sequence written
    got, flags = run_prefill(dtype, q, kp, vp, tables, lens, qs, 0.125, n_q, n_kv, d, max_query_len=64)
    assert flags & pkv.PKV_DEV_BAD_QUERY_RANGE
    assert np.all(np.isnan(got[:100])) and np.max(np.abs(got[100:] - ok[100:])) <= TOL[dtype]


def test_host_argument_errors():
    import torch
    desc = pkv.make_desc("f16", 1, 8, 2, 2, 64)
    q = torch.zeros((4, 2, 64), dtype=torch.float16, device="cuda")
    pool = torch.zeros(pkv.pool_shape(desc), dtype=torch.float16, device="cuda")
    t = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    ln = torch.full((1,), 4, dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):   # max_query_len > n_tokens
        pkv.pkv_paged_prefill_attention(desc, 0, q, pool, pool, t, ln, qs, 5, 1.0, q.clone())
    with pytest.raises(RuntimeError):   # layer out of range
        pkv.pkv_paged_prefill_attention(desc, 1, q, pool, pool, t, ln, qs, 4, 1.0, q.clone())
    out = q.clone()
    pkv.pkv_paged_prefill_attention(desc, 0, q, pool, pool, t, ln, qs, 0, 1.0, out)   # no-op
    assert pkv.pkv_get_device_status() == 0


@pytest.mark.parametrize("trial", range(12))
def test_random_batches_stress(trial):
    """Random mixes of sequences, chunk lengths, contexts and GQA groups (query tiles with no rows,
    ragged last key tiles and chunks shorter than a tile appear throughout; at head_dim 256 CTA
    pairs, one of whose query tiles may have no rows or fewer keys than the other). Every output
    against the oracle; the status word must stay clean (no bounded wait may give up)."""
    rng = np.random.default_rng(1000 + trial)
    dtype = ["bf16", "f16"][trial % 2]
    d = [256, 256, 128, 64][trial % 4]
    group = int(rng.choice([1, 2, 4, 8]))
    n_kv = int(rng.integers(1, 3))
    n_seqs = int(rng.integers(1, 5))
    lens, new = [], []
    for _ in range(n_seqs):
        c = int(rng.integers(1, 1200))
        n = int(rng.integers(0, min(c, 700) + 1))
        lens.append(c)
        new.append(n)
    if sum(new) == 0:
        new[0] = lens[0]
    check(dtype, lens, new, group * n_kv, n_kv, d, seed=2000 + trial)


@pytest.mark.parametrize("d,group", [(256, 4), (128, 1)])
def test_cuda_graph_replay_of_prefill(d, group):
    """A captured prefill launch (CTA pairs at head_dim 256) replays bit-identically to the eager
    call, several times."""
    import torch
    dtype, n_kv = "bf16", 2
    n_q = n_kv * group
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [700, 1300], [300, 500], n_q, n_kv, d, seed=77)
    desc = pkv.make_desc(dtype, 1, kp.shape[1], n_q, n_kv, d)
    args = [to_torch(q, dtype), to_torch(kp, dtype), to_torch(vp, dtype),
            torch.from_numpy(np.ascontiguousarray(tables, np.int32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda(),
            torch.from_numpy(np.ascontiguousarray(qs, np.int32)).cuda()]
    mql = int(np.max(np.diff(qs)))
    scale = 1.0 / np.sqrt(d)
    eager = torch.empty_like(args[0])
    pkv.pkv_paged_prefill_attention(desc, 0, args[0], args[1], args[2], args[3], args[4], args[5], mql, scale, eager)
    out = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.pkv_paged_prefill_attention(desc, 0, args[0], args[1], args[2], args[3], args[4], args[5], mql, scale,
                                        out)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pkv.pkv_get_device_status() == 0
    want = oracle.paged_prefill(dtype, q, kp[0], vp[0], tables, lens, qs, scale, n_threads=THREADS)
    assert np.max(np.abs(as_f64(out) - want)) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_pair_skips_bad_blocks_in_either_half(dtype):
    """head_dim 256 runs as CTA pairs, each CTA loading half of every 128-key tile (blocks 0-3 the
    even CTA, 4-7 the odd one) and half of every V block's columns. Out-of-range table entries in
    both halves are skipped, their keys masked, and flagged. Attention is a sum over the set of
    visible keys, so a query at position p equals a decode over the sequence with the skipped blocks
    removed and |{0..p} minus the skipped positions| keys (which stay a prefix in that order)."""
    n_q, n_kv, d = 8, 2, 256
    c, n = 700, 300                                          # chunk at positions 400 .. 699
    q, kp, vp, tables, lens, qs = prefill_case(dtype, [c], [n], n_q, n_kv, d, seed=23)
    skipped = [30, 33]                                       # tile 3 block 6 (odd CTA), tile 4 block 1 (even)
    bad = tables.copy()
    for i, b in enumerate(skipped):
        bad[0, b] = kp.shape[1] + 5 + i
    scale = 1.0 / np.sqrt(d)
    got, flags = run_prefill(dtype, q, kp, vp, bad, lens, qs, scale, n_q, n_kv, d)
    assert flags & pkv.PKV_DEV_BAD_BLOCK_ID
    assert np.all(np.isfinite(got))
    reduced = np.delete(tables[0], skipped)
    pos = np.arange(c - n, c)
    visible = pos + 1 - sum(np.clip(pos + 1 - 16 * b, 0, 16) for b in skipped)
    t_rep = np.ascontiguousarray(np.broadcast_to(reduced, (n, reduced.shape[0])))
    want = oracle.paged_decode(dtype, q, kp[0], vp[0], t_rep, visible.astype(np.int32), scale)
    assert np.max(np.abs(got - want)) <= TOL[dtype]


def test_prefill_wave_tokens_fill_whole_waves():
    """pkv_prefill_wave_tokens: the chunk tokens of one sequence that fill exactly one wave of the
    prefill grid (SMs x CTAs per SM x tokens per CTA / KV heads); at head_dim 256 one CTA holds an SM
    (its shared and tensor memory), so the wave is one CTA per SM."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    d256 = pkv.make_desc("bf16", 16, 4096, 16, 4, 256)
    w = pkv.pkv_prefill_wave_tokens(d256)
    # one CTA per SM, in pairs: all SMs where every SM finds a partner (a GB300), else whole pairs fewer
    pairs = w * 4 // (128 // 4) // 2
    assert w == sms * (128 // 4) // 4 or (w < sms * (128 // 4) // 4 and w == pairs * 2 * (128 // 4) // 4)
    assert pkv.wave_aligned_chunk(d256, 2048) == w * max(1, round(2048 / w))
    for dtype, n_q, n_kv, d in [("f16", 32, 32, 128), ("bf16", 8, 8, 64), ("f32", 4, 2, 64)]:
        desc = pkv.make_desc(dtype, 1, 1024, n_q, n_kv, d)
        w = pkv.pkv_prefill_wave_tokens(desc)
        per_cta = (32 if dtype == "f32" else 128) // (n_q // n_kv)
        ctas = w * n_kv // per_cta
        assert w >= 1 and ctas % sms == 0 and ctas // sms >= 1, (dtype, d, w)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pools_past_32_bit_rows_are_refused(dtype):
    """A layer of 2^31 rows or more (num_blocks x n_kv_heads x 16) cannot be addressed by the tensor
    copies' 32-bit row coordinates: prefill and decode return PKV_ERR_UNSUPPORTED before launching.
    The descriptor claims such a pool over small buffers; every other argument keeps a launch, were
    one to happen, inside them (one sequence of one token in block 0)."""
    import ctypes
    import torch
    n_kv, d = 2, 64
    huge = pkv.make_desc(dtype, 1, (1 << 31) // (n_kv * 16), 2, n_kv, d)
    dt = pkv.torch_dtype(dtype)
    small = torch.zeros((1, 4, n_kv, 16, d), dtype=dt, device="cuda")
    q = torch.zeros((1, 2, d), dtype=dt, device="cuda")
    out = torch.zeros_like(q)
    tables = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones((1,), dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ws = torch.zeros((1 << 20,), dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    L = pkv.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.pkv_paged_prefill_attention(ctypes.byref(huge), 0, p(q), p(small), p(small), p(tables), 1, p(lens),
                                       p(qs), 1, 1, 1, ctypes.c_float(0.125), p(out), stream)
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    rc = L.pkv_paged_decode_attention(ctypes.byref(huge), 0, p(q), p(small), p(small), p(tables), 1, p(lens), 1,
                                      ctypes.c_float(0.125), p(out), p(ws), ctypes.c_size_t(ws.numel()), stream)
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    rc = L.pkv_paged_decode_attention_static(ctypes.byref(huge), 0, p(q), p(small), p(small), p(tables), 1, p(lens),
                                             1, ctypes.c_float(0.125), p(out), stream)
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0
