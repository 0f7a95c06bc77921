"""Paged decode attention on the GPU against the fp64 oracle, element by element.

Tolerance (max abs error): 1e-5 for fp32 storage, 2e-2 for fp16 / bf16 storage (fp32
accumulation, output rounded to the storage type). Unused pool rows are NaN-poisoned in
every case, so a stray read of a tail row or an unreferenced block turns the output to NaN.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, as_f64, paged_case, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_decode(dtype, q, kp, vp, tables, lens, scale, n_q, n_kv, d, layer=0, num_blocks=None):
    import torch
    n_layers = kp.shape[0]
    num_blocks = kp.shape[1] if num_blocks is None else num_blocks
    desc = pkv.make_desc(dtype, n_layers, num_blocks, n_q, n_kv, d)
    k_t, v_t = to_torch(kp, dtype), to_torch(vp, dtype)
    q_t = to_torch(q, dtype)
    t_t = torch.from_numpy(np.ascontiguousarray(tables, dtype=np.int32)).cuda()
    l_t = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    out = torch.full_like(q_t, float("nan"))
    ws = pkv.alloc_workspace(desc, len(lens), tables.shape[1])
    pkv.pkv_paged_decode_attention(desc, layer, q_t, k_t, v_t, t_t, l_t, scale, out, ws)
    flags = pkv.pkv_get_device_status()
    return as_f64(out), flags


def check(dtype, lens, n_q, n_kv, d, seed, n_layers=1, layer=0, max_blocks=None):
    q, kp, vp, tables, lens, nb = paged_case(dtype, lens, n_q, n_kv, d, seed, n_layers=n_layers,
                                             max_blocks=max_blocks)
    scale = 1.0 / np.sqrt(d)
    got, flags = run_decode(dtype, q, kp, vp, tables, lens, scale, n_q, n_kv, d, layer=layer)
    want = oracle.paged_decode(dtype, q, kp[layer], vp[layer], tables, lens, scale)
    assert flags == 0
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - want))
    assert err <= TOL[dtype], f"max abs error {err:.3e}"
    return got, want


def test_tiny_config():
    wl = W.tiny()
    check(wl.dtype, wl.context_lens, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.seed)


RAGGED = [1, 15, 16, 17, 100, 511, 512, 513, 1500]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_shapes_split_k(dtype, d, group):
    """Many tiles, ragged tails, split-K partitions (the small grid shrinks partitions)."""
    n_kv = 2
    check(dtype, RAGGED, n_kv * group, n_kv, d, seed=100 + d + group)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d,group", [(64, 1), (128, 4), (256, 8)])
def test_shapes_single_partition(dtype, d, group):
    """Contexts of at most 4 blocks: one partition per sequence, output written directly."""
    check(dtype, [1, 2, 15, 16, 17, 33, 48, 64], 2 * group, 2, d, seed=200 + d)


def test_many_sequences_large_grid():
    """Large grid (no partition shrinking): partitions of 32 blocks, 64 sequences."""
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 1400, size=64)
    check("f16", lens, 8, 8, 128, seed=5)


def test_layer_offset():
    check("bf16", [40, 300, 17], 8, 2, 128, seed=6, n_layers=3, layer=2)


def test_wide_table_and_zero_context():
    """ctx = 0 gives a zero row; entries past ceil(ctx/16) are never read (they hold -1)."""
    got, _ = check("f16", [0, 5, 0, 160], 4, 4, 64, seed=7, max_blocks=40)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)


def test_full_table_context():
    check("f32", [64, 64], 2, 1, 64, seed=8, max_blocks=4)


def test_single_token_is_exact_value_row():
    q, kp, vp, tables, lens, nb = paged_case("f32", [1, 1, 1], 4, 2, 128, seed=9)
    got, flags = run_decode("f32", q, kp, vp, tables, lens, 0.1, 4, 2, 128)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(got[s, h], vp[0, tables[s, 0], h // 2, 0].astype(np.float64))


def test_equal_keys_average_values():
    q, kp, vp, tables, lens, nb = paged_case("f32", [700], 1, 1, 64, seed=10, poison=False)
    kp[...] = kp[0, 0, 0, 0]
    got, _ = run_decode("f32", q, kp, vp, tables, lens, 0.125, 1, 1, 64)
    rows = np.stack([vp[0, tables[0, j // 16], 0, j % 16] for j in range(700)]).astype(np.float64)
    np.testing.assert_allclose(got[0, 0], rows.mean(axis=0), rtol=0, atol=1e-5)


def test_peaky_softmax():
    q, kp, vp, tables, lens, nb = paged_case("f16", [300, 2000], 4, 4, 128, seed=11)
    q = (q.astype(np.float32) * 8).astype(np.float16)
    got, _ = run_decode("f16", q, kp, vp, tables, lens, 1 / np.sqrt(128), 4, 4, 128)
    want = oracle.paged_decode("f16", q, kp[0], vp[0], tables, lens, 1 / np.sqrt(128))
    assert np.max(np.abs(got - want)) <= TOL["f16"]


def test_physical_permutation_is_bit_identical():
    q, kp, vp, tables, lens, nb = paged_case("bf16", [700, 33, 1200], 8, 2, 128, seed=12)
    base, _ = run_decode("bf16", q, kp, vp, tables, lens, 0.1, 8, 2, 128)
    perm = np.random.default_rng(13).permutation(nb)
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[:, perm], vp2[:, perm] = kp, vp
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    got, _ = run_decode("bf16", q, kp2, vp2, t2, lens, 0.1, 8, 2, 128)
    assert np.array_equal(got, base)


def test_shared_prefix_equals_private_copy():
    q, kp, vp, tables, lens, nb = paged_case("f16", [600, 600], 4, 4, 64, seed=14, slack=40, poison=False)
    # make sequence 1's first 30 blocks hold the same rows as sequence 0's (private copies)
    kp[:, tables[1, :30]] = kp[:, tables[0, :30]]
    vp[:, tables[1, :30]] = vp[:, tables[0, :30]]
    q[1] = q[0]
    priv, _ = run_decode("f16", q, kp, vp, tables, lens, 0.125, 4, 4, 64)
    shared_t = tables.copy()
    shared_t[1, :30] = tables[0, :30]                  # now they point at the same blocks
    shared, _ = run_decode("f16", q, kp, vp, shared_t, lens, 0.125, 4, 4, 64)
    assert np.array_equal(priv, shared)


def test_bad_table_entry_and_length_are_flagged_not_read():
    q, kp, vp, tables, lens, nb = paged_case("f16", [40, 40], 2, 2, 64, seed=15, max_blocks=3)
    bad = tables.copy()
    bad[0, 1] = nb + 7                                 # outside the pool
    got, flags = run_decode("f16", q, kp, vp, bad, lens, 0.125, 2, 2, 64)
    assert flags & pkv.PKV_DEV_BAD_BLOCK_ID
    want = oracle.paged_decode("f16", q[1:], kp[0], vp[0], tables[1:], lens[1:], 0.125)
    assert np.max(np.abs(got[1:] - want)) <= TOL["f16"]   # the other sequence is untouched
    lens2 = lens.copy()
    lens2[1] = 3 * 16 + 5                              # longer than the table
    _, flags = run_decode("f16", q, kp, vp, tables, lens2, 0.125, 2, 2, 64)
    assert flags & pkv.PKV_DEV_BAD_CONTEXT_LEN
    assert pkv.pkv_get_device_status() == 0            # reading clears the word


@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("f16", 8, 8, 128), ("bf16", 16, 4, 256), ("f32", 4, 2, 64),
                                              ("f16", 4, 1, 64)])
def test_fused_append_equals_separate_calls(dtype, n_q, n_kv, d):
    """pkv_paged_decode_append_attention == pkv_kv_append(slot of position len-1) + decode, bit for bit."""
    import torch
    lens = [1, 16, 17, 40, 513, 1500, 0]
    q, kp, vp, tables, lens_a, nb = paged_case(dtype, lens, n_q, n_kv, d, seed=41, n_layers=2)
    rng = np.random.default_rng(42)
    kn = W.normal_values(rng, (len(lens), n_kv, d), dtype)
    vn = W.normal_values(rng, (len(lens), n_kv, d), dtype)
    desc = pkv.make_desc(dtype, 2, nb, n_q, n_kv, d)
    t_t = torch.from_numpy(tables).cuda()
    l_t = torch.from_numpy(lens_a).cuda()
    ws = pkv.alloc_workspace(desc, len(lens), tables.shape[1])
    # separate calls: append at the slot of the last position (padding for empty sequences)
    slots = np.array([tables[s, (n - 1) // 16] * 16 + (n - 1) % 16 if n > 0 else -1 for s, n in enumerate(lens_a)],
                     dtype=np.int64)
    k1, v1 = to_torch(kp, dtype), to_torch(vp, dtype)
    out1 = torch.full_like(to_torch(q, dtype), float("nan"))
    pkv.pkv_kv_append(desc, 1, to_torch(kn, dtype), to_torch(vn, dtype), torch.from_numpy(slots).cuda(), k1, v1)
    pkv.pkv_paged_decode_attention(desc, 1, to_torch(q, dtype), k1, v1, t_t, l_t, 0.1, out1, ws)
    k2, v2 = to_torch(kp, dtype), to_torch(vp, dtype)
    out2 = torch.full_like(out1, float("nan"))
    pkv.pkv_paged_decode_append_attention(desc, 1, to_torch(q, dtype), to_torch(kn, dtype), to_torch(vn, dtype),
                                          k2, v2, t_t, l_t, 0.1, out2, ws)
    assert pkv.pkv_get_device_status() == 0
    for a_, b_ in ((k1, k2), (v1, v2)):
        assert torch.equal(a_.contiguous().view(torch.uint8), b_.contiguous().view(torch.uint8))
    assert torch.equal(out1.contiguous().view(torch.uint8), out2.contiguous().view(torch.uint8))
    # and against the oracle, whose pools receive the same rows at the same slots
    want_k, want_v = kp.copy(), vp.copy()
    oracle.kv_append(kn, vn, slots, want_k[1], want_v[1])
    want = oracle.paged_decode(dtype, q, want_k[1], want_v[1], tables, lens_a, 0.1)
    got = as_f64(out2)
    assert np.max(np.abs(got - want)) <= TOL[dtype]


def test_workspace_garbage_and_reuse_across_shapes():
    """Split-K arrival counters self-initialise: a garbage-filled workspace, reused by calls of
    different shapes (whose counters land on each other's partials), gives correct rows."""
    import torch
    ws = torch.randint(-2 ** 31, 2 ** 31 - 1, (4 << 20,), dtype=torch.int32, device="cuda")
    for dtype, lens, n_q, n_kv, d, seed in (("f16", [700, 1500, 33], 8, 2, 128, 51),
                                            ("bf16", [2100, 5, 900, 64, 1200], 4, 4, 64, 52),
                                            ("f32", [1000, 17], 2, 1, 256, 53),
                                            ("f16", [700, 1500, 33], 8, 2, 128, 54)):
        q, kp, vp, tables, lens_a, nb = paged_case(dtype, lens, n_q, n_kv, d, seed)
        desc = pkv.make_desc(dtype, 1, nb, n_q, n_kv, d)
        assert pkv.pkv_decode_workspace_bytes(desc, len(lens), tables.shape[1]) > 0
        out = torch.full_like(to_torch(q, dtype), float("nan"))
        pkv.pkv_paged_decode_attention(desc, 0, to_torch(q, dtype), to_torch(kp, dtype), to_torch(vp, dtype),
                                       torch.from_numpy(tables).cuda(), torch.from_numpy(lens_a).cuda(), 0.1, out,
                                       ws)
        assert pkv.pkv_get_device_status() == 0
        want = oracle.paged_decode(dtype, q, kp[0], vp[0], tables, lens_a, 0.1)
        assert np.max(np.abs(as_f64(out) - want)) <= TOL[dtype]


def test_cuda_graph_replay_of_split_decode():
    """A captured decode launch replays with the same call tag; the merging CTA's counter reset
    keeps every replay correct."""
    import torch
    dtype, n_q, n_kv, d = "bf16", 8, 2, 128
    q, kp, vp, tables, lens, nb = paged_case(dtype, [1500, 3000, 70], n_q, n_kv, d, seed=55)
    desc = pkv.make_desc(dtype, 1, nb, n_q, n_kv, d)
    args = [to_torch(q, dtype), to_torch(kp, dtype), to_torch(vp, dtype), torch.from_numpy(tables).cuda(),
            torch.from_numpy(lens).cuda()]
    ws = pkv.alloc_workspace(desc, 3, tables.shape[1])
    eager = torch.empty_like(args[0])
    pkv.pkv_paged_decode_attention(desc, 0, args[0], args[1], args[2], args[3], args[4], 0.1, eager, ws)
    out = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.pkv_paged_decode_attention(desc, 0, args[0], args[1], args[2], args[3], args[4], 0.1, out, ws)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert pkv.pkv_get_device_status() == 0


@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("f16", 4, 2, 64), ("bf16", 8, 1, 128)])
def test_large_batch(dtype, n_q, n_kv, d):
    """1,100 sequences of mostly short contexts (many idle partitions), split-K included."""
    rng = np.random.default_rng(61)
    lens = rng.integers(0, 90, size=1100)
    lens[:8] = (1, 16, 17, 300, 700, 1100, 0, 64)
    check(dtype, lens, n_q, n_kv, d, seed=61)


def test_bounded_wait_gives_up_and_context_stays_usable():
    """Failure detection without a fault: a wait on an mbarrier nothing completes gives up after its
    limit, the kernel records PKV_DEV_WAIT_TIMEOUT and returns; the context then runs a normal
    decode that matches the oracle."""
    import time
    assert pkv.pkv_get_device_status() == 0
    t0 = time.perf_counter()
    pkv.pkv_selftest_wait_timeout()
    flags = pkv.pkv_get_device_status()
    waited = time.perf_counter() - t0
    assert flags == pkv.PKV_DEV_WAIT_TIMEOUT
    assert 0.5 < waited < 10.0
    assert pkv.pkv_get_device_status() == 0          # reading cleared it
    check("f16", [5, 40, 300], 4, 2, 64, seed=31)     # the context is still healthy


def test_workspace_query_and_launch_use_the_devices_sm_count():
    """The workspace query reads this device's SM count and the decode kernel's occupancy; a
    workspace of exactly that size is accepted and one byte less is refused before launch, so query
    and launch agree."""
    import ctypes

    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    lens = [3000, 17, 900]
    q, kp, vp, tables, lens, nb = paged_case("bf16", lens, 16, 4, 256, seed=77)
    desc = pkv.make_desc("bf16", 1, nb, 16, 4, 256)
    per_sm, got_sms = pkv.pkv_decode_ctas_per_sm(desc)
    assert got_sms == sms and 1 <= per_sm <= 32
    mb = tables.shape[1]
    need = pkv.pkv_decode_workspace_bytes(desc, len(lens), mb)
    assert need == pkv.pkv_decode_split_geometry(desc, len(lens), mb, sms, per_sm)[2] > 0
    k_t, v_t, q_t = to_torch(kp, "bf16"), to_torch(vp, "bf16"), to_torch(q, "bf16")
    t_t = torch.from_numpy(np.ascontiguousarray(tables)).cuda()
    l_t = torch.from_numpy(lens).cuda()
    ws = torch.zeros(need // 4 + 4, dtype=torch.float32, device="cuda")
    out = torch.full_like(q_t, float("nan"))
    L = pkv.lib()
    vp_ = ctypes.c_void_p

    def call(nbytes):
        return L.pkv_paged_decode_attention(ctypes.byref(desc), 0, vp_(q_t.data_ptr()), vp_(k_t.data_ptr()),
                                            vp_(v_t.data_ptr()), vp_(t_t.data_ptr()), mb, vp_(l_t.data_ptr()),
                                            len(lens), ctypes.c_float(1 / 16), vp_(out.data_ptr()),
                                            vp_(ws.data_ptr()), nbytes, vp_(0))
    assert call(need - 1) == pkv.PKV_ERR_INVALID_ARG
    assert call(need) == pkv.PKV_OK
    assert pkv.pkv_get_device_status() == 0
    want = oracle.paged_decode("bf16", q, kp[0], vp[0], tables, lens, 1 / 16)
    assert np.max(np.abs(as_f64(out) - want)) <= TOL["bf16"]


def test_pools_on_the_host_are_refused_before_launch():
    """The tensor copies read the pools directly: host memory is refused (PKV_ERR_INVALID_ARG)."""
    import ctypes

    import torch
    q, kp, vp, tables, lens, nb = paged_case("f16", [40, 70], 4, 4, 64, seed=78)
    desc = pkv.make_desc("f16", 1, nb, 4, 4, 64)
    k_host = torch.from_numpy(np.ascontiguousarray(kp)).pin_memory()
    v_t, q_t = to_torch(vp, "f16"), to_torch(q, "f16")
    t_t = torch.from_numpy(np.ascontiguousarray(tables)).cuda()
    l_t = torch.from_numpy(lens).cuda()
    qs = torch.tensor([0, 40, 80], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q_t)
    before = pkv.pkv_launch_count()
    L = pkv.lib()
    vp_ = ctypes.c_void_p
    rc = L.pkv_paged_decode_attention(ctypes.byref(desc), 0, vp_(q_t.data_ptr()), vp_(k_host.data_ptr()),
                                      vp_(v_t.data_ptr()), vp_(t_t.data_ptr()), tables.shape[1],
                                      vp_(l_t.data_ptr()), 2, ctypes.c_float(0.125), vp_(out.data_ptr()),
                                      vp_(0), 0, vp_(0))
    assert rc == pkv.PKV_ERR_INVALID_ARG
    q80 = torch.zeros((80, 4, 64), dtype=torch.float16, device="cuda")
    o80 = torch.empty_like(q80)
    rc = L.pkv_paged_prefill_attention(ctypes.byref(desc), 0, vp_(q80.data_ptr()), vp_(k_host.data_ptr()),
                                       vp_(v_t.data_ptr()), vp_(t_t.data_ptr()), tables.shape[1],
                                       vp_(l_t.data_ptr()), vp_(qs.data_ptr()), 2, 80, 40, ctypes.c_float(0.125),
                                       vp_(o80.data_ptr()), vp_(0))
    assert rc == pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_launch_count() == before
    assert pkv.pkv_get_device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_one_wave_long_partitions(dtype):
    """Few sequences with long contexts take the one-wave split: partitions far longer than 64
    blocks, whose table entries the kernel streams in chunks of 32 per warp (several chunks per
    warp here). Against the oracle, also with a block id out of range deep inside a partition."""
    n_q, n_kv, d = 8, 8, 64
    probe = pkv.make_desc(dtype, 1, 1000, n_q, n_kv, d)
    per_sm, sms = pkv.pkv_decode_ctas_per_sm(probe)
    parts = sms * per_sm // (5 * n_kv)                  # 5 sequences x 8 KV heads = 40 pairs
    top = 16 * 130 * parts                              # partitions of ~130 blocks: 5 chunks per warp
    lens = [top, top // 2 + 3, 1, top - 5, 17]
    q, kp, vp, tables, lens, nb = paged_case(dtype, lens, n_q, n_kv, d, seed=91)
    desc = pkv.make_desc(dtype, 1, nb, n_q, n_kv, d)
    bpp, n_parts, _ = pkv.pkv_decode_split_geometry(desc, len(lens), tables.shape[1], sms, per_sm)
    assert bpp > 4 * 32 and n_parts == parts
    scale = 1.0 / np.sqrt(d)
    got, flags = run_decode(dtype, q, kp, vp, tables, lens, scale, n_q, n_kv, d)
    want = oracle.paged_decode(dtype, q, kp[0], vp[0], tables, lens, scale)
    assert flags == 0 and np.all(np.isfinite(got))
    assert np.max(np.abs(got - want)) <= TOL[dtype]
    # a bad table entry deep inside a partition is skipped (its rows masked) and flagged
    bad = tables.copy()
    bad[0, 300] = nb + 5
    got_bad, flags = run_decode(dtype, q, kp, vp, bad, lens, scale, n_q, n_kv, d)
    assert flags & pkv.PKV_DEV_BAD_BLOCK_ID
    # attention is a sum over the set of visible keys: dropping the full block 300 (16 keys) equals
    # the same sequence without that table entry and 16 positions shorter (the tail block unchanged)
    t0 = np.delete(tables[:1], 300, axis=1)
    want0 = oracle.paged_decode(dtype, q[:1], kp[0], vp[0], t0, np.array([lens[0] - 16], np.int32), scale)
    assert np.all(np.isfinite(got_bad))
    assert np.max(np.abs(got_bad[:1] - want0)) <= TOL[dtype]
    assert np.max(np.abs(got_bad[1:] - want[1:])) <= TOL[dtype]   # other sequences unaffected
