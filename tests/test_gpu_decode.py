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
