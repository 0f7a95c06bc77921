"""Pins for the oracle's paged prefill attention, checked against things other than itself.

"PagedAttention e continuous batching" ("01 - Conceito", paragraph 5) slices a long prompt into
chunks; "La idea de PagedAttention" (step 5) has the kernel gather the rows through the block
table. The chunk's tokens are the sequence's newest, at positions lens - n .. lens - 1, each
attending causally to positions 0 .. its own.

* a special case that reduces to library routines: scipy softmax over a dense cache with an
  explicit lower-triangular mask (numpy.tril), for every dtype, head size and GQA group;
* the pinned decode oracle: a chunk of one token is exactly one decode query;
* invariants: a prompt prefilled in chunks equals the whole prompt prefilled at once; the
  physical placement of blocks does not matter; keys after a query's position cannot change it
  and keys at or before it do; the first position of a prompt returns its own V row exactly.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from paged_kv_cache_258_gb300 import workloads as W
from test_oracle_pins import decode_np, scatter_dense

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def prefill_case(dtype, lens, n_new, n_q, n_kv, d, seed, slack=4):
    """Dense rows per sequence, their paged pools, shuffled tables and packed chunk queries."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    n_new = np.asarray(n_new, dtype=np.int32)
    num_blocks = int(np.sum(-(-lens // W.BLOCK))) + slack
    max_blocks = max(1, int(np.max(-(-lens // W.BLOCK))))
    tables = W.shuffled_tables(lens, num_blocks, seed, max_blocks=max_blocks)
    kd = [W.normal_values(rng, (int(n), n_kv, d), dtype) for n in lens]
    vd = [W.normal_values(rng, (int(n), n_kv, d), dtype) for n in lens]
    qs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    q = W.normal_values(rng, (int(qs[-1]), n_q, d), dtype)
    kp = scatter_dense(kd, tables, num_blocks, dtype)
    vp = scatter_dense(vd, tables, num_blocks, dtype)
    return q, kd, vd, kp, vp, tables, lens, qs


def causal_reference(q, kd, vd, lens, qs, scale, dtype):
    """scipy softmax with an explicit causal mask (numpy.tril) over each dense cache."""
    n_tok, n_q, d = q.shape
    out = np.zeros((n_tok, n_q, d))
    for s in range(len(lens)):
        c, n = int(lens[s]), int(qs[s + 1] - qs[s])
        if n == 0:
            continue
        grp = n_q // kd[s].shape[1]
        # mask[i, j] = key j visible to chunk query i, which sits at position c - n + i
        mask = np.tril(np.ones((n, c), dtype=bool), k=c - n)
        for h in range(n_q):
            K = decode_np(dtype, kd[s][:, h // grp, :])
            V = decode_np(dtype, vd[s][:, h // grp, :])
            Q = decode_np(dtype, q[qs[s]:qs[s + 1], h, :])
            Z = np.where(mask, scale * (Q @ K.T), -np.inf)
            out[qs[s]:qs[s + 1], h] = softmax(Z, axis=1) @ V
    return out


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d,n_q,n_kv", [(64, 2, 2), (128, 4, 1), (256, 8, 2), (64, 8, 1)])
def test_prefill_equals_masked_dense_softmax(dtype, d, n_q, n_kv):
    lens, n_new = [37, 16, 70, 5, 1], [37, 9, 20, 0, 1]   # whole prompt, chunk, empty chunk
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, lens, n_new, n_q, n_kv, d, seed=d + n_q)
    scale = 1.0 / np.sqrt(d)
    got = oracle.paged_prefill(dtype, q, kp, vp, tables, lens, qs, scale)
    want = causal_reference(q, kd, vd, lens, qs, scale, dtype)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token_chunk_is_decode(dtype):
    lens = [1, 17, 64, 200]
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, lens, [1, 1, 1, 1], 4, 2, 64, seed=3)
    got = oracle.paged_prefill(dtype, q, kp, vp, tables, lens, qs, 0.125)
    want = oracle.paged_decode(dtype, q, kp, vp, tables, lens, 0.125)
    np.testing.assert_array_equal(got, want)


def test_chunks_equal_whole_prompt():
    dtype, c = "f16", 150
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, [c], [c], 4, 4, 64, seed=11)
    whole = oracle.paged_prefill(dtype, q, kp, vp, tables, lens, qs, 0.125)
    start = 0
    for chunk in (48, 48, 33, 21):                      # cache holds start + chunk tokens
        part = oracle.paged_prefill(dtype, q[start:start + chunk], kp, vp, tables, [start + chunk],
                                    [0, chunk], 0.125)
        np.testing.assert_allclose(part, whole[start:start + chunk], rtol=1e-12, atol=1e-14)
        start += chunk
    assert start == c


def test_physical_placement_does_not_matter():
    dtype = "bf16"
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, [90, 33], [40, 33], 4, 2, 128, seed=5)
    a = oracle.paged_prefill(dtype, q, kp, vp, tables, lens, qs, 0.1)
    perm = np.random.default_rng(9).permutation(kp.shape[0])
    inv = np.argsort(perm)
    t2 = tables.copy()
    for s in range(len(lens)):
        nb = -(-int(lens[s]) // W.BLOCK)
        t2[s, :nb] = inv[tables[s, :nb]]
    b = oracle.paged_prefill(dtype, q, kp[perm], vp[perm], t2, lens, qs, 0.1)
    np.testing.assert_array_equal(a, b)


def test_causality_and_first_position():
    dtype, c, d = "f32", 40, 64
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, [c], [c], 2, 2, d, seed=8)
    base = oracle.paged_prefill(dtype, q, kp, vp, tables, lens, qs, 0.125)
    # position 0 sees only itself: its own V row, exactly
    np.testing.assert_array_equal(base[0, :, :], vd[0][0].astype(np.float64))
    # change the key and value of position 25: rows 0..24 unchanged, rows 25.. change
    kp2, vp2 = kp.copy(), vp.copy()
    blk, off = tables[0, 25 // 16], 25 % 16
    kp2[blk, :, off, :] += 3.0
    vp2[blk, :, off, :] -= 2.0
    pert = oracle.paged_prefill(dtype, q, kp2, vp2, tables, lens, qs, 0.125)
    np.testing.assert_array_equal(pert[:25], base[:25])
    assert np.all(np.abs(pert[25:] - base[25:]).max(axis=(1, 2)) > 1e-6)


def test_refuses_malformed_chunks():
    dtype = "f32"
    q, kd, vd, kp, vp, tables, lens, qs = prefill_case(dtype, [20], [10], 2, 2, 64, seed=1)
    with pytest.raises(ValueError):   # chunk longer than its context
        oracle.paged_prefill(dtype, np.concatenate([q, q, q]), kp, vp, tables, [20], [0, 30], 0.1)
    with pytest.raises(ValueError):   # query_start out of order
        oracle.paged_prefill(dtype, q, kp, vp, np.vstack([tables, tables]), [20, 20], [0, 8, 4], 0.1)
