"""Pins for the oracle: it is checked against things other than itself.

* values printed on the pages (tests/golden/pages_numbers.json, each cited);
* special cases that reduce to a library routine (scipy's softmax over a dense cache,
  numpy's float16 decoder);
* closed forms (one-token context, equal keys, one dominant logit, empty context);
* invariants the pages state (physical blocks are interchangeable; shared blocks and
  private copies give the same result).

A dropped term, a wrong sign, a wrong index or a transposed operand in the oracle fails at
least one of these.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------------------
# helpers (test-side, independent of the oracle's indexing code)

def decode_np(dtype, raw):
    """Library decoding to float64: numpy float16 / float32; bf16 via the top half of fp32."""
    if dtype == "f32":
        return raw.astype(np.float64)
    if dtype == "f16":
        return raw.astype(np.float64)
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scatter_dense(dense, tables, num_blocks, dtype):
    """Place each sequence's logical rows dense[s] [len_s, n_kv, d] into a paged pool."""
    n_kv, d = dense[0].shape[1], dense[0].shape[2]
    pool = np.zeros((num_blocks, n_kv, W.BLOCK, d), dtype=dense[0].dtype)
    pool[...] = W.nan_value(dtype)
    for s, rows in enumerate(dense):
        for j in range(rows.shape[0]):
            pool[tables[s, j // W.BLOCK], :, j % W.BLOCK, :] = rows[j]
    return pool


def dense_reference(q, kd, vd, scale, dtype):
    """scipy softmax attention on dense caches: out[s,h] = softmax(scale K q) V."""
    n_seqs, n_q, d = q.shape
    out = np.zeros((n_seqs, n_q, d))
    for s in range(n_seqs):
        n_kv = kd[s].shape[1]
        grp = n_q // n_kv
        for h in range(n_q):
            if kd[s].shape[0] == 0:
                continue
            K = decode_np(dtype, kd[s][:, h // grp, :])
            V = decode_np(dtype, vd[s][:, h // grp, :])
            z = scale * (K @ decode_np(dtype, q[s, h]))
            out[s, h] = softmax(z) @ V
    return out


def make_case(dtype, lens, n_q, n_kv, d, seed, slack=5, mb_extra=1):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nb_total = int(np.sum(-(-lens // W.BLOCK)))
    num_blocks = nb_total + slack
    max_blocks = max(1, int(np.max(-(-lens // W.BLOCK)))) + mb_extra
    tables = W.shuffled_tables(lens, num_blocks, seed, max_blocks=max_blocks)
    kd = [W.normal_values(rng, (int(n), n_kv, d), dtype) for n in lens]
    vd = [W.normal_values(rng, (int(n), n_kv, d), dtype) for n in lens]
    q = W.normal_values(rng, (len(lens), n_q, d), dtype)
    kp = scatter_dense(kd, tables, num_blocks, dtype)
    vp = scatter_dense(vd, tables, num_blocks, dtype)
    return q, kd, vd, kp, vp, tables, lens


# ---------------------------------------------------------------------------------------
# values printed on the pages

def test_kv_bytes_per_token_matches_pages(golden):
    g = golden["kv_bytes_per_token_gpt"]
    assert oracle.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["elem_bytes"]) == g["value"]
    # 16 attention layers, 4 KV heads x 256, bf16: 64 KiB per token, 1 MiB per 16-token block
    per_tok = oracle.kv_bytes_per_token(16, 4, 256, 2)
    assert per_tok == golden["longdoc_kv_bytes_per_token"]["value"]
    assert per_tok * golden["block_size_tokens"]["value"] == golden["longdoc_block_bytes"]["value"]
    assert per_tok * golden["native_context_tokens"]["value"] == golden["native_context_tokens"]["kv_bytes_per_sequence"]
    assert per_tok * golden["session_tokens"]["value"] == golden["session_tokens"]["kv_bytes_per_sequence"]
    # a transposed or dropped factor changes the number
    assert oracle.kv_bytes_per_token(32, 32, 128, 4) == 2 * g["value"]
    assert oracle.kv_bytes_per_token(1, 1, 1, 1) == 2


def _admit_sessions(mgr, kv_tokens, state_blocks):
    """Admit (KV sequence, fixed state) pairs until the pool refuses; returns the count."""
    n = 0
    while True:
        st, _ = mgr.add_seq(2 * n, kv_tokens, reserve_tokens=state_blocks * W.BLOCK)
        if st != "ok":
            return n, st
        if state_blocks:
            st2, _ = mgr.add_seq(2 * n + 1, state_blocks * W.BLOCK)
            assert st2 == "ok"
        n += 1


def test_capacity_example_matches_pages(golden):
    """23,859 one-MiB blocks hold 10 sessions of 32,768 tokens + 144 MiB state, not 11."""
    pool = golden["pool_mib"]["value"]
    state = golden["state_mib_per_sequence"]["value"]
    tokens = golden["session_tokens"]["value"]
    assert tokens // W.BLOCK + state == golden["session_mib_total"]["value"]
    n, st = _admit_sessions(oracle.BlockManagerOracle(pool), tokens, state)
    assert n == golden["paged_sessions"]["value"] and st == "no_blocks"
    # KV alone: floor(23859 / 2048) = 11
    n, _ = _admit_sessions(oracle.BlockManagerOracle(pool), tokens, 0)
    assert n == pool // (tokens // W.BLOCK) == 11
    # maximum reservation: 262,144 tokens (16 GiB) + state per session -> exactly one
    n, st = _admit_sessions(oracle.BlockManagerOracle(pool), golden["native_context_tokens"]["value"], state)
    assert n == golden["max_reservation_sessions"]["value"] and st == "no_blocks"


def test_dense_waste_example(golden):
    g = golden["dense_waste_fraction"]
    waste = 1 - g["mean_len"] / g["s_max"]
    assert waste == g["numerator"] / g["denominator"]
    assert round(g["cache_gb"] * waste) == g["wasted_gb"]
    # paged: the same 32 sequences of 512 tokens waste nothing (512 is a multiple of 16)
    mgr = oracle.BlockManagerOracle(32 * 512 // W.BLOCK)
    for s in range(g["batch"]):
        assert mgr.add_seq(s, g["mean_len"])[0] == "ok"
    assert mgr.tail_waste_rows() == 0 and mgr.stats()["free_blocks"] == 0


# ---------------------------------------------------------------------------------------
# element decoders against library conversions, exhaustively

def test_f16_decoder_exhaustive():
    raw = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    got = oracle.elems_to_double("f16", raw)
    want = raw.astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_decoder_exhaustive():
    raw = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.elems_to_double("bf16", raw)
    want = (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_f32_decoder_samples():
    x = np.random.default_rng(1).standard_normal(1000).astype(np.float32)
    x[:4] = [0.0, -0.0, np.inf, 1e-45]
    assert np.array_equal(oracle.elems_to_double("f32", x), x.astype(np.float64))


# ---------------------------------------------------------------------------------------
# attention: reduces to dense softmax attention (scipy) on the gathered rows

@pytest.mark.parametrize("dtype,n_q,n_kv,d", [
    ("f32", 2, 2, 64), ("f16", 4, 1, 64), ("bf16", 8, 2, 128), ("f16", 8, 8, 128),
    ("bf16", 16, 4, 256), ("f32", 8, 1, 256), ("f16", 2, 1, 128),
])
def test_paged_equals_dense_scipy(dtype, n_q, n_kv, d):
    lens = [1, 5, 16, 17, 33, 60]
    q, kd, vd, kp, vp, tables, lens = make_case(dtype, lens, n_q, n_kv, d, seed=7 + d + n_q)
    scale = 1.0 / np.sqrt(d)
    got = oracle.paged_decode(dtype, q, kp, vp, tables, lens, scale)
    want = dense_reference(q, kd, vd, scale, dtype)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_tiny_config_against_scipy():
    wl = W.tiny()
    q, kd, vd, kp, vp, tables, lens = make_case(wl.dtype, wl.context_lens, wl.n_q_heads, wl.n_kv_heads,
                                                wl.head_dim, seed=wl.seed,
                                                slack=wl.num_blocks - int(wl.blocks_per_seq().sum()))
    assert kp.shape[0] == wl.num_blocks
    got = oracle.paged_decode(wl.dtype, q, kp, vp, tables, lens, wl.scale)
    np.testing.assert_allclose(got, dense_reference(q, kd, vd, wl.scale, wl.dtype), rtol=0, atol=1e-12)


def test_peaky_softmax_stays_finite():
    """Logits near 1e3 overflow exp() unless the maximum is subtracted (scipy does)."""
    q, kd, vd, kp, vp, tables, lens = make_case("f32", [40, 3], 2, 1, 64, seed=3)
    q = (q * 400.0).astype(np.float32)
    got = oracle.paged_decode("f32", q, kp, vp, tables, lens, 0.125)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, dense_reference(q, kd, vd, 0.125, "f32"), rtol=0, atol=1e-10)


# ---------------------------------------------------------------------------------------
# closed forms

def test_single_token_context_returns_its_value_row():
    q, kd, vd, kp, vp, tables, lens = make_case("f16", [1, 1], 4, 2, 64, seed=11)
    got = oracle.paged_decode("f16", q, kp, vp, tables, lens, 0.3)
    for s in range(2):
        for h in range(4):
            assert np.array_equal(got[s, h], vd[s][0, h // 2].astype(np.float64))


def test_equal_keys_give_mean_of_values():
    q, kd, vd, kp, vp, tables, lens = make_case("f32", [37], 2, 2, 64, seed=12)
    kd = [np.repeat(kd[0][:1], 37, axis=0)]
    kp = scatter_dense(kd, tables, kp.shape[0], "f32")
    got = oracle.paged_decode("f32", q, kp, vp, tables, lens, 0.125)
    for h in range(2):
        np.testing.assert_allclose(got[0, h], vd[0][:, h].astype(np.float64).mean(axis=0), rtol=0, atol=1e-13)


def test_dominant_logit_selects_its_value_row():
    """Key j* = 40 q, every other key orthogonal-ish noise: out ~ V[j*]."""
    rng = np.random.default_rng(13)
    q, kd, vd, kp, vp, tables, lens = make_case("f32", [50], 1, 1, 64, seed=13)
    kd = [(0.01 * rng.standard_normal(kd[0].shape)).astype(np.float32)]
    jstar = 29
    kd[0][jstar, 0] = 40.0 * q[0, 0]
    kp = scatter_dense(kd, tables, kp.shape[0], "f32")
    got = oracle.paged_decode("f32", q, kp, vp, tables, lens, 1.0)
    np.testing.assert_allclose(got[0, 0], vd[0][jstar, 0].astype(np.float64), rtol=0, atol=1e-12)


def test_empty_context_outputs_zeros():
    q, kd, vd, kp, vp, tables, lens = make_case("bf16", [0, 5], 2, 1, 64, seed=14)
    got = oracle.paged_decode("bf16", q, kp, vp, tables, lens, 0.125)
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert np.all(np.isfinite(got[1]))


# ---------------------------------------------------------------------------------------
# invariants the pages state

def test_physical_permutation_invariance():
    """'los bloques libres son intercambiables': moving blocks and remapping tables changes nothing."""
    q, kd, vd, kp, vp, tables, lens = make_case("f16", [70, 33, 129], 4, 2, 128, seed=15)
    base = oracle.paged_decode("f16", q, kp, vp, tables, lens, 0.1)
    nb = kp.shape[0]
    perm = np.random.default_rng(16).permutation(nb)          # new position of old block b is perm[b]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    got = oracle.paged_decode("f16", q, kp2, vp2, t2, lens, 0.1)
    assert np.array_equal(got, base)


def test_shared_prefix_equals_private_copy():
    """Two sequences pointing at the same prefix blocks == the same rows copied privately."""
    rng = np.random.default_rng(17)
    d, n_kv, n_q = 64, 2, 2
    prefix, t0, t1 = 40, 9, 23                    # 40 = 2 full blocks + 8 rows
    kpre = W.normal_values(rng, (prefix, n_kv, d), "f16")
    vpre = W.normal_values(rng, (prefix, n_kv, d), "f16")
    k0 = np.concatenate([kpre, W.normal_values(rng, (t0, n_kv, d), "f16")])
    v0 = np.concatenate([vpre, W.normal_values(rng, (t0, n_kv, d), "f16")])
    k1 = np.concatenate([kpre, W.normal_values(rng, (t1, n_kv, d), "f16")])
    v1 = np.concatenate([vpre, W.normal_values(rng, (t1, n_kv, d), "f16")])
    q = W.normal_values(rng, (2, n_q, d), "f16")
    lens = np.array([prefix + t0, prefix + t1], dtype=np.int32)
    # private: every block distinct
    priv = W.shuffled_tables(lens, 20, seed=18, max_blocks=5)
    kp = scatter_dense([k0, k1], priv, 20, "f16")
    vp = scatter_dense([v0, v1], priv, 20, "f16")
    out_priv = oracle.paged_decode("f16", q, kp, vp, priv, lens, 0.125)
    # shared: sequence 1 reuses sequence 0's two full prefix blocks
    shared = priv.copy()
    shared[1, :2] = priv[0, :2]
    kp_s = scatter_dense([k0, k1], shared, 20, "f16")
    vp_s = scatter_dense([v0, v1], shared, 20, "f16")
    out_shared = oracle.paged_decode("f16", q, kp_s, vp_s, shared, lens, 0.125)
    assert np.array_equal(out_priv, out_shared)


# ---------------------------------------------------------------------------------------
# append and copy oracles against numpy fancy indexing

def test_kv_append_matches_fancy_indexing():
    rng = np.random.default_rng(19)
    nb, n_kv, d = 12, 3, 64
    kp = np.zeros((nb, n_kv, 16, d), np.float16)
    vp = np.zeros_like(kp)
    n_tok = 30
    slots = rng.choice(nb * 16, size=n_tok, replace=False).astype(np.int64)
    slots[[3, 17]] = -1
    k = W.normal_values(rng, (n_tok, n_kv, d), "f16")
    v = W.normal_values(rng, (n_tok, n_kv, d), "f16")
    oracle.kv_append(k, v, slots, kp, vp)
    want_k = np.zeros_like(kp)
    want_v = np.zeros_like(vp)
    keep = slots >= 0
    want_k[slots[keep] // 16, :, slots[keep] % 16, :] = k[keep]
    want_v[slots[keep] // 16, :, slots[keep] % 16, :] = v[keep]
    assert np.array_equal(kp.view(np.uint16), want_k.view(np.uint16))
    assert np.array_equal(vp.view(np.uint16), want_v.view(np.uint16))
    with pytest.raises(ValueError):
        oracle.kv_append(k[:1], v[:1], np.array([nb * 16]), kp, vp)


def test_copy_blocks_matches_fancy_indexing():
    rng = np.random.default_rng(20)
    L, nb, n_kv, d = 3, 10, 2, 64
    kp = W.normal_values(rng, (L, nb, n_kv, 16, d), "bf16")
    vp = W.normal_values(rng, (L, nb, n_kv, 16, d), "bf16")
    pairs = np.array([[1, 7], [4, 2], [9, 0]], dtype=np.int32)
    want_k, want_v = kp.copy(), vp.copy()
    want_k[:, pairs[:, 1]] = kp[:, pairs[:, 0]]
    want_v[:, pairs[:, 1]] = vp[:, pairs[:, 0]]
    oracle.copy_blocks(kp, vp, pairs)
    assert np.array_equal(kp, want_k) and np.array_equal(vp, want_v)


def test_oracle_refuses_malformed_tables():
    q, kd, vd, kp, vp, tables, lens = make_case("f32", [20], 2, 2, 64, seed=21)
    bad = tables.copy()
    bad[0, 1] = kp.shape[0]
    with pytest.raises(ValueError):
        oracle.paged_decode("f32", q, kp, vp, bad, lens, 0.1)
    with pytest.raises(ValueError):
        oracle.paged_decode("f32", q, kp, vp, tables, np.array([tables.shape[1] * 16 + 1]), 0.1)
