"""KV append scatter and copy-on-write block copy on the GPU: bit-exact against the oracle.

The expected pools come from the oracle's own byte copies applied to host copies of the
same generated inputs; the comparison is over every byte of both pools (all rows: the
kernels must not touch rows they were not asked to write).
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import to_host, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,n_kv,d", [("f32", 2, 64), ("f16", 4, 128), ("bf16", 4, 256), ("f16", 1, 256),
                                          ("f32", 8, 256), ("bf16", 3, 64)])
def test_append_bitexact(dtype, n_kv, d):
    rng = np.random.default_rng(d + n_kv)
    L, nb = 2, 40
    kp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    vp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    n_tok = 300
    slots = rng.choice(nb * 16, size=n_tok, replace=False).astype(np.int64)
    slots[rng.choice(n_tok, size=20, replace=False)] = -1          # padding tokens
    k = W.normal_values(rng, (n_tok, n_kv, d), dtype)
    v = W.normal_values(rng, (n_tok, n_kv, d), dtype)
    desc = pkv.make_desc(dtype, L, nb, n_kv, n_kv, d)
    kt, vt = to_torch(kp, dtype), to_torch(vp, dtype)
    pkv.pkv_kv_append(desc, 1, to_torch(k, dtype), to_torch(v, dtype), torch.from_numpy(slots).cuda(), kt, vt)
    assert pkv.pkv_get_device_status() == 0
    want_k, want_v = kp.copy(), vp.copy()
    oracle.kv_append(k, v, slots, want_k[1], want_v[1])
    assert np.array_equal(to_host(kt, dtype).view(np.uint8), want_k.view(np.uint8))
    assert np.array_equal(to_host(vt, dtype).view(np.uint8), want_v.view(np.uint8))


def test_append_prefill_size_and_bad_slot():
    dtype, n_kv, d, nb = "bf16", 4, 256, 2100
    rng = np.random.default_rng(1)
    n_tok = 32768                                                   # one long-document prompt
    slots = (W.free_order(nb, 1)[: n_tok // 16].astype(np.int64)[:, None] * 16 + np.arange(16)).reshape(-1)
    k = W.normal_values(rng, (n_tok, n_kv, d), dtype)
    v = W.normal_values(rng, (n_tok, n_kv, d), dtype)
    desc = pkv.make_desc(dtype, 1, nb, 16, n_kv, d)
    kt = torch.zeros(pkv.pool_shape(desc), dtype=torch.bfloat16, device="cuda")
    vt = torch.zeros_like(kt)
    slots_bad = slots.copy()
    slots_bad[5] = nb * 16 + 3                                      # past the pool: skipped, flagged
    pkv.pkv_kv_append(desc, 0, to_torch(k, dtype), to_torch(v, dtype), torch.from_numpy(slots_bad).cuda(), kt, vt)
    assert pkv.pkv_get_device_status() == pkv.PKV_DEV_BAD_SLOT
    want_k = np.zeros((nb, n_kv, 16, d), np.uint16)
    want_v = np.zeros_like(want_k)
    slots_ok = slots.copy()
    slots_ok[5] = -1
    oracle.kv_append(k, v, slots_ok, want_k, want_v)
    assert np.array_equal(to_host(kt, dtype)[0], want_k)
    assert np.array_equal(to_host(vt, dtype)[0], want_v)


@pytest.mark.parametrize("dtype,L,n_kv,d", [("f16", 32, 4, 128), ("bf16", 3, 4, 256), ("f32", 1, 2, 64)])
def test_copy_blocks_bitexact(dtype, L, n_kv, d):
    rng = np.random.default_rng(L + d)
    nb = 64
    kp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    vp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    ids = rng.permutation(nb)
    pairs = np.stack([ids[:20], ids[20:40]], axis=1).astype(np.int32)   # disjoint src / dst sets
    desc = pkv.make_desc(dtype, L, nb, n_kv, n_kv, d)
    kt, vt = to_torch(kp, dtype), to_torch(vp, dtype)
    pkv.pkv_copy_blocks(desc, kt, vt, torch.from_numpy(pairs).cuda())
    assert pkv.pkv_get_device_status() == 0
    want_k, want_v = kp.copy(), vp.copy()
    oracle.copy_blocks(want_k, want_v, pairs)
    assert np.array_equal(to_host(kt, dtype).view(np.uint8), want_k.view(np.uint8))
    assert np.array_equal(to_host(vt, dtype).view(np.uint8), want_v.view(np.uint8))


def test_copy_blocks_bad_pair_is_skipped():
    dtype, L, n_kv, d, nb = "f16", 2, 2, 64, 8
    rng = np.random.default_rng(3)
    kp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    vp = W.normal_values(rng, (L, nb, n_kv, 16, d), dtype)
    pairs = np.array([[1, 2], [3, nb], [-1, 4]], dtype=np.int32)
    desc = pkv.make_desc(dtype, L, nb, n_kv, n_kv, d)
    kt, vt = to_torch(kp, dtype), to_torch(vp, dtype)
    pkv.pkv_copy_blocks(desc, kt, vt, torch.from_numpy(pairs).cuda())
    assert pkv.pkv_get_device_status() == pkv.PKV_DEV_BAD_PAIR
    want_k, want_v = kp.copy(), vp.copy()
    oracle.copy_blocks(want_k, want_v, pairs[:1])
    assert np.array_equal(to_host(kt, dtype), want_k) and np.array_equal(to_host(vt, dtype), want_v)
