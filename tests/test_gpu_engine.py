"""Whole decode steps with prefix sharing and churn, GPU engine against the oracle.

GPU side: the C block manager plans every step, copy-on-write pairs go through copy_blocks,
the new rows through kv_append, and attention through the decode kernel (engine.DecodeBatch).
Oracle side, independently: the Python block-manager oracle replays the same operations; its
slots, pairs and tables must equal the C manager's bit for bit; its own host pools receive the
same generated rows through the oracle's copy and append; the fp64 oracle attention is then
compared element by element with the GPU outputs of every layer at every step.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import NP_STORAGE, TOL, as_f64, to_torch
from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W
from paged_kv_cache_258_gb300.engine import DecodeBatch, PagedKVCache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("f16", 4, 4, 64), ("bf16", 8, 2, 128), ("f32", 4, 1, 64)])
def test_prefix_churn_steps_match_oracle(dtype, n_q, n_kv, d, fused):
    rng = np.random.default_rng(77)
    L, n_groups, n_members, n_steps = 2, 3, 12, 24
    prompts = [int(100 + rng.integers(1, 16)) for _ in range(n_groups)]   # partial shared tails
    nb = 160
    order = W.free_order(nb, 5)
    desc = pkv.make_desc(dtype, L, nb, n_q, n_kv, d)
    cache = PagedKVCache(desc, free_order=order)
    mo = BlockManagerOracle(nb, free_order=order)
    hk = np.zeros((L, nb, n_kv, 16, d), NP_STORAGE[dtype])
    hv = np.zeros_like(hk)
    roots = [1000 + g for g in range(n_groups)]
    for g, r in enumerate(roots):
        slots = cache.add_sequence(r, prompts[g])
        st, slots_o = mo.add_seq(r, prompts[g])
        assert st == "ok" and slots.tolist() == slots_o
        for layer in range(L):
            k = W.normal_values(rng, (prompts[g], n_kv, d), dtype)
            v = W.normal_values(rng, (prompts[g], n_kv, d), dtype)
            pkv.pkv_kv_append(desc, layer, to_torch(k, dtype), to_torch(v, dtype), torch.from_numpy(slots).cuda(),
                              cache.k_pool, cache.v_pool)
            oracle.kv_append(k, v, slots_o, hk[layer], hv[layer])
    live = []
    for m in range(n_members):
        cache.fork(roots[m % n_groups], m)
        assert mo.fork(roots[m % n_groups], m) == "ok"
        live.append(m)
    batch = DecodeBatch(cache, live, max_blocks=(max(prompts) + n_steps + 32) // 16 + 1, fused=fused)
    next_id = n_members
    scale = 1.0 / np.sqrt(d)
    cow_seen = 0
    for step in range(n_steps):
        q = W.normal_values(rng, (L, n_members, n_q, d), dtype)
        kn = W.normal_values(rng, (L, n_members, n_kv, d), dtype)
        vn = W.normal_values(rng, (L, n_members, n_kv, d), dtype)
        out = torch.full((L, n_members, n_q, d), float("nan"), dtype=pkv.torch_dtype(dtype), device="cuda")
        st = batch.step(to_torch(q, dtype), to_torch(kn, dtype), to_torch(vn, dtype), out, scale)
        # oracle replay of the same step
        slots_o, pairs_o = [], []
        for sid in live:
            s_, slot, src, dst = mo.append_slot(sid)
            assert s_ == "ok"
            slots_o.append(slot)
            if src >= 0:
                pairs_o.append((src, dst))
        assert st["slots"].numpy().tolist() == slots_o
        assert st["pairs"].numpy()[: st["npairs"]].tolist() == [list(p) for p in pairs_o]
        cow_seen += len(pairs_o)
        if pairs_o:
            oracle.copy_blocks(hk, hv, np.array(pairs_o, dtype=np.int32))
        tables = st["tables"].numpy()
        lens = st["lens"].numpy()
        for i, sid in enumerate(live):
            t_o, ctx_o = mo.block_table(sid)
            assert tables[i, : len(t_o)].tolist() == t_o and lens[i] == ctx_o
        got = as_f64(out)
        for layer in range(L):
            oracle.kv_append(kn[layer], vn[layer], np.array(slots_o), hk[layer], hv[layer])
            want = oracle.paged_decode(dtype, q[layer], hk[layer], hv[layer], tables, lens, scale)
            err = np.max(np.abs(got[layer] - want))
            assert err <= TOL[dtype], f"step {step} layer {layer}: {err:.3e}"
        # churn: two members finish, two forks of random roots replace them
        for _ in range(2):
            j = int(rng.integers(0, n_members))
            g = int(rng.integers(0, n_groups))
            cache.free(live[j])
            assert mo.free_seq(live[j]) == "ok"
            cache.fork(roots[g], next_id)
            assert mo.fork(roots[g], next_id) == "ok"
            live[j] = next_id
            next_id += 1
        batch.set_sequences(live)
    assert cow_seen >= n_members                      # every member copied its shared tail once
    assert pkv.pkv_get_device_status() == 0
    assert cache.mgr.stats() == mo.stats()
