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
def test_prefix_churn_steps_match_oracle(dtype, n_q, n_kv, d, fused, monkeypatch):
    # every planned step also passes the host-side metadata check (no false alarms on real steps)
    from paged_kv_cache_258_gb300 import engine
    monkeypatch.setattr(engine, "CHECK_METADATA", True)
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


@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("bf16", 8, 2, 128), ("f16", 4, 4, 64), ("f32", 4, 2, 64)])
def test_chunked_prefill_steps_match_oracle(dtype, n_q, n_kv, d):
    """Chunked prefill through the engine: admissions, extends and copy-on-write of a shared tail,
    C manager vs oracle manager bit for bit, attention vs the oracle on its own host pools."""
    from paged_kv_cache_258_gb300.engine import PrefillStep
    rng = np.random.default_rng(91)
    L, nb = 2, 220
    order = W.free_order(nb, 8)
    desc = pkv.make_desc(dtype, L, nb, n_q, n_kv, d)
    cache = PagedKVCache(desc, free_order=order)
    mo = BlockManagerOracle(nb, free_order=order)
    hk = np.zeros((L, nb, n_kv, 16, d), NP_STORAGE[dtype])
    hv = np.zeros_like(hk)
    ps = PrefillStep(cache, max_tokens=300, max_seqs=4, max_blocks=40)
    scale = 1.0 / np.sqrt(d)
    plan = [
        [(100, 37, True), (1, 128, True), (2, 70, True)],
        "fork",
        [(1, 128, False), (10, 50, False), (11, 20, False)],
        [(1, 44, False), (10, 30, False), (2, 1, False), (3, 200, True)],
    ]
    cow_seen = 0
    for chunks in plan:
        if chunks == "fork":
            for child in (10, 11):
                cache.fork(100, child)
                assert mo.fork(100, child) == "ok"
            continue
        T = sum(c[1] for c in chunks)
        q = W.normal_values(rng, (L, T, n_q, d), dtype)
        kn = W.normal_values(rng, (L, T, n_kv, d), dtype)
        vn = W.normal_values(rng, (L, T, n_kv, d), dtype)
        out = torch.full((L, T, n_q, d), float("nan"), dtype=pkv.torch_dtype(dtype), device="cuda")
        st = ps.step(chunks, to_torch(q, dtype), to_torch(kn, dtype), to_torch(vn, dtype), out, scale)
        got_slots = st["np"][: 2 * ps.max_tokens].view(np.int64)[:T].tolist()
        slots_o, pairs_o = [], []
        for sid, n, first in chunks:
            if first:
                s_, sl = mo.add_seq(sid, n)
            else:
                s_, sl, src, dst = mo.extend(sid, n)
                if src >= 0:
                    pairs_o.append((src, dst))
            assert s_ == "ok"
            slots_o += list(sl)
        assert got_slots == slots_o
        assert st["npairs"] == len(pairs_o)
        cow_seen += len(pairs_o)
        if pairs_o:
            oracle.copy_blocks(hk, hv, np.array(pairs_o, dtype=np.int32))
        ids = [c[0] for c in chunks]
        tables = np.full((len(ids), ps.max_blocks), -1, dtype=np.int32)
        lens = np.zeros(len(ids), dtype=np.int32)
        for i, sid in enumerate(ids):
            t_o, ctx_o = mo.block_table(sid)
            tables[i, : len(t_o)] = t_o
            lens[i] = ctx_o
        assert np.array_equal(st["lens"], lens)
        qs = np.concatenate([[0], np.cumsum([c[1] for c in chunks])]).astype(np.int32)
        got = as_f64(out)
        for layer in range(L):
            oracle.kv_append(kn[layer], vn[layer], np.array(slots_o), hk[layer], hv[layer])
            want = oracle.paged_prefill(dtype, q[layer], hk[layer], hv[layer], tables, lens, qs, scale)
            err = np.max(np.abs(got[layer] - want))
            assert err <= TOL[dtype], f"layer {layer}: {err:.3e}"
    assert cow_seen == 2                       # both forks copied the root's partial tail once
    assert pkv.pkv_get_device_status() == 0
    assert cache.mgr.stats() == mo.stats()


@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("f16", 8, 8, 128), ("bf16", 16, 4, 256)])
def test_layer_overlap_is_bit_identical(dtype, n_q, n_kv, d):
    """Decode steps whose layer launches overlap (PKV_DECODE_OVERLAP_PREVIOUS: each layer's kernel
    may start while the previous layer's finishes, all layers sharing one split-K workspace) give
    outputs and pools bit-identical to the same steps launched one after the other."""
    L, nb = 4, 600
    lens = [2500, 1, 700, 1800, 33, 1100]  # split-K and single-partition sequences
    order = W.free_order(nb, 8)
    results = []
    for overlap in (True, False):
        desc = pkv.make_desc(dtype, L, nb, n_q, n_kv, d)
        cache = PagedKVCache(desc, free_order=order, init="randn", seed=21)
        for s, n in enumerate(lens):
            cache.add_sequence(s, n - 1)
        batch = DecodeBatch(cache, list(range(len(lens))), max_blocks=200)
        batch.overlap = overlap
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        dt = pkv.torch_dtype(dtype)
        q = torch.randn((L, len(lens), n_q, d), device="cuda", generator=g).to(dt)
        kn = torch.randn((L, len(lens), n_kv, d), device="cuda", generator=g).to(dt)
        vn = torch.randn((L, len(lens), n_kv, d), device="cuda", generator=g).to(dt)
        outs = []
        for _ in range(3):
            out = torch.empty_like(q)
            batch.step(q, kn, vn, out, 1.0 / np.sqrt(d))
            outs.append(out)
        torch.cuda.synchronize()
        assert pkv.pkv_get_device_status() == 0
        results.append((torch.stack(outs), cache.k_pool.clone(), cache.v_pool.clone()))
    for a, b in zip(results[0], results[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("dtype,n_q,n_kv,d", [("bf16", 16, 4, 256), ("f16", 8, 8, 128)])
def test_prefill_layer_overlap_is_bit_identical(dtype, n_q, n_kv, d):
    """Chunked-prefill steps whose attention launches overlap (all layers' appends first, then
    PKV_PREFILL_OVERLAP_PREVIOUS launches) give outputs and pools bit-identical to the per-layer
    append-then-attend order."""
    from paged_kv_cache_258_gb300.engine import PrefillStep
    L, nb, T = 3, 400, 1024
    prompts = {0: 2100, 1: 700}
    order = W.free_order(nb, 4)
    results = []
    for overlap in (True, False):
        desc = pkv.make_desc(dtype, L, nb, n_q, n_kv, d)
        cache = PagedKVCache(desc, free_order=order, init="randn", seed=31)
        ps = PrefillStep(cache, max_tokens=T, max_seqs=2, max_blocks=160)
        ps.overlap = overlap
        g = torch.Generator(device="cuda")
        g.manual_seed(9)
        dt = pkv.torch_dtype(dtype)
        done = {s: 0 for s in prompts}
        outs = []
        while any(done[s] < prompts[s] for s in prompts):
            chunks, budget = [], T
            for s, n in prompts.items():
                take = min(n - done[s], budget // 2 if len(prompts) > 1 else budget)
                if take > 0:
                    chunks.append((s, take, done[s] == 0))
                    budget -= take
            n_tok = sum(c[1] for c in chunks)
            q = torch.randn((L, n_tok, n_q, d), device="cuda", generator=g).to(dt)
            kn = torch.randn((L, n_tok, n_kv, d), device="cuda", generator=g).to(dt)
            vn = torch.randn((L, n_tok, n_kv, d), device="cuda", generator=g).to(dt)
            out = torch.empty_like(q)
            ps.step(chunks, q, kn, vn, out, 1.0 / np.sqrt(d))
            outs.append(out)
            for s, n, _ in chunks:
                done[s] += n
        torch.cuda.synchronize()
        assert pkv.pkv_get_device_status() == 0
        results.append((outs, cache.k_pool.clone(), cache.v_pool.clone()))
    for a, b in zip(results[0][0], results[1][0]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(results[0][1].view(torch.int16), results[1][1].view(torch.int16))
    assert torch.equal(results[0][2].view(torch.int16), results[1][2].view(torch.int16))


def test_step_copy_pipeline_matches_direct_steps():
    """Decode steps fed through engine.StepCopyPipeline (inputs from pinned host memory into two
    alternating device sets, outputs copied back while the next step runs) return on the host
    exactly what the same steps return on the device when fed directly."""
    from paged_kv_cache_258_gb300.engine import StepCopyPipeline
    dtype, n_q, n_kv, d, L, nb = "f16", 8, 4, 128, 3, 300
    lens = [900, 40, 1500, 300]
    dt = pkv.torch_dtype(dtype)
    g = torch.Generator()
    g.manual_seed(3)
    n_steps = 4
    hq = [torch.randn((L, len(lens), n_q, d), generator=g).to(dt).pin_memory() for _ in range(n_steps)]
    hk = [torch.randn((L, len(lens), n_kv, d), generator=g).to(dt).pin_memory() for _ in range(n_steps)]
    hv = [torch.randn((L, len(lens), n_kv, d), generator=g).to(dt).pin_memory() for _ in range(n_steps)]
    caches = []
    for _ in range(2):
        cache = PagedKVCache(pkv.make_desc(dtype, L, nb, n_q, n_kv, d), free_order=W.free_order(nb, 6),
                             init="randn", seed=12)
        for s, n in enumerate(lens):
            cache.add_sequence(s, n - 1)
        caches.append((cache, DecodeBatch(cache, list(range(len(lens))), max_blocks=120)))
    # direct
    cache, batch = caches[0]
    want = []
    for i in range(n_steps):
        out = torch.empty(hq[i].shape, dtype=dt, device="cuda")
        batch.step(hq[i].cuda(), hk[i].cuda(), hv[i].cuda(), out, 0.09)
        want.append(out.cpu())
    # pipelined
    cache, batch = caches[1]
    stream = batch.stream
    pipe = StepCopyPipeline(stream, cache.device, lambda: {"q": torch.empty_like(hq[0], device="cuda"),
                                                           "k": torch.empty_like(hk[0], device="cuda"),
                                                           "v": torch.empty_like(hv[0], device="cuda"),
                                                           "out": torch.empty_like(hq[0], device="cuda")})
    got = [torch.empty_like(hq[0]).pin_memory() for _ in range(n_steps)]
    with torch.cuda.stream(stream):
        pipe.upload({"q": hq[0], "k": hk[0], "v": hv[0]})
        for i in range(n_steps):
            dev = pipe.begin()
            batch.step(dev["q"], dev["k"], dev["v"], dev["out"], 0.09)
            pipe.end({"out": got[i]})
            if i + 1 < n_steps:
                pipe.upload({"q": hq[i + 1], "k": hk[i + 1], "v": hv[i + 1]})
        pipe.finish()
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_status() == 0
    for a, b in zip(want, got):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(caches[0][0].k_pool.view(torch.int16), caches[1][0].k_pool.view(torch.int16))
