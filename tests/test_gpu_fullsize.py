"""Full-size parity, in the launch configuration bench.py times, on sampled outputs.

For the gpt, ragged and longdoc workloads this builds exactly what bench.py builds (same
pools, same batch, same table width and therefore the same grid and split-K partitions),
runs warm-up steps plus one step, and checks sampled (layer, sequence) outputs against the
oracle. The oracle's inputs are independent of the CUDA path: host copies of the sampled
layers' pools taken before any step (they come from the seeded device generator), the Python
block-manager oracle's own replay of the run, and its own byte appends of the generated rows.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import TOL, as_f64, to_host
from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W

pytestmark = pytest.mark.gpu

WARMUP, STEPS = 10, 100          # bench.py's defaults: they fix the table width and grid


@pytest.mark.parametrize("config,layers,seqs", [
    ("gpt", (0, 31), (0, 17, 40, 63)),
    ("ragged", (0,), tuple(range(32))),
    ("longdoc", (0, 15), (0, 9)),
])
def test_fullsize_sampled(config, layers, seqs):
    device = torch.device("cuda", 0)
    wl, _, cache, batch, (q, kn, vn, out), state = bench.setup_gpu_case(config, WARMUP, STEPS, device)
    dtype = wl.dtype
    host_k = {l: to_host(cache.k_pool[l], dtype) for l in layers}
    host_v = {l: to_host(cache.v_pool[l], dtype) for l in layers}
    # oracle replay of the admissions
    mo = BlockManagerOracle(wl.num_blocks, free_order=W.free_order(wl.num_blocks, wl.seed))
    for s, n in enumerate(wl.context_lens):
        assert mo.add_seq(s, int(n) - 1)[0] == "ok"
    # row r of q, the tables and out is sequence ids[r] (bench.py orders the ragged batch longest
    # first), and the appends go in row order
    ids = [int(x) for x in batch.seq_ids]
    assert sorted(ids) == list(range(wl.n_seqs))
    if config in bench.ORDER_LONGEST_FIRST:
        assert all(wl.context_lens[a] >= wl.context_lens[b] for a, b in zip(ids, ids[1:]))
    n_steps = 4
    for _ in range(n_steps):
        st = batch.step(q, kn, vn, out, wl.scale)
        slots = [mo.append_slot(s)[1] for s in ids]
        assert st["slots"].numpy().tolist() == slots
        for l in layers:
            oracle.kv_append(to_host(kn[l], dtype), to_host(vn[l], dtype), np.array(slots), host_k[l], host_v[l])
    assert pkv.pkv_get_device_status() == 0
    tables = np.full((wl.n_seqs, batch.max_blocks), -1, dtype=np.int32)
    lens = np.zeros(wl.n_seqs, dtype=np.int32)
    for r, s in enumerate(ids):
        t, lens[r] = mo.block_table(s)
        tables[r, : len(t)] = t
    assert np.array_equal(tables, st["tables"].numpy()) and np.array_equal(lens, st["lens"].numpy())
    got = as_f64(out)
    sel = np.array(seqs)
    for l in layers:
        ql = to_host(q[l], dtype)[sel]
        want = oracle.paged_decode(dtype, ql, host_k[l], host_v[l], tables[sel], lens[sel], wl.scale,
                                   n_threads=oracle.max_threads())
        err = np.max(np.abs(got[l][sel] - want))
        assert err <= TOL[dtype], f"{config} layer {l}: max abs error {err:.3e}"
    # every output row of the step is finite
    assert torch.isfinite(out.float()).all()


def test_prefill30k_fullsize_sampled():
    """The 30,000-token prompt of the prefill30k line, chunked exactly as bench.py runs it (2 of its
    16 layers: every launch is identical per layer), sampled query positions of every chunk checked
    against the oracle one query at a time. The oracle's pools are its own byte appends of the
    generated rows at the slots of its own block-manager replay (add_seq for the first chunk,
    extend for the others)."""
    device = torch.device("cuda", 0)
    P, cache, ps, (q, kn, vn, out), chunks = bench.setup_prefill_case(device, layers=2)
    dtype, L, d = P["dtype"], P["n_layers"], P["d"]
    scale = 1.0 / np.sqrt(d)
    mo = BlockManagerOracle(cache.desc.num_blocks, free_order=P["free_order"])
    nb = cache.desc.num_blocks
    host_k = np.zeros((L, nb, P["n_kv"], 16, d), np.uint16)
    host_v = np.zeros_like(host_k)
    kn_h, vn_h, q_h = to_host(kn, dtype), to_host(vn, dtype), to_host(q, dtype)
    for i, (c0, n) in enumerate(chunks):
        st = ps.step([(1, n, i == 0)], q[:, c0:c0 + n], kn[:, c0:c0 + n], vn[:, c0:c0 + n], out[:, c0:c0 + n],
                     scale)
        s_, slots = mo.add_seq(1, n) if i == 0 else mo.extend(1, n)[:2]
        assert s_ == "ok"
        assert st["np"][: 2 * ps.max_tokens].view(np.int64)[:n].tolist() == list(slots)
        for layer in range(L):
            oracle.kv_append(kn_h[layer, c0:c0 + n], vn_h[layer, c0:c0 + n], np.array(slots), host_k[layer],
                             host_v[layer])
    assert pkv.pkv_get_device_status() == 0
    t, ctx = mo.block_table(1)
    assert ctx == P["prompt"]
    # sampled positions: first, middle and last token of every chunk, plus the prompt's last token
    pos = sorted({p for c0, n in chunks for p in (c0, c0 + n // 2, c0 + n - 1)})
    tables = np.tile(np.array(t, dtype=np.int32), (len(pos), 1))
    lens = np.array(pos, dtype=np.int32) + 1          # each sample: one query at its own position
    qs = np.arange(len(pos) + 1, dtype=np.int32)
    got = as_f64(out)
    for layer in range(L):
        want = oracle.paged_prefill(dtype, q_h[layer, pos], host_k[layer], host_v[layer], tables, lens, qs, scale,
                                    n_threads=oracle.max_threads())
        err = np.max(np.abs(got[layer, pos] - want))
        assert err <= TOL[dtype], f"layer {layer}: {err:.3e}"


def test_prefix_fullsize_sampled():
    """The prefix-sharing workload at full size (200 members forked from 8 roots, 5 % churn per
    step, copy-on-write of each member's shared tail on its first write), in bench.py's launch
    configuration. The Python manager oracle replays the same churn and appends; its copy-on-write
    pairs and byte appends go into host copies of the pool; sampled members are checked."""
    device = torch.device("cuda", 0)
    wl, _, cache, batch, (q, kn, vn, out), state = bench.setup_gpu_case("prefix", WARMUP, STEPS, device)
    dtype, churn, roots = wl.dtype, state["churn"], state["roots"]
    host_k = np.ascontiguousarray(to_host(cache.k_pool[0], dtype)[None])  # [1, blocks, kv, 16, d]
    host_v = np.ascontiguousarray(to_host(cache.v_pool[0], dtype)[None])
    mo = BlockManagerOracle(wl.num_blocks, free_order=W.free_order(wl.num_blocks, wl.seed))
    for g in range(churn.n_groups):
        assert mo.add_seq(roots[g], churn.group_prompt[g])[0] == "ok"
    for m, g in enumerate(churn.member_group):
        assert mo.fork(roots[g], m) == "ok"
    live = list(range(len(churn.member_group)))
    n_cow = 0
    for step in range(3):
        if step < len(churn.steps):  # the same churn, in the same order, as bench.apply_churn
            for old, new, g in churn.steps[step]:
                assert mo.free_seq(old) == "ok" and mo.fork(roots[g], new) == "ok"
                live[live.index(old)] = new
        bench.apply_churn(cache, batch, state)
        st = batch.step(q, kn, vn, out, wl.scale)
        slots, pairs = [], []
        for sid in live:  # append_batch = successive appends in batch order
            status, slot, src, dst = mo.append_slot(sid)
            assert status == "ok"
            slots.append(slot)
            if src >= 0:
                pairs.append((src, dst))
        assert st["slots"].numpy().tolist() == slots
        n_cow += len(pairs)
        if pairs:  # copies first, then the new rows (the step's order)
            oracle.copy_blocks(host_k, host_v, np.array(pairs, dtype=np.int32))
        oracle.kv_append(to_host(kn[0], dtype), to_host(vn[0], dtype), np.array(slots), host_k[0], host_v[0])
    assert n_cow > 0
    assert pkv.pkv_get_device_status() == 0
    tables = np.full((len(live), batch.max_blocks), -1, dtype=np.int32)
    lens = np.zeros(len(live), dtype=np.int32)
    for i, sid in enumerate(live):
        t, lens[i] = mo.block_table(sid)
        tables[i, : len(t)] = t
    assert np.array_equal(tables, st["tables"].numpy()) and np.array_equal(lens, st["lens"].numpy())
    sel = np.array([0, 37, 101, 150, 199])
    want = oracle.paged_decode(dtype, to_host(q[0], dtype)[sel], host_k[0], host_v[0], tables[sel], lens[sel],
                               wl.scale, n_threads=oracle.max_threads())
    err = np.max(np.abs(as_f64(out)[0][sel] - want))
    assert err <= TOL[dtype], f"prefix: max abs error {err:.3e}"
    assert torch.isfinite(out.float()).all()
