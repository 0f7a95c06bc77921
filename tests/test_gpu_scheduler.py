"""Continuous batching end to end on the GPU, every iteration against the oracle.

The scheduler plans each iteration on the C block manager (mirrored into the oracle manager and
compared call by call); the executor runs copy-on-write copies, chunk appends + paged prefill
attention and fused append + paged decode attention. The oracle keeps its own host pools,
applying the same copies and appends, and computes every decode and prefill output of every
layer of every iteration from its own block tables.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import NP_STORAGE, TOL, as_f64, to_torch
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W
from paged_kv_cache_258_gb300.engine import PagedKVCache, StepExecutor
from paged_kv_cache_258_gb300.scheduler import Request, Scheduler, serve
from test_scheduler import MirroredManager, VirtualClock

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("overlap", [True, False])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_continuous_batching_matches_oracle(dtype, overlap):
    L, n_q, n_kv, d, nb = 2, 4, 2, 64, 90
    rng = np.random.default_rng(123)
    order = W.free_order(nb, 77)
    desc = pkv.make_desc(dtype, L, nb, n_q, n_kv, d)
    cache = PagedKVCache(desc, free_order=order)
    mm = MirroredManager(nb, order)
    cache.mgr = mm.c                       # the executor and the scheduler share the C manager
    sched = Scheduler(mm, max_batch_tokens=96, chunk=48, max_running=12, max_blocks=40)
    sched.add_prefix(3, 37)
    reqs = []
    for i in range(16):
        pre = 3 if i % 3 == 0 else None
        prompt = int(rng.integers(40, 200)) if pre is None else 37 + int(rng.integers(1, 60))
        reqs.append(Request(rid=i, klass="a" if i % 2 else "b", prompt=prompt,
                            response=int(rng.integers(2, 40)), arrival=float(rng.integers(0, 20)),
                            priority=i % 2, prefix=pre))
    ex = StepExecutor(cache, max_decode=12, max_tokens=96, max_chunks=16, max_blocks=40)
    ex.overlap = overlap  # launches chained as programmatic dependents, or one after the other
    hk = np.zeros((L, nb, n_kv, 16, d), NP_STORAGE[dtype])
    hv = np.zeros_like(hk)
    scale = 1.0 / np.sqrt(d)
    clock = VirtualClock()
    stats = {"dec": 0, "pre": 0, "pairs": 0}

    def table_of(seq, mb=40):
        t, ctx = mm.o.block_table(int(seq))
        row = np.full(mb, -1, np.int32)
        row[: len(t)] = t
        return row, ctx

    def execute(plan):
        nd, nt = plan.n_dec, plan.n_pre_tokens
        dq = W.normal_values(rng, (L, max(nd, 1), n_q, d), dtype)
        dk = W.normal_values(rng, (L, max(nd, 1), n_kv, d), dtype)
        dv = W.normal_values(rng, (L, max(nd, 1), n_kv, d), dtype)
        pq = W.normal_values(rng, (L, max(nt, 1), n_q, d), dtype)
        pk = W.normal_values(rng, (L, max(nt, 1), n_kv, d), dtype)
        pv = W.normal_values(rng, (L, max(nt, 1), n_kv, d), dtype)
        dt = pkv.torch_dtype(dtype)
        d_out = torch.full((L, max(nd, 1), n_q, d), float("nan"), dtype=dt, device="cuda")
        p_out = torch.full((L, max(nt, 1), n_q, d), float("nan"), dtype=dt, device="cuda")
        dec_io = (to_torch(dq, dtype)[:, :nd], to_torch(dk, dtype)[:, :nd], to_torch(dv, dtype)[:, :nd], d_out[:, :nd])
        pre_io = (to_torch(pq, dtype)[:, :nt], to_torch(pk, dtype)[:, :nt], to_torch(pv, dtype)[:, :nt], p_out[:, :nt])
        ex.run(plan, dec_io, pre_io, scale)
        torch.cuda.synchronize()
        # oracle side, from its own manager's tables
        if len(plan.pairs):
            oracle.copy_blocks(hk, hv, plan.pairs)
            stats["pairs"] += len(plan.pairs)
        dt_rows = [table_of(s) for s in plan.dec_seq]
        pt_rows = [table_of(o.seq) for o, _ in plan.pre_chunks]
        got_d, got_p = as_f64(d_out), as_f64(p_out)
        for layer in range(L):
            if nt:
                oracle.kv_append(pk[layer, :nt], pv[layer, :nt], plan.pre_slots, hk[layer], hv[layer])
            if nd:
                oracle.kv_append(dk[layer, :nd], dv[layer, :nd], plan.dec_slots, hk[layer], hv[layer])
            if nt:
                tabs = np.stack([r for r, _ in pt_rows])
                lens = np.array([c for _, c in pt_rows], np.int32)
                want = oracle.paged_prefill(dtype, pq[layer, :nt], hk[layer], hv[layer], tabs, lens, plan.pre_qs, scale)
                assert np.max(np.abs(got_p[layer, :nt] - want)) <= TOL[dtype]
            if nd:
                tabs = np.stack([r for r, _ in dt_rows])
                lens = np.array([c for _, c in dt_rows], np.int32)
                want = oracle.paged_decode(dtype, dq[layer, :nd], hk[layer], hv[layer], tabs, lens, scale)
                assert np.max(np.abs(got_d[layer, :nd] - want)) <= TOL[dtype]
        stats["dec"] += nd
        stats["pre"] += nt
        clock.t += 1.0

    serve(sched, reqs, execute, clock, clock.wait_until)
    assert all(r.state == "done" and r.generated == r.response for r in reqs)
    assert stats["dec"] > 0 and stats["pre"] > 0 and stats["pairs"] > 0
    assert sched.prefix_forks > 0
    assert pkv.pkv_get_device_status() == 0
