"""Continuous-batching scheduler (host only), on the C block manager with a virtual clock.

"PagedAttention e continuous batching", "01 - Conceito", paragraphs 5-8: iteration-level refill,
a token budget per iteration with long prefills sliced, admission in blocks that refuses early,
preemption when an append finds no block, shared prefixes, and per-class latency metrics.
Every manager call the scheduler makes is mirrored into the block-manager oracle and compared.
"""
import math

import numpy as np
import pytest

from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300.scheduler import Request, Scheduler, serve, synthetic_trace


class MirroredManager:
    """The C manager with every mutating call replayed on the oracle manager and compared."""

    def __init__(self, num_blocks, order=None):
        self.c = pkv.BlockManager(num_blocks, free_order=order)
        self.o = BlockManagerOracle(num_blocks, free_order=order)
        self.num_blocks, self.block_size = num_blocks, 16
        self.calls = 0

    def _st(self, rc):
        return pkv.STATUS_NAMES[rc]

    def add_seq(self, sid, n, reserve=0):
        rc, slots = self.c.add_seq(sid, n, reserve)
        st, want = self.o.add_seq(sid, n, reserve)
        assert self._st(rc) == st and slots.tolist() == want
        self.calls += 1
        return rc, slots

    def extend(self, sid, n, slots_out=None):
        rc, slots, src, dst = self.c.extend(sid, n)
        st, want, s_o, d_o = self.o.extend(sid, n)
        assert self._st(rc) == st
        if st == "ok":
            assert (slots.tolist(), src, dst) == (want, s_o, d_o)
        self.calls += 1
        return rc, slots, src, dst

    def append_slot(self, sid):
        r = self.c.append_slot(sid)
        st, slot, src, dst = self.o.append_slot(sid)
        assert self._st(r[0]) == st
        if st == "ok":
            assert r[1:] == (slot, src, dst)
        self.calls += 1
        return r

    def append_batch(self, sids):
        """One C call for the batch; the oracle appends the same sequences one at a time, up to and
        including the first that fails, and must agree on every slot, pair, count and status."""
        rc, slots, pairs, n_done = self.c.append_batch(sids)
        want_slots, want_pairs, st = [], [], "ok"
        for sid in sids:
            st, slot, src, dst = self.o.append_slot(int(sid))
            if st != "ok":
                break
            want_slots.append(slot)
            if src >= 0:
                want_pairs.append([src, dst])
        assert self._st(rc) == st and n_done == len(want_slots)
        assert slots.tolist() == want_slots and pairs.tolist() == want_pairs
        self.calls += 1
        return rc, slots, pairs, n_done

    def fork(self, p, c):
        rc = self.c.fork(p, c)
        assert self._st(rc) == self.o.fork(p, c)
        return rc

    def free_seq(self, sid):
        rc = self.c.free_seq(sid)
        assert self._st(rc) == self.o.free_seq(sid)
        return rc

    def pack_tables(self, ids, mb):
        rc, t, ln = self.c.pack_tables(ids, mb)
        for i, sid in enumerate(ids):
            t_o, ctx = self.o.block_table(int(sid))
            assert t[i, : len(t_o)].tolist() == t_o and np.all(t[i, len(t_o):] == -1) and ln[i] == ctx
        return rc, t, ln

    def stats(self):
        s = self.c.stats()
        assert s == self.o.stats()
        return s

    def refcount(self, b):
        return self.c.refcount(b)


class VirtualClock:
    def __init__(self):
        self.t = 0.0

    def __call__(self):
        return self.t

    def wait_until(self, t):
        self.t = max(self.t, t)


def run(sched, reqs, check_plan=None):
    clock = VirtualClock()
    plans = []

    def execute(plan):
        if check_plan:
            check_plan(plan)
        plans.append(plan)
        clock.t += 1.0

    steps = serve(sched, reqs, execute, clock, clock.wait_until)
    return steps, plans


def plan_invariants(sched):
    def check(plan):
        assert plan.n_dec + plan.n_pre_tokens <= sched.max_batch_tokens
        assert all(n <= sched.chunk for _, n in plan.pre_chunks)
        slots = np.concatenate([plan.dec_slots, plan.pre_slots])
        assert len(np.unique(slots)) == len(slots)                    # no two tokens share a slot
        for i in range(plan.n_dec):                                    # decode slot = position len-1
            p = int(plan.dec_lens[i]) - 1
            assert plan.dec_slots[i] == int(plan.dec_tables[i, p // 16]) * 16 + p % 16
        assert set(plan.pairs[:, 1].tolist()).isdisjoint(plan.pairs[:, 0].tolist())
    return check


def test_all_requests_complete_with_budget_and_metrics():
    mgr = MirroredManager(600)
    sched = Scheduler(mgr, max_batch_tokens=256, chunk=128, max_blocks=140)
    reqs = synthetic_trace(40, seed=1, rate_per_s=2.0,
                           classes=[("chat", 0.8, 1), ("doc", 0.2, 0)])
    for r in reqs:                     # shrink the long class to fit the small pool
        if r.klass == "doc":
            r.prompt, r.response = 700 + r.rid, 20
        r.response = min(r.response, 200)
    steps, plans = run(sched, reqs, plan_invariants(sched))
    assert len(sched.done) == 40 and not sched.rejected
    for r in sched.done:
        assert r.generated == r.response == len(r.token_times)
        assert r.arrival <= r.t_admit <= r.t_first
        assert all(b > a for a, b in zip(r.token_times, r.token_times[1:]))
    m = sched.metrics()
    assert set(m["classes"]) == {"chat", "doc"}
    assert m["classes"]["chat"]["tokens"] == sum(r.response for r in reqs if r.klass == "chat")
    assert m["blocks"]["used_blocks"] == 0 and mgr.stats()["n_seqs"] == 0
    # long prompts were sliced: some doc request needed several chunks
    assert any(sum(1 for p in plans for o, _ in p.pre_chunks if o is r) >= 5 for r in sched.done if r.klass == "doc")


def test_decode_is_not_stalled_by_a_long_prompt():
    """A 6,000-token prompt arriving mid-stream is prefilled in chunks; running chat requests
    keep emitting one token every iteration (inter-token gap of exactly one iteration)."""
    mgr = MirroredManager(1200)
    sched = Scheduler(mgr, max_batch_tokens=512, chunk=256, max_blocks=400)
    chat = [Request(rid=i, klass="chat", prompt=100, response=60, arrival=0.0, priority=1) for i in range(8)]
    doc = Request(rid=99, klass="doc", prompt=6000, response=4, arrival=5.0, priority=0)
    run(sched, chat + [doc], plan_invariants(sched))
    for r in chat:
        gaps = np.diff(r.token_times)
        assert np.all(gaps == 1.0)
    m = sched.metrics()["classes"]
    assert m["chat"]["itl_p99"] == 1.0
    assert doc.t_first - doc.t_admit >= math.ceil(6000 / 256) - 1


def test_refuses_early_what_can_never_fit():
    mgr = MirroredManager(64)
    sched = Scheduler(mgr, max_blocks=64)
    ok = Request(rid=0, klass="chat", prompt=100, response=10, arrival=0.0)
    big = Request(rid=1, klass="chat", prompt=64 * 16, response=10, arrival=0.0)
    empty = Request(rid=2, klass="chat", prompt=0, response=10, arrival=0.0)
    assert sched.submit(ok) and not sched.submit(big) and not sched.submit(empty)
    assert big.state == "rejected" and "blocks" in big.error
    clock = VirtualClock()

    def execute(plan):
        clock.t += 1

    serve(sched, [], execute, clock, clock.wait_until)
    assert ok.state == "done" and sched.metrics()["rejected"] == 2


def test_preemption_on_append_oom_and_recompute():
    """A pool too small for every response to run to the end: the scheduler preempts (lowest
    priority, latest arrival), the victim recomputes its cache and still emits each token once."""
    mgr = MirroredManager(60)
    sched = Scheduler(mgr, max_batch_tokens=256, chunk=64, max_blocks=60, headroom_blocks=1)
    reqs = [Request(rid=i, klass="hi" if i < 2 else "lo", prompt=120, response=200, arrival=0.1 * i,
                    priority=1 if i < 2 else 0) for i in range(5)]
    steps, plans = run(sched, reqs, plan_invariants(sched))
    assert sched.preemptions > 0
    assert all(r.state == "done" and r.generated == 200 == len(r.token_times) for r in reqs)
    # the high-priority pair is never the victim while low-priority work is running
    assert all(r.preemptions == 0 for r in reqs[:2])
    assert sum(r.preemptions for r in reqs[2:]) == sched.preemptions
    assert mgr.stats()["append_oom"] >= sched.preemptions
    assert mgr.stats()["used_blocks"] == 0


def test_shared_prefix_roots_fork_and_copy_on_write():
    mgr = MirroredManager(400)
    sched = Scheduler(mgr, max_batch_tokens=256, chunk=128, max_blocks=80)
    sched.add_prefix(7, 200)            # 12 full blocks + a partial one
    reqs = [Request(rid=i, klass="chat", prompt=200 + 30 + i, response=12, arrival=0.0, prefix=7) for i in range(10)]
    run(sched, reqs, plan_invariants(sched))
    st = mgr.stats()
    assert all(r.state == "done" for r in reqs)
    assert sched.prefix_forks == 10 and sched.metrics()["blocks"]["prefix_hit_rate"] == 1.0
    assert st["cow_copies"] == 10       # each request copied the root's partial tail once
    assert st["prefix_hits"] == 10 * 13
    assert st["n_seqs"] == 1 and st["used_blocks"] == 13   # only the resident root remains


def test_priorities_order_admission():
    mgr = MirroredManager(40)
    sched = Scheduler(mgr, max_batch_tokens=64, chunk=64, max_blocks=40, max_running=1)
    lo = Request(rid=0, klass="lo", prompt=50, response=3, arrival=0.0, priority=0)
    hi = Request(rid=1, klass="hi", prompt=50, response=3, arrival=0.5, priority=5)
    first = Request(rid=2, klass="lo", prompt=50, response=3, arrival=0.0, priority=0)
    run(sched, [first, lo, hi])
    # "first"/"lo" arrive together; once the slot frees, hi (higher priority) goes before the other lo
    order = sorted([first, lo, hi], key=lambda r: r.t_admit)
    assert order[0].priority == 0 and order[1] is hi


def test_deterministic():
    def once():
        mgr = MirroredManager(300)
        sched = Scheduler(mgr, max_batch_tokens=128, chunk=64, max_blocks=100)
        reqs = synthetic_trace(25, seed=3, rate_per_s=1.0)
        for r in reqs:
            r.prompt, r.response = min(r.prompt, 600), min(r.response, 150)
        run(sched, reqs)
        return [(r.rid, r.t_admit, r.t_first, tuple(r.token_times)) for r in sched.done]
    assert once() == once()
