"""The C block manager (libpkv) against the Python block-manager oracle, bit-exact.

After every operation of every log: status, returned slots and copy-on-write pairs, every
block table and context length, every refcount, the free list in order, and the counters.
Runs on the CPU (the manager is host code).
"""
import copy
import itertools
import random

import numpy as np
import pytest

from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W


def status(rc: int) -> str:
    return pkv.STATUS_NAMES[rc]


def compare(c: pkv.BlockManager, o: BlockManagerOracle):
    assert c.free_list() == o.free_list()
    assert c.refcounts() == o.refcounts()
    for sid in o.tables:
        rc, table, ctx = c.block_table(sid)
        assert rc == pkv.PKV_OK
        assert table == o.tables[sid] and ctx == o.ctx[sid]
    assert c.stats() == o.stats()


def apply_both(c, o, op):
    kind = op[0]
    if kind == "add":
        rc, slots = c.add_seq(op[1], op[2], op[3] if len(op) > 3 else 0)
        st, want = o.add_seq(op[1], op[2], op[3] if len(op) > 3 else 0)
        assert status(rc) == st
        assert slots.tolist() == want
    elif kind == "fork":
        assert status(c.fork(op[1], op[2])) == o.fork(op[1], op[2])
    elif kind == "append":
        rc, slot, src, dst = c.append_slot(op[1])
        st, slot_o, src_o, dst_o = o.append_slot(op[1])
        assert status(rc) == st
        if st == "ok":
            assert (slot, src, dst) == (slot_o, src_o, dst_o)
    elif kind == "extend":
        rc, slots, src, dst = c.extend(op[1], op[2])
        st, want, src_o, dst_o = o.extend(op[1], op[2])
        assert status(rc) == st
        if st == "ok":
            assert (slots.tolist(), src, dst) == (want, src_o, dst_o)
    elif kind == "free":
        assert status(c.free_seq(op[1])) == o.free_seq(op[1])
    else:
        raise ValueError(kind)


ALPHABET = [("add", 0, 17), ("add", 1, 1), ("fork", 0, 2), ("append", 0), ("append", 2), ("free", 0),
            ("add", 3, 40)]


def test_bruteforce_depth6_bitexact():
    """Every operation sequence up to depth 6 over a 7-op alphabet on a 4-block pool."""
    visited = 0

    def dfs(c, o, depth):
        nonlocal visited
        if depth == 0:
            return
        for op in ALPHABET:
            c2, o2 = c.clone(), copy.deepcopy(o)
            apply_both(c2, o2, op)
            compare(c2, o2)
            visited += 1
            dfs(c2, o2, depth - 1)

    dfs(pkv.BlockManager(4, free_order=[2, 0, 3, 1]), BlockManagerOracle(4, free_order=[2, 0, 3, 1]), 6)
    assert visited == sum(7 ** k for k in range(1, 7))


@pytest.mark.parametrize("seed", range(6))
def test_random_logs_bitexact(seed):
    rng = random.Random(seed)
    nb = rng.choice([8, 33, 200])
    order = W.free_order(nb, seed)
    c, o = pkv.BlockManager(nb, free_order=order), BlockManagerOracle(nb, free_order=order)
    next_id = 0
    for _ in range(2500):
        live = list(o.tables)
        r = rng.random()
        if r < 0.12 or not live:
            op = ("add", next_id, rng.randint(0, 90), rng.choice([0, 0, 16, 100]))
            next_id += 1
        elif r < 0.22:
            op = ("fork", rng.choice(live), next_id)
            next_id += 1
        elif r < 0.78:
            op = ("append", rng.choice(live + [10 ** 9]))
        elif r < 0.85:
            op = ("extend", rng.choice(live + [10 ** 9]), rng.choice([0, 1, 5, 16, 37, 200]))
        else:
            op = ("free", rng.choice(live + [-5]))
        apply_both(c, o, op)
        compare(c, o)


def test_append_batch_matches_single_appends():
    order = W.free_order(64, 3)
    c, o = pkv.BlockManager(64, free_order=order), BlockManagerOracle(64, free_order=order)
    for s, n in enumerate([15, 16, 1, 33]):
        apply_both(c, o, ("add", s, n))
    apply_both(c, o, ("fork", 0, 10))
    apply_both(c, o, ("fork", 2, 11))
    ids = [0, 10, 1, 2, 11, 3]
    for _ in range(20):
        rc, slots, pairs, n_done = c.append_batch(ids)
        assert rc == pkv.PKV_OK and n_done == len(ids)
        want_pairs = []
        for i, sid in enumerate(ids):
            st, slot, src, dst = o.append_slot(sid)
            assert st == "ok" and slots[i] == slot
            if src >= 0:
                want_pairs.append([src, dst])
        assert pairs.tolist() == want_pairs
        compare(c, o)


def test_extend_equals_successive_appends_and_is_all_or_nothing():
    order = W.free_order(40, 4)
    c, o = pkv.BlockManager(40, free_order=order), BlockManagerOracle(40, free_order=order)
    apply_both(c, o, ("add", 0, 20))
    apply_both(c, o, ("fork", 0, 1))
    apply_both(c, o, ("fork", 0, 2))
    # chunk into a shared partial tail: one copy, then fresh blocks, slots in position order
    rc, slots, src, dst = c.extend(1, 50)
    assert rc == pkv.PKV_OK and src == o.tables[0][-1] and dst >= 0
    st, want, src_o, dst_o = o.extend(1, 50)
    assert (st, slots.tolist(), src, dst) == ("ok", want, src_o, dst_o)
    compare(c, o)
    # a chunk the pool cannot hold changes nothing (counts one failure and one append OOM)
    before = (c.free_list(), c.refcounts(), c.block_table(2))
    rc, slots, src, dst = c.extend(2, 16 * 40)
    assert rc == pkv.PKV_ERR_NO_BLOCKS and len(slots) == 0
    assert o.extend(2, 16 * 40)[0] == "no_blocks"
    assert (c.free_list(), c.refcounts(), c.block_table(2)) == before
    compare(c, o)
    # a cloned manager replaying the chunk as single appends ends in the same state
    c2 = c.clone()
    rc, slots, _, _ = c.extend(2, 33)
    singles = [c2.append_slot(2) for _ in range(33)]
    assert [s_[1] for s_ in singles] == slots.tolist()
    assert c2.free_list() == c.free_list() and c2.stats() == c.stats()


def test_injected_failure_in_extend_rolls_back():
    c = pkv.BlockManager(12)
    assert c.add_seq(0, 20)[0] == pkv.PKV_OK
    assert c.fork(0, 1) == pkv.PKV_OK
    before = (c.free_list(), c.refcounts(), c.block_table(0), c.block_table(1))
    for after in range(4):                             # the copy, then each fresh block
        c.inject_alloc_failure(after)
        rc, _, _, _ = c.extend(1, 60)
        assert rc == pkv.PKV_ERR_NO_BLOCKS
        assert (c.free_list(), c.refcounts(), c.block_table(0), c.block_table(1)) == before
    rc, slots, src, dst = c.extend(1, 60)
    assert rc == pkv.PKV_OK and src >= 0 and len(slots) == 60


def test_append_batch_stops_at_first_failure():
    c = pkv.BlockManager(3)
    assert c.add_seq(0, 16)[0] == pkv.PKV_OK
    assert c.add_seq(1, 16)[0] == pkv.PKV_OK
    rc, slots, pairs, n_done = c.append_batch([0, 1, 0])
    assert rc == pkv.PKV_ERR_NO_BLOCKS and n_done == 1 and len(slots) == 1
    assert c.stats()["append_oom"] == 1


def test_injected_allocation_failure_rolls_back_completely():
    order = W.free_order(16, 9)
    c = pkv.BlockManager(16, free_order=order)
    assert c.add_seq(0, 20)[0] == pkv.PKV_OK
    before = (c.free_list(), c.refcounts(), c.block_table(0))
    for after in range(3):
        assert c.inject_alloc_failure(after) == pkv.PKV_OK
        rc, _ = c.add_seq(1, 60)                       # needs 4 blocks; allocation `after` fails
        assert rc == pkv.PKV_ERR_NO_BLOCKS
        assert (c.free_list(), c.refcounts(), c.block_table(0)) == before
        assert c.block_table(1)[0] == pkv.PKV_ERR_INVALID_ARG
    # the injection fires once; afterwards the same admission succeeds
    assert c.add_seq(1, 60)[0] == pkv.PKV_OK


def test_injected_failure_on_cow_append_is_transactional():
    c = pkv.BlockManager(8)
    assert c.add_seq(0, 20)[0] == pkv.PKV_OK
    assert c.fork(0, 1) == pkv.PKV_OK
    before = (c.free_list(), c.refcounts(), c.block_table(0), c.block_table(1))
    c.inject_alloc_failure(0)
    rc, slot, src, dst = c.append_slot(1)
    assert rc == pkv.PKV_ERR_NO_BLOCKS
    assert (c.free_list(), c.refcounts(), c.block_table(0), c.block_table(1)) == before
    rc, slot, src, dst = c.append_slot(1)
    assert rc == pkv.PKV_OK and src >= 0


def test_capacity_example_through_the_c_manager(golden):
    """The pages' 23,859 MiB pool admits 10 sessions (KV + 144 MiB state), refusing the 11th."""
    pool = golden["pool_mib"]["value"]
    state = golden["state_mib_per_sequence"]["value"]
    tokens = golden["session_tokens"]["value"]
    c = pkv.BlockManager(pool)
    n = 0
    while True:
        rc, _ = c.add_seq(2 * n, tokens, state * 16)
        if rc != pkv.PKV_OK:
            break
        assert c.add_seq(2 * n + 1, state * 16)[0] == pkv.PKV_OK
        n += 1
    assert n == golden["paged_sessions"]["value"] and rc == pkv.PKV_ERR_NO_BLOCKS
    assert c.stats()["alloc_failures"] == 1


def test_pack_tables_pads_with_minus_one():
    c = pkv.BlockManager(10, free_order=list(range(9, -1, -1)))
    c.add_seq(7, 20)
    c.add_seq(8, 3)
    rc, tables, lens = c.pack_tables([8, 7], 4)
    assert rc == pkv.PKV_OK
    assert tables.tolist() == [[7, -1, -1, -1], [9, 8, -1, -1]] and lens.tolist() == [3, 20]
    assert c.pack_tables([7], 1)[0] == pkv.PKV_ERR_INVALID_ARG
    assert c.pack_tables([99], 4)[0] == pkv.PKV_ERR_INVALID_ARG


def test_prefix_churn_log_replays_identically():
    """The shared-prefix churn workload's operation log (first 40 steps) on both managers."""
    wl = W.prefix_churn(n_steps=40)
    order = W.free_order(wl.num_blocks, wl.seed)
    c, o = pkv.BlockManager(wl.num_blocks, free_order=order), BlockManagerOracle(wl.num_blocks, free_order=order)
    roots = [10 ** 6 + g for g in range(wl.n_groups)]
    for g, r in enumerate(roots):
        apply_both(c, o, ("add", r, wl.group_prompt[g]))
    live = []
    for m, g in enumerate(wl.member_group):
        apply_both(c, o, ("fork", roots[g], m))
        live.append(m)
    for events in wl.steps:
        for sid in live:
            apply_both(c, o, ("append", sid))
        for old, new, g in events:
            apply_both(c, o, ("free", old))
            apply_both(c, o, ("fork", roots[g], new))
            live[live.index(old)] = new
        compare(c, o)
    assert o.cow_copies > 0 and o.prefix_hits > 0
