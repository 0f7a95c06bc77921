"""Pins for the block-manager oracle, independent of its own code paths.

Checked after every operation, over every operation sequence up to depth 6 on a 4-block
pool and over long seeded random logs:
  * conservation: refcount of every block == number of tables holding it; the free list is
    exactly the blocks with refcount 0, without duplicates;
  * bounded internal fragmentation ("Propiedades": at most B_block - 1 = 15 rows per
    sequence) and full coverage (16 * n_blocks >= context);
  * failed operations leave the state unchanged ("refuse early with a clear error");
  * an append writes position ctx-1 of the sequence's last block, and that block is then
    referenced by no other sequence (nobody else can read the row being written);
  * copy-on-write only ever copies a block that another sequence still references.
"""
import itertools
import random

import pytest

from oracle import BlockManagerOracle

BS = 16


def snapshot(m: BlockManagerOracle):
    return (tuple(m.free), tuple(m.ref), tuple(sorted((k, tuple(v)) for k, v in m.tables.items())),
            tuple(sorted(m.ctx.items())))


def check_invariants(m: BlockManagerOracle):
    count = [0] * m.num_blocks
    for t in m.tables.values():
        for b in t:
            count[b] += 1
    assert count == m.ref
    free = list(m.free)
    assert len(free) == len(set(free))
    assert sorted(free) == [b for b in range(m.num_blocks) if m.ref[b] == 0]
    for s, t in m.tables.items():
        n = m.ctx[s]
        assert len(t) * BS >= n
        assert len(t) * BS - n <= BS - 1
        assert len(t) == -(-n // BS)


def apply(m, op):
    kind = op[0]
    if kind == "add":
        return m.add_seq(op[1], op[2])[0]
    if kind == "fork":
        return m.fork(op[1], op[2])
    if kind == "append":
        return m.append_slot(op[1])[0]
    if kind == "free":
        return m.free_seq(op[1])
    raise ValueError(kind)


ALPHABET = [("add", 0, 17), ("add", 1, 1), ("fork", 0, 2), ("append", 0), ("append", 2), ("free", 0)]


def test_bruteforce_depth6_invariants():
    n_checked = 0
    for depth in range(1, 7):
        for ops in itertools.product(ALPHABET, repeat=depth):
            m = BlockManagerOracle(4)
            for op in ops:
                before = snapshot(m)
                st = apply(m, op)
                if st != "ok":
                    assert snapshot(m) == before, (ops, op)
                check_invariants(m)
                n_checked += 1
    assert n_checked > 50000


def test_cow_only_copies_a_still_shared_block():
    m = BlockManagerOracle(8)
    assert m.add_seq(1, 20)[0] == "ok"           # 2 blocks, tail has 4 rows
    assert m.fork(1, 2) == "ok"
    tail = m.tables[1][-1]
    st, slot, src, dst = m.append_slot(2)
    assert st == "ok" and src == tail and dst != tail and m.ref[tail] == 1
    assert slot == dst * BS + 20 % BS
    # the original holder is now the last one: it writes in place
    st, slot, src, dst = m.append_slot(1)
    assert st == "ok" and src == -1 and slot == tail * BS + 4


def test_full_shared_tail_opens_a_new_block():
    m = BlockManagerOracle(8)
    assert m.add_seq(1, 32)[0] == "ok"           # exactly 2 full blocks
    assert m.fork(1, 2) == "ok"
    st, slot, src, dst = m.append_slot(2)
    assert st == "ok" and src == -1 and slot % BS == 0 and slot // BS not in m.tables[1]


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_logs_invariants_and_slots(seed):
    rng = random.Random(seed)
    m = BlockManagerOracle(64, free_order=rng.sample(range(64), 64))
    next_id = 0
    for _ in range(3000):
        live = list(m.tables)
        r = rng.random()
        before = snapshot(m)
        if r < 0.15 or not live:
            n = rng.randint(0, 70)
            st, slots = m.add_seq(next_id, n)
            if st == "ok":
                t = m.tables[next_id]
                assert slots == [t[j // BS] * BS + j % BS for j in range(n)]
            next_id += 1
        elif r < 0.25:
            p = rng.choice(live)
            st = m.fork(p, next_id)
            next_id += 1
        elif r < 0.85:
            s = rng.choice(live)
            st, slot, src, dst = m.append_slot(s)
            if st == "ok":
                assert slot // BS == m.tables[s][-1]
                assert slot % BS == (m.ctx[s] - 1) % BS
                assert m.ref[m.tables[s][-1]] == 1
                if src >= 0:
                    assert m.ref[src] >= 1 and m.ref[dst] == 1
        else:
            s = rng.choice(live)
            st = m.free_seq(s)
        if st != "ok":
            assert snapshot(m) == before
        check_invariants(m)


def test_error_statuses():
    m = BlockManagerOracle(2)
    assert m.add_seq(5, 17)[0] == "ok"
    assert m.add_seq(5, 1)[0] == "invalid"        # id in use
    assert m.add_seq(6, -1)[0] == "invalid"
    assert m.add_seq(6, 1)[0] == "no_blocks"      # pool empty
    assert m.fork(9, 10) == "invalid"             # unknown parent
    assert m.fork(5, 5) == "invalid"
    assert m.append_slot(9)[0] == "invalid"
    for _ in range(15):
        assert m.append_slot(5)[0] == "ok"
    assert m.append_slot(5)[0] == "no_blocks"     # 32 rows used, no block left
    assert m.stats()["append_oom"] == 1
    assert m.free_seq(5) == "ok"
    assert m.free_seq(5) == "invalid"             # double free
    assert m.stats()["free_blocks"] == 2
