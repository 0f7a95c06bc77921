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


# ---- extend by a chunk (chunked prefill, "01 - Conceito" paragraph 5) --------------------------
# The reading: a chunk of n tokens is all or nothing, and when it is admitted it equals n single
# appends of "La idea de PagedAttention" step 3. The pin below checks exactly that against the
# single-append path (itself pinned above), never against extend's own block arithmetic: extend(s, n)
# is "ok" iff n successive append_slot(s) calls on a deep copy all succeed, and then the two
# managers are equal (tables, lengths, reference counts, free-list order, counters), the slots
# agree and the one copy-on-write pair, if any, is the appends' pair.

import copy  # noqa: E402


def full_state(m: BlockManagerOracle):
    return snapshot(m) + (m.alloc_failures, m.prefix_hits, m.cow_copies, m.append_oom)


def extend_agrees_with_appends(m: BlockManagerOracle, seq: int, n: int) -> bool:
    """True when extend(seq, n) on a copy of m behaves like n appends on another copy."""
    ref = copy.deepcopy(m)
    slots, pairs, ok = [], [], True
    for _ in range(n):
        st, slot, src, dst = ref.append_slot(seq)
        if st != "ok":
            ok = False
            break
        slots.append(slot)
        if src >= 0:
            pairs.append((src, dst))
    ext = copy.deepcopy(m)
    before = full_state(ext)
    try:
        st, got_slots, src, dst = ext.extend(seq, n)
    except AssertionError:      # a wrong admission test lets the chunk run out of blocks midway
        return False
    if not ok:
        # refused: nothing moves but one allocation failure and one append OOM
        want = before[:-4] + (before[-4] + 1, before[-3], before[-2], before[-1] + 1)
        return st == "no_blocks" and full_state(ext) == want
    if st != "ok" or got_slots != slots or full_state(ext) != full_state(ref) or len(pairs) > 1:
        return False
    return (src, dst) == (pairs[0] if pairs else (-1, -1))


def random_manager(rng: random.Random):
    """A seeded manager state with shared prefixes, shared partial tails and a small free list."""
    nb = rng.randint(6, 40)
    m = BlockManagerOracle(nb, free_order=rng.sample(range(nb), nb))
    next_id = 0
    for _ in range(rng.randint(2, 30)):
        live = list(m.tables)
        r = rng.random()
        if r < 0.35 or not live:
            m.add_seq(next_id, rng.randint(0, 60))
            next_id += 1
        elif r < 0.6:
            m.fork(rng.choice(live), next_id)    # shares every block, the partial tail included
            next_id += 1
        elif r < 0.9:
            m.append_slot(rng.choice(live))
        else:
            m.free_seq(rng.choice(live))
    return m


def boundary_chunks(m: BlockManagerOracle, seq: int):
    """Chunk sizes around the largest chunk the pool can hold (found by single appends)."""
    ref = copy.deepcopy(m)
    fit = 0
    while ref.append_slot(seq)[0] == "ok":
        fit += 1
    return sorted({0, 1, 2, BS - 1, BS, BS + 1, max(fit - BS, 0), max(fit - 1, 0), fit, fit + 1, fit + 2,
                   fit + BS})


def test_extend_equals_successive_appends_at_the_admission_boundary():
    rng = random.Random(2024)
    n_checked = n_refused = n_cow = 0
    for _ in range(400):
        m = random_manager(rng)
        if not m.tables:
            continue
        for seq in list(m.tables):
            shared_tail = m.ctx[seq] % BS != 0 and m.ref[m.tables[seq][-1]] > 1
            for n in boundary_chunks(m, seq):
                assert extend_agrees_with_appends(m, seq, n), (seq, n)
                n_checked += 1
                probe = copy.deepcopy(m)
                st = probe.extend(seq, n)[0]
                n_refused += st == "no_blocks"
                n_cow += st == "ok" and n > 0 and shared_tail
    assert n_checked > 2000 and n_refused > 300 and n_cow > 100   # both sides of the boundary, with CoW


def _planted_extend(m, seq_id, n_tokens, slack: int, cow_block: bool):
    """extend with its admission test altered: `slack` extra blocks believed free, and the copy-on-
    write block counted only if cow_block. The rest follows the oracle's steps."""
    if seq_id not in m.tables or n_tokens <= 0:
        return BlockManagerOracle.extend(m, seq_id, n_tokens)
    cow = m.ctx[seq_id] % BS != 0 and m.ref[m.tables[seq_id][-1]] > 1
    need = -(-(m.ctx[seq_id] + n_tokens) // BS) - len(m.tables[seq_id]) + (1 if cow and cow_block else 0)
    if need > len(m.free) + slack:
        m.alloc_failures += 1
        m.append_oom += 1
        return "no_blocks", [], -1, -1
    slots, src, dst = [], -1, -1
    for _ in range(n_tokens):
        st, slot, s_, d_ = m.append_slot(seq_id)
        assert st == "ok"
        slots.append(slot)
        if s_ >= 0:
            src, dst = s_, d_
    return "ok", slots, src, dst


class _OffByOne(BlockManagerOracle):
    """Planted mistake: admits a chunk that needs one block more than the pool holds."""

    def extend(self, seq_id, n_tokens):
        return _planted_extend(self, seq_id, n_tokens, slack=1, cow_block=True)


class _NoCowBlock(BlockManagerOracle):
    """Planted mistake: forgets the extra block a copy-on-write first token takes."""

    def extend(self, seq_id, n_tokens):
        return _planted_extend(self, seq_id, n_tokens, slack=0, cow_block=False)


@pytest.mark.parametrize("mutant", [_OffByOne, _NoCowBlock])
def test_extend_pin_catches_planted_mistakes(mutant):
    """The pin above has teeth: each planted admission mistake breaks it on some seeded state."""
    rng = random.Random(2024)
    for _ in range(400):
        m = random_manager(rng)
        bad = mutant(m.num_blocks)
        bad.__dict__.update(copy.deepcopy(m.__dict__))
        for seq in list(bad.tables):
            for n in boundary_chunks(bad, seq):
                if not extend_agrees_with_appends(bad, seq, n):
                    return
    pytest.fail(f"{mutant.__name__} was not caught")
