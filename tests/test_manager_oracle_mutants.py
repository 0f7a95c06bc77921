"""The block-manager pins reject a plausible mistake anywhere in the manager oracle.

Each mutant below is the oracle with one step of "La idea de PagedAttention" (steps 1-4) or of
"01 - Conceito" paragraphs 6-7 done wrong. The pin functions of test_manager_oracle_pins.py run
against it (their manager class swapped for the mutant): at least one of them must fail. The
unchanged oracle, run the same way, passes them all.
"""
import pytest

import test_manager_oracle_pins as P
from oracle import BlockManagerOracle


class _CowForgotten(BlockManagerOracle):
    """Appends into a partially filled tail that another sequence still holds, in place."""

    def append_slot(self, seq_id):
        if seq_id in self.tables and self.ctx[seq_id] % self.block_size != 0:
            tail = self.tables[seq_id][-1]
            n = self.ctx[seq_id]
            self.ctx[seq_id] = n + 1
            return "ok", self._slot(tail, n), -1, -1
        return super().append_slot(seq_id)


class _CowOfFullTail(BlockManagerOracle):
    """Treats a full shared tail like a partial one: replaces it instead of opening a new block."""

    def append_slot(self, seq_id):
        if seq_id in self.tables and self.tables[seq_id] and self.ctx[seq_id] % self.block_size == 0:
            tail = self.tables[seq_id][-1]
            if self.ref[tail] > 1 and self.free:
                b = self.free.popleft()
                self.ref[b] = 1
                self.ref[tail] -= 1
                self.tables[seq_id][-1] = b
                n = self.ctx[seq_id]
                self.ctx[seq_id] = n + 1
                return "ok", self._slot(b, n), tail, b
        return super().append_slot(seq_id)


class _CowKeepsOldReference(BlockManagerOracle):
    """Copies on write but leaves the reference the sequence held on the old tail."""

    def append_slot(self, seq_id):
        out = super().append_slot(seq_id)
        if out[0] == "ok" and out[2] >= 0:
            self.ref[out[2]] += 1
        return out


class _SlotOffByOne(BlockManagerOracle):
    """Hands out the slot of the position after the new token."""

    def append_slot(self, seq_id):
        st, slot, src, dst = super().append_slot(seq_id)
        if st == "ok":
            slot = self._slot(slot // self.block_size, self.ctx[seq_id])
        return st, slot, src, dst


class _OomNotCounted(BlockManagerOracle):
    """Refuses an append that finds no block but does not count it as an append OOM."""

    def append_slot(self, seq_id):
        out = super().append_slot(seq_id)
        if out[0] == "no_blocks":
            self.append_oom -= 1
        return out


class _OneBlockTooMany(BlockManagerOracle):
    """Admits a prompt with one block more than it needs."""

    def _blocks_for(self, n_tokens):
        return super()._blocks_for(n_tokens) + (1 if n_tokens > 0 else 0)


class _RefusesWhenExactlyEnough(BlockManagerOracle):
    """Admission refuses a prompt that needs exactly the blocks left."""

    def add_seq(self, seq_id, n_prompt, reserve_tokens=0):
        if seq_id not in self.tables and n_prompt >= 0 and reserve_tokens >= 0 and \
                self._blocks_for(n_prompt) + self._blocks_for(reserve_tokens) == len(self.free) > 0:
            self.alloc_failures += 1
            return "no_blocks", []
        return super().add_seq(seq_id, n_prompt, reserve_tokens)


class _ForkWithoutReferences(BlockManagerOracle):
    """Shares the parent's blocks without counting the child's references."""

    def fork(self, parent, child):
        st = super().fork(parent, child)
        if st == "ok":
            for b in self.tables[child]:
                self.ref[b] -= 1
        return st


class _FreeLeaks(BlockManagerOracle):
    """Drops the references of a freed sequence but never returns its blocks to the free list."""

    def free_seq(self, seq_id):
        if seq_id not in self.tables:
            return "invalid"
        for b in self.tables.pop(seq_id):
            self.ref[b] -= 1
        del self.ctx[seq_id]
        return "ok"


class _FreeReleasesShared(BlockManagerOracle):
    """Returns every block of a freed sequence to the free list, shared ones included."""

    def free_seq(self, seq_id):
        if seq_id not in self.tables:
            return "invalid"
        for b in self.tables.pop(seq_id):
            self.ref[b] = max(self.ref[b] - 1, 0)
            if b not in self.free:
                self.free.append(b)
        del self.ctx[seq_id]
        return "ok"


MUTANTS = [_CowForgotten, _CowOfFullTail, _CowKeepsOldReference, _SlotOffByOne, _OomNotCounted, _OneBlockTooMany,
           _RefusesWhenExactlyEnough, _ForkWithoutReferences, _FreeLeaks, _FreeReleasesShared]

# cheapest first; the exhaustive search last
PINS = [P.test_error_statuses, P.test_cow_only_copies_a_still_shared_block, P.test_full_shared_tail_opens_a_new_block,
        lambda: P.test_random_logs_invariants_and_slots(0), lambda: P.test_random_logs_invariants_and_slots(1),
        P.test_bruteforce_depth6_invariants]


def failing_pins(monkeypatch, cls):
    monkeypatch.setattr(P, "BlockManagerOracle", cls)
    failed = []
    for i, pin in enumerate(PINS):
        try:
            pin()
        except Exception:  # an assertion, or the mutant's state breaking an operation outright
            failed.append(i)
            break
    return failed


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m.__name__.lstrip("_") for m in MUTANTS])
def test_manager_pins_reject_planted_mistake(monkeypatch, mutant):
    assert failing_pins(monkeypatch, mutant), f"{mutant.__name__} passed every pin"


def test_unchanged_manager_passes_the_same_pins(monkeypatch):
    assert failing_pins(monkeypatch, BlockManagerOracle) == []
