"""Host-side validation of a step's device arguments (engine.validate_step_metadata), the stand-in
for a sanitizer on this pool: steps planned by the C block manager pass it, and each kind of bad
entry (a table id outside the pool, a length past the table, a repeated slot, a slot that is not the
sequence's last position, overlapping copy-on-write pairs) is named before anything is uploaded.
No GPU is involved.
"""
import numpy as np
import pytest

from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W
from paged_kv_cache_258_gb300.engine import validate_step_metadata


def planned_step(seed=3):
    """A decode step planned by the C manager after prefix sharing: returns tables, lens, slots, pairs."""
    nb = 64
    mgr = pkv.BlockManager(nb, free_order=W.free_order(nb, seed))
    assert mgr.add_seq(0, 37)[0] == pkv.PKV_OK
    assert mgr.add_seq(1, 100)[0] == pkv.PKV_OK
    assert mgr.fork(0, 2) == pkv.PKV_OK
    ids = [0, 1, 2]
    rc, slots, pairs, done = mgr.append_batch(ids)
    assert rc == pkv.PKV_OK and done == 3 and len(pairs) == 1  # the shared partial tail is copied once
    rc, tables, lens = mgr.pack_tables(ids, 8)
    assert rc == pkv.PKV_OK
    return nb, tables, lens, slots, pairs


def test_manager_planned_step_passes():
    nb, tables, lens, slots, pairs = planned_step()
    validate_step_metadata(nb, 16, tables, lens, slots, pairs)


@pytest.mark.parametrize("kind", ["table_id", "negative_id", "length", "dup_slot", "wrong_slot", "slot_range",
                                  "pair_overlap", "pair_dup", "pair_range"])
def test_bad_entries_are_named(kind):
    nb, tables, lens, slots, pairs = planned_step()
    tables, lens, slots, pairs = tables.copy(), lens.copy(), slots.copy(), pairs.copy()
    if kind == "table_id":
        tables[1, 2] = nb
    elif kind == "negative_id":
        tables[0, 0] = -1
    elif kind == "length":
        lens[1] = 8 * 16 + 1
    elif kind == "dup_slot":
        slots[2] = slots[0]
    elif kind == "wrong_slot":
        slots[1] += 1 if slots[1] % 16 < 15 else -1
    elif kind == "slot_range":
        slots[0] = nb * 16
    elif kind == "pair_overlap":
        pairs = np.concatenate([pairs, [[pairs[0, 1], 5]]]).astype(np.int32)
    elif kind == "pair_dup":
        pairs = np.concatenate([pairs, [[7, pairs[0, 1]]]]).astype(np.int32)
    elif kind == "pair_range":
        pairs[0, 1] = nb
    with pytest.raises(ValueError):
        validate_step_metadata(nb, 16, tables, lens, slots, pairs)


def test_negative_slots_and_empty_sequences_pass():
    nb, tables, lens, slots, pairs = planned_step()
    slots = slots.copy()
    slots[1] = -1                       # a padding token is skipped by kv_append
    validate_step_metadata(nb, 16, tables, lens, slots, pairs)
    validate_step_metadata(nb, 16, np.full((2, 4), -1, np.int32), np.zeros(2, np.int32))  # nothing used
