"""Checkpoint / resume of the C block manager (pkv_mgr_save / pkv_mgr_load), on the CPU.

A manager resumed from an image must behave exactly like the one that was saved: at random points
of seeded operation logs (adds with headroom, forks, appends with copy-on-write, multi-token
extends, frees, failures), the state is saved, loaded into a new manager, and the rest of the log
runs on the resumed manager and on the Python block-manager oracle (which never stopped): status,
slots, copy-on-write pairs, every table, every refcount, the free list in order and the counters
stay bit-identical. Malformed images (truncated, corrupted, wrong magic, a block both free and
held) are refused.
"""
import random

import pytest

from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import workloads as W
from test_manager_parity import apply_both, compare


def random_op(rng, o, next_id):
    live = list(o.tables)
    r = rng.random()
    if r < 0.12 or not live:
        return ("add", next_id, rng.randint(0, 90), rng.choice([0, 0, 16, 100])), next_id + 1
    if r < 0.22:
        return ("fork", rng.choice(live), next_id), next_id + 1
    if r < 0.78:
        return ("append", rng.choice(live + [10 ** 9])), next_id
    if r < 0.85:
        return ("extend", rng.choice(live + [10 ** 9]), rng.choice([0, 1, 5, 16, 37, 200])), next_id
    return ("free", rng.choice(live + [-5])), next_id


@pytest.mark.parametrize("seed", range(4))
def test_resume_matches_oracle(seed):
    rng = random.Random(100 + seed)
    nb = rng.choice([8, 33, 200])
    order = W.free_order(nb, seed)
    c, o = pkv.BlockManager(nb, free_order=order), BlockManagerOracle(nb, free_order=order)
    next_id = 0
    for i in range(1500):
        if i % 250 == 125:  # checkpoint and resume mid-log
            image = c.save()
            c = pkv.BlockManager.load(image)
            compare(c, o)
            assert c.save() == image  # the resumed state saves to the same bytes
        op, next_id = random_op(rng, o, next_id)
        apply_both(c, o, op)
        compare(c, o)


def test_empty_and_fresh_managers_round_trip():
    for m in (pkv.BlockManager(1), pkv.BlockManager(64, free_order=W.free_order(64, 1))):
        r = pkv.BlockManager.load(m.save())
        assert r.free_list() == m.free_list() and r.stats() == m.stats() and r.save() == m.save()


def _shared_state():
    m = pkv.BlockManager(16, free_order=W.free_order(16, 2))
    assert m.add_seq(5, 37)[0] == pkv.PKV_OK
    assert m.fork(5, 6) == pkv.PKV_OK
    assert m.append_slot(6)[0] == pkv.PKV_OK  # copy-on-write of the shared tail
    return m


def test_malformed_images_are_refused():
    image = bytearray(_shared_state().save())
    assert pkv.BlockManager.load(bytes(image)).refcounts() == _shared_state().refcounts()
    bad = []
    bad.append(bytes(image[:-1]))                      # truncated
    flip = bytearray(image)
    flip[20] ^= 1                                      # a free-list entry, checksum now wrong
    bad.append(bytes(flip))
    magic = bytearray(image)
    magic[0] ^= 0xFF                                   # wrong magic
    bad.append(bytes(magic))
    bad.append(b"")
    for img in bad:
        with pytest.raises(pkv.PkvError):
            pkv.BlockManager.load(img)


def test_inconsistent_state_is_refused_even_with_a_valid_checksum():
    """An image whose checksum is right but whose state is impossible (a block both free and held,
    a table shorter than its context) is refused: the loader re-derives the refcounts."""
    import struct
    m = _shared_state()
    image = bytearray(m.save())
    n_free = struct.unpack_from("<I", image, 16)[0]
    free0 = struct.unpack_from("<I", image, 20)[0]
    # the first sequence record follows the free list, 4 counters and the sequence count
    rec = 20 + 4 * n_free + 5 * 8
    first_block = 20 + 4 * n_free + 5 * 8 + 16
    for mutate in ("held_and_free", "short_table"):
        img = bytearray(image)
        if mutate == "held_and_free":
            struct.pack_into("<I", img, first_block, free0)         # a table now holds a free block
        else:
            ctx = struct.unpack_from("<I", img, rec + 8)[0]
            struct.pack_into("<I", img, rec + 8, ctx + 16)          # context past its blocks
        body = bytes(img[:-8])
        img[-8:] = _fnv1a64(body).to_bytes(8, "little")
        with pytest.raises(pkv.PkvError):
            pkv.BlockManager.load(bytes(img))


def _fnv1a64(data: bytes) -> int:
    h = 0xcbf29ce484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001b3) & 0xFFFFFFFFFFFFFFFF
    return h
