"""Naive vs paged utilisation sweep (host only), pinned to closed forms and the manager oracle.

"Paged Attention em Large Language Models LLMs" ("Configurando as Constantes", "Cache KV Ingenuo"):
the naive allocator reserves MAX_SEQ_LEN tokens per request; the paged cache holds whole 16-token
blocks, so its waste is below one block per request; with copy-on-write prefix sharing the full
blocks of the common prompt are stored once and each request copies only the partial tail.
"""
import numpy as np
import pytest

from oracle import BlockManagerOracle
from paged_kv_cache_258_gb300 import pkv
from paged_kv_cache_258_gb300 import utilization as U


def test_constants_match_the_page():
    # 2 (K and V) x 32 layers x 32 heads x 128 dims x 2 bytes = 524,288 bytes = 512 KiB per token
    assert U.KV_BYTES_PER_TOKEN == 524288 == 512 * 1024
    assert U.PAGE == 16 and U.MAX_SEQ_LEN == 2048 and U.AVG_RESPONSE == 500


def test_sweep_closed_forms():
    sp = 200
    rows = U.sweep(seed=42, system_prompt=sp)
    assert [r["n"] for r in rows] == [10, 20, 50, 100, 200]
    for r in rows:
        lens, prompt = U.request_lengths(r["n"], 42)
        assert np.all((lens >= 65) & (lens <= U.MAX_SEQ_LEN)) and np.all(lens > prompt)
        assert r["tokens"] == int(lens.sum())
        assert r["naive_reserved"] == r["n"] * 2048
        blocks = -(-lens // 16)
        assert r["paged_reserved"] == 16 * int(blocks.sum())
        # waste below one block per request; naive wastes everything up to 2048
        assert 0 <= r["paged_reserved"] - r["tokens"] < 16 * r["n"]
        assert r["paged_util"] > 0.95 and r["naive_util"] < 0.5
        # shared: root keeps ceil(sp/16) blocks; each request shares floor(sp/16) full ones and owns
        # the rest, its copy of the partial tail included (the root stays live, so every request copies)
        ls = np.maximum(lens, sp + 1)
        want = -(-sp // 16) + int(np.sum(-(-ls // 16) - sp // 16))
        assert r["shared_blocks"] == want
        assert r["shared_cow_copies"] == (r["n"] if sp % 16 else 0)
        assert r["shared_gib"] < r["paged_gib"]


def test_utilization_monotone_in_reserved_memory():
    # the same requests at a larger MAX_SEQ_LEN only lower the naive utilisation; paged is unaffected
    lens, _ = U.request_lengths(50, 42)
    assert lens.sum() / (50 * 4096) < lens.sum() / (50 * 2048)


@pytest.mark.parametrize("n", [10, 20])
def test_shared_prefix_manager_matches_oracle(n):
    sp = 200
    lens, _ = U.request_lengths(n, 42)
    ls = np.maximum(lens, sp + 1)
    cap = 1 + int(np.sum(-(-(ls - sp + 16) // 16))) + (-(-sp // 16))
    mgr = pkv.BlockManager(cap)
    mo = BlockManagerOracle(cap)
    rc, slots = mgr.add_seq(-1, sp)
    st, slots_o = mo.add_seq(-1, sp)
    assert rc == pkv.PKV_OK and st == "ok" and list(slots) == list(slots_o)
    for i, n_tok in enumerate(ls):
        assert mgr.fork(-1, i) == pkv.PKV_OK and mo.fork(-1, i) == "ok"
        for _ in range(int(n_tok) - sp):
            rc, slot, src, dst = mgr.append_slot(i)
            s_, slot_o, src_o, dst_o = mo.append_slot(i)
            assert rc == pkv.PKV_OK and s_ == "ok"
            assert (slot, src, dst) == (slot_o, src_o, dst_o)
    assert mgr.stats() == mo.stats()
    row = U.sweep(batch_sizes=(n,), seed=42, system_prompt=sp)[0]
    assert row["shared_blocks"] == mo.stats()["used_blocks"]
