"""Block-manager oracle -- TEST INFRASTRUCTURE, not part of the product.

A plain Python restatement of the paged KV cache's host-side bookkeeping. Only tests/,
``__graft_entry__.smoke()`` and bench.py's cpu_baseline leg may import it. It shares no
code with the C block manager in the library; the two are compared operation by operation.

What it restates:
  * "04 - Hacia PagedAttention (vista previa)", section "La idea de PagedAttention":
      step 1  fixed blocks of ``block_size`` tokens (16 in every configuration here);
      step 2  one block table per sequence: logical block i -> physical block X;
      step 3  to extend a sequence by one token, write into the last block if it has room,
              otherwise take a new physical block and append it to the table;
      step 4  freeing a sequence returns its physical blocks to a free list.
    "Propiedades": every sequence wastes at most block_size - 1 rows of its last block;
    free blocks are interchangeable; sequences with the same prompt share initial blocks
    through reference counts.
  * "PagedAttention e continuous batching", section "01 - Conceito":
      paragraph 6  shared read-only blocks; copy-on-write allocates a new block when a
                   branch diverges; reference counts decide when a block returns to the pool;
      paragraph 7  admission reasons in countable blocks and refuses early with a clear error;
      paragraph 8  block metrics: free and used blocks, allocation failures, tail waste,
                   prefix hits, preemptions.

Readings taken where the pages are silent (listed in the design notes):
  * the free list is FIFO: allocation pops the front, release pushes to the back, and a
    freed sequence releases its blocks in ascending logical order;
  * slot of a token = physical block * block_size + (position mod block_size);
  * copy-on-write triggers only when the token goes into a partially filled last block
    whose reference count is above 1; a full shared last block is never copied (the new
    token opens a fresh block instead);
  * admission of a new sequence needs ceil(n_prompt / block_size) +
    ceil(reserve_tokens / block_size) free blocks; only the prompt blocks are taken;
  * an append that finds no free block fails with "no_blocks" and counts one append OOM
    (the signal a scheduler would preempt on);
  * every failed operation leaves the state unchanged.

Statuses are plain strings: "ok", "invalid", "no_blocks".
"""
from __future__ import annotations

from collections import deque


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool shape")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.ctx: dict[int, int] = {}
        self.alloc_failures = 0
        self.prefix_hits = 0
        self.cow_copies = 0
        self.append_oom = 0

    # -- helpers -----------------------------------------------------------------------
    def _blocks_for(self, n_tokens: int) -> int:
        return -(-n_tokens // self.block_size)

    def _slot(self, block: int, position: int) -> int:
        return block * self.block_size + position % self.block_size

    # -- operations --------------------------------------------------------------------
    def add_seq(self, seq_id: int, n_prompt: int, reserve_tokens: int = 0):
        """Admit a sequence with n_prompt tokens. Returns (status, slots)."""
        if seq_id in self.tables or n_prompt < 0 or reserve_tokens < 0:
            return "invalid", []
        need = self._blocks_for(n_prompt)
        if need + self._blocks_for(reserve_tokens) > len(self.free):
            self.alloc_failures += 1
            return "no_blocks", []
        table = [self.free.popleft() for _ in range(need)]
        for b in table:
            self.ref[b] = 1
        self.tables[seq_id] = table
        self.ctx[seq_id] = n_prompt
        return "ok", [self._slot(table[p // self.block_size], p) for p in range(n_prompt)]

    def fork(self, parent: int, child: int):
        """child starts as a copy of parent's table; every shared block gains a reference."""
        if parent not in self.tables or child in self.tables or parent == child:
            return "invalid"
        table = list(self.tables[parent])
        for b in table:
            self.ref[b] += 1
        self.tables[child] = table
        self.ctx[child] = self.ctx[parent]
        self.prefix_hits += len(table)
        return "ok"

    def append_slot(self, seq_id: int):
        """Reserve the slot of one new token. Returns (status, slot, cow_src, cow_dst)."""
        if seq_id not in self.tables:
            return "invalid", -1, -1, -1
        table = self.tables[seq_id]
        n = self.ctx[seq_id]
        if n % self.block_size == 0:
            # the last block is full (or there is none): take a fresh block
            if not self.free:
                self.alloc_failures += 1
                self.append_oom += 1
                return "no_blocks", -1, -1, -1
            b = self.free.popleft()
            self.ref[b] = 1
            table.append(b)
            self.ctx[seq_id] = n + 1
            return "ok", self._slot(b, n), -1, -1
        tail = table[-1]
        if self.ref[tail] == 1:
            self.ctx[seq_id] = n + 1
            return "ok", self._slot(tail, n), -1, -1
        # partially filled tail shared with another sequence: copy on write
        if not self.free:
            self.alloc_failures += 1
            self.append_oom += 1
            return "no_blocks", -1, -1, -1
        b = self.free.popleft()
        self.ref[b] = 1
        self.ref[tail] -= 1
        table[-1] = b
        self.ctx[seq_id] = n + 1
        self.cow_copies += 1
        return "ok", self._slot(b, n), tail, b

    def extend(self, seq_id: int, n_tokens: int):
        """Extend a sequence by n_tokens at once (one prefill chunk), all or nothing.

        "01 - Conceito" paragraph 5 slices long prompts into chunks. Reading: a chunk succeeds
        only if the pool holds every block it needs (one more when the first token must copy a
        shared partial tail); it is then exactly n_tokens appends of step 3. A failing chunk
        counts one allocation failure and one append OOM and changes nothing.
        Returns (status, slots, cow_src, cow_dst).
        """
        if seq_id not in self.tables or n_tokens < 0:
            return "invalid", [], -1, -1
        if n_tokens == 0:
            return "ok", [], -1, -1
        table, n = self.tables[seq_id], self.ctx[seq_id]
        cow = n % self.block_size != 0 and self.ref[table[-1]] > 1
        need = self._blocks_for(n + n_tokens) - len(table) + (1 if cow else 0)
        if need > len(self.free):
            self.alloc_failures += 1
            self.append_oom += 1
            return "no_blocks", [], -1, -1
        slots, src, dst = [], -1, -1
        for i in range(n_tokens):
            st, slot, s_, d_ = self.append_slot(seq_id)
            assert st == "ok"
            slots.append(slot)
            if s_ >= 0:
                src, dst = s_, d_
        return "ok", slots, src, dst

    def free_seq(self, seq_id: int):
        if seq_id not in self.tables:
            return "invalid"
        for b in self.tables.pop(seq_id):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.ctx[seq_id]
        return "ok"

    # -- queries -----------------------------------------------------------------------
    def block_table(self, seq_id: int):
        return list(self.tables[seq_id]), self.ctx[seq_id]

    def free_list(self):
        return list(self.free)

    def refcounts(self):
        return list(self.ref)

    def tail_waste_rows(self) -> int:
        return sum(len(t) * self.block_size - self.ctx[s] for s, t in self.tables.items())

    def stats(self) -> dict:
        return {
            "free_blocks": len(self.free),
            "used_blocks": self.num_blocks - len(self.free),
            "n_seqs": len(self.tables),
            "alloc_failures": self.alloc_failures,
            "tail_waste_rows": self.tail_waste_rows(),
            "prefix_hits": self.prefix_hits,
            "cow_copies": self.cow_copies,
            "append_oom": self.append_oom,
        }
