"""Seeded synthetic workloads for the paged KV cache.

This module holds random draws and shapes only -- none of the method's arithmetic -- so
both the CUDA path and the CPU oracle can consume the same inputs. It imports neither the
library binding nor the oracle.

Shapes follow the pages:
  * "Paged Attention em Large Language Models LLMs", "Configurando as Constantes" and
    "Cache KV Ingenuo": GPT-style 32 layers x 32 heads x head_dim 128 in fp16, blocks of 16
    tokens, MAX_SEQ_LEN 2048, mean response 500, seed 42.
  * "04 - Hacia PagedAttention (vista previa)", "Problema 3": concurrent decodes with very
    different cache lengths (200 / 1500 / 60, and 5 vs 10000-token generations).
  * "PagedAttention e continuous batching", "01 - Conceito" paragraphs 1, 3, 4: long-document
    sessions of 32,768 tokens, 16 attention layers, 64 KiB of KV per token, 1 MiB blocks.
  * same page, paragraph 6: requests with an identical prompt prefix sharing blocks.

No public dataset or benchmark is involved anywhere; every value is N(0, 1) from a seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK = 16
BASE_SEED = 42


@dataclass
class Workload:
    name: str
    dtype: str            # "f32" | "f16" | "bf16"
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    context_lens: np.ndarray           # int32 [n_seqs]
    num_blocks: int
    seed: int
    block_size: int = BLOCK
    notes: dict = field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return int(len(self.context_lens))

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    def blocks_per_seq(self) -> np.ndarray:
        return -(-self.context_lens.astype(np.int64) // self.block_size)


def _pool_size(lens: np.ndarray, slack: float = 0.125, extra_tokens_per_seq: int = 0) -> int:
    need = int(np.sum(-(-(lens.astype(np.int64) + extra_tokens_per_seq) // BLOCK)))
    return max(1, int(np.ceil(need * (1.0 + slack))))


def tiny(seed: int = BASE_SEED) -> Workload:
    """1 layer, 4 sequences {5, 17, 33, 60}, 2 heads x 64, fp32, 32 physical blocks."""
    lens = np.array([5, 17, 33, 60], dtype=np.int32)
    return Workload("tiny", "f32", 1, 2, 2, 64, lens, 32, seed)


def gpt(seed: int = BASE_SEED + 1, batch: int = 64, extra_tokens_per_seq: int = 0) -> Workload:
    """Batch-64 decode snapshot of the GPT-style model.

    prompt ~ U{64..512}, response ~ Geometric(1/500) on {1, 2, ...}, context = min(prompt +
    response, 2048). ``extra_tokens_per_seq`` sizes the pool for that many decode steps more.
    """
    rng = np.random.default_rng(seed)
    prompt = rng.integers(64, 513, size=batch)
    response = rng.geometric(1.0 / 500.0, size=batch)
    lens = np.minimum(prompt + response, 2048).astype(np.int32)
    return Workload("gpt", "f16", 32, 32, 32, 128, lens,
                    _pool_size(lens, extra_tokens_per_seq=extra_tokens_per_seq), seed)


def ragged(seed: int = BASE_SEED + 2, n_seqs: int = 32, extra_tokens_per_seq: int = 0) -> Workload:
    """32 sequences, lengths log-uniform over [5, 8192], including 60, 200 and 1500."""
    rng = np.random.default_rng(seed)
    lens = np.floor(np.exp(rng.uniform(np.log(5.0), np.log(8192.0), size=n_seqs))).astype(np.int32)
    lens[:3] = (60, 200, 1500)
    return Workload("ragged", "f16", 1, 32, 32, 128, lens,
                    _pool_size(lens, extra_tokens_per_seq=extra_tokens_per_seq), seed)


def longdoc(seed: int = BASE_SEED + 3, n_seqs: int = 10, ctx: int = 32768,
            n_layers: int = 16, extra_tokens_per_seq: int = 0) -> Workload:
    """10 sessions x 32,768 tokens; GQA 16 query / 4 KV heads x 256 in bf16; 16 layers."""
    lens = np.full(n_seqs, ctx, dtype=np.int32)
    return Workload("longdoc", "bf16", n_layers, 16, 4, 256, lens,
                    _pool_size(lens, extra_tokens_per_seq=extra_tokens_per_seq), seed)


@dataclass
class PrefixChurn:
    """Operation log of the shared-prefix churn workload.

    8 groups; group g has a root holding a prompt of 1024 + t_g tokens (t_g in [1, 15], so the
    last shared block is partially filled and the first divergent write copies it). 200 members
    fork from the roots. Each step appends one token to every live member; afterwards a seeded
    5 % of members finish and are replaced by fresh forks of a random group root.
    """
    n_groups: int
    group_prompt: list          # tokens per group root
    member_group: list          # group of each initial member (member ids 0..n-1)
    steps: list                 # per step: list of (finished_member_id, new_member_id, group)
    num_blocks: int
    seed: int


def prefix_churn(seed: int = BASE_SEED + 4, n_members: int = 200, n_groups: int = 8,
                 n_steps: int = 256, finish_frac: float = 0.05, prefix: int = 1024) -> PrefixChurn:
    rng = np.random.default_rng(seed)
    tails = 1 + rng.integers(0, 15, size=n_groups)
    group_prompt = [int(prefix + t) for t in tails]
    member_group = [int(i % n_groups) for i in range(n_members)]
    live = list(range(n_members))
    next_id = n_members
    steps = []
    n_finish = int(round(finish_frac * n_members))
    for _ in range(n_steps):
        picks = rng.choice(len(live), size=n_finish, replace=False)
        events = []
        for p in sorted(int(x) for x in picks):
            g = int(rng.integers(0, n_groups))
            events.append((live[p], next_id, g))
            live[p] = next_id
            next_id += 1
        steps.append(events)
    # blocks: shared prefixes + private growth of every member over the run + slack
    shared = sum(-(-p // BLOCK) for p in group_prompt)
    private = n_members * (-(-(n_steps + BLOCK) // BLOCK) + 1)
    num_blocks = int(np.ceil((shared + private) * 1.125))
    return PrefixChurn(n_groups, group_prompt, member_group, steps, num_blocks, seed)


def free_order(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of the physical block ids: the initial (fragmented) free list."""
    return np.random.default_rng(seed + 1000).permutation(num_blocks).astype(np.int32)


def shuffled_tables(lens, num_blocks: int, seed: int, max_blocks: int | None = None,
                    pad: int = -1) -> np.ndarray:
    """Block tables that take physical ids, in order, from a seeded permutation of the pool.

    Sequence s gets ceil(len_s / 16) distinct blocks; unused table entries hold ``pad``.
    """
    lens = np.asarray(lens, dtype=np.int64)
    nb = -(-lens // BLOCK)
    if max_blocks is None:
        max_blocks = max(1, int(nb.max()) if len(nb) else 1)
    if int(nb.sum()) > num_blocks:
        raise ValueError("pool too small for the requested contexts")
    perm = free_order(num_blocks, seed)
    tables = np.full((len(lens), max_blocks), pad, dtype=np.int32)
    off = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[off:off + n]
        off += int(n)
    return tables


def normal_values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0, 1) values as raw storage: float32, float16, or uint16 bf16 bit patterns."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        return (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 value is valid input
    raise ValueError(dtype)


def nan_value(dtype: str):
    """The NaN bit pattern used to poison rows that no table references."""
    if dtype == "f32":
        return np.float32(np.nan)
    if dtype == "f16":
        return np.float16(np.nan)
    return np.uint16(0x7FC0)


def poison_unreferenced(pool: np.ndarray, tables: np.ndarray, lens, dtype: str) -> None:
    """Set every pool row that is not a valid row of some sequence to NaN (in place).

    pool [num_blocks, n_kv, 16, d]. Valid rows are the first len_s rows of sequence s's
    logical order; everything else (unreferenced blocks, tails of last blocks) is poisoned.
    """
    num_blocks = pool.shape[0]
    valid = np.zeros((num_blocks, BLOCK), dtype=bool)
    for s, n in enumerate(np.asarray(lens, dtype=np.int64)):
        for j in range(int(n)):
            valid[tables[s, j // BLOCK], j % BLOCK] = True
    nanv = nan_value(dtype)
    for b in range(num_blocks):
        for o in range(BLOCK):
            if not valid[b, o]:
                pool[b, :, o, :] = nanv
