"""Naive vs paged KV-cache utilisation at 10-200 concurrent requests (host only).

"Paged Attention em Large Language Models LLMs" ("Configurando as Constantes", "Cache KV Ingenuo")
compares a naive allocator -- every request reserves MAX_SEQ_LEN tokens up front, since its final
length is unknown -- against a paged cache with a block table and copy-on-write prefix sharing, at
10 to 200 concurrent requests, for the GPT-style model (32 layers x 32 heads x 128, fp16:
524,288 bytes per token; 16-token pages; MAX_SEQ_LEN 2048; mean response 500; seed 42). The page
is cut off before its results, so this module recomputes the comparison with this library's block
manager:

  naive   reserved tokens = N * MAX_SEQ_LEN
  paged   reserved tokens = 16 * (blocks the manager holds), every request admitted with its
          final length (prompt + response, capped at MAX_SEQ_LEN)
  shared  as paged, but all requests fork from one root holding a common system prompt, so its
          full blocks are stored once (the partial tail is copied on the first divergent write)

utilisation = tokens actually stored / tokens reserved. Request lengths follow the GPT-style
workload: prompt ~ U{64..512}, response ~ Geometric(1/500), capped at 2048.
"""
from __future__ import annotations

import numpy as np

from . import pkv

KV_BYTES_PER_TOKEN = 2 * 32 * 32 * 128 * 2  # 524,288 (the page's constant)
PAGE = 16
MAX_SEQ_LEN = 2048
AVG_RESPONSE = 500


def request_lengths(n: int, seed: int = 42):
    rng = np.random.default_rng(seed)
    prompt = rng.integers(64, 513, size=n)
    response = rng.geometric(1.0 / AVG_RESPONSE, size=n)
    return np.minimum(prompt + response, MAX_SEQ_LEN).astype(np.int64), prompt.astype(np.int64)


def sweep(batch_sizes=(10, 20, 50, 100, 200), seed: int = 42, system_prompt: int = 200):
    """Rows of {n, tokens, naive/paged/shared reserved tokens, utilisations, GiB}."""
    rows = []
    for n in batch_sizes:
        lens, _ = request_lengths(n, seed)
        tokens = int(lens.sum())
        naive = n * MAX_SEQ_LEN
        # paged: one sequence per request
        need = int(np.sum(-(-lens // PAGE)))
        mgr = pkv.BlockManager(need)
        for i, n_tok in enumerate(lens):
            rc, _ = mgr.add_seq(i, int(n_tok))
            if rc != pkv.PKV_OK:
                raise RuntimeError(f"admission failed at request {i}")
        paged_blocks = mgr.stats()["used_blocks"]
        # shared: every request = a fork of one root holding the system prompt, then its own tokens
        lens_s = np.maximum(lens, system_prompt + 1)
        cap = 1 + int(np.sum(-(-(lens_s - system_prompt + PAGE) // PAGE))) + (-(-system_prompt // PAGE))
        mgr2 = pkv.BlockManager(cap)
        rc, _ = mgr2.add_seq(-1, system_prompt)
        if rc != pkv.PKV_OK:
            raise RuntimeError("root admission failed")
        for i, n_tok in enumerate(lens_s):
            if mgr2.fork(-1, i) != pkv.PKV_OK:
                raise RuntimeError("fork failed")
            for _ in range(int(n_tok) - system_prompt):
                rc, _, _, _ = mgr2.append_slot(i)
                if rc != pkv.PKV_OK:
                    raise RuntimeError("append failed")
        shared_blocks = mgr2.stats()["used_blocks"]
        tokens_s = int(lens_s.sum())
        rows.append({
            "n": n,
            "tokens": tokens,
            "naive_reserved": naive,
            "paged_reserved": paged_blocks * PAGE,
            "naive_util": tokens / naive,
            "paged_util": tokens / (paged_blocks * PAGE),
            "naive_gib": naive * KV_BYTES_PER_TOKEN / 2 ** 30,
            "paged_gib": paged_blocks * PAGE * KV_BYTES_PER_TOKEN / 2 ** 30,
            "shared_tokens_logical": tokens_s,
            "shared_blocks": shared_blocks,
            "shared_gib": shared_blocks * PAGE * KV_BYTES_PER_TOKEN / 2 ** 30,
            "shared_cow_copies": mgr2.stats()["cow_copies"],
        })
    return rows


def main():
    print("| requests | tokens stored | naive reserved (GiB) | naive util | paged reserved (GiB) | paged util | "
          "shared-prefix (GiB, logical tokens) |")
    print("|---|---|---|---|---|---|---|")
    for r in sweep():
        print(f"| {r['n']} | {r['tokens']} | {r['naive_gib']:.1f} | {r['naive_util']:.3f} | {r['paged_gib']:.2f} | "
              f"{r['paged_util']:.4f} | {r['shared_gib']:.2f} ({r['shared_tokens_logical']}) |")


if __name__ == "__main__":
    main()
