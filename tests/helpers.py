"""Test helpers: host <-> torch conversions and paged-case builders (no method arithmetic)."""
from __future__ import annotations

import numpy as np

from paged_kv_cache_258_gb300 import workloads as W

NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}
TOL = {"f32": 1e-5, "f16": 2e-2, "bf16": 2e-2}


def to_torch(a: np.ndarray, dtype: str, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t, dtype: str) -> np.ndarray:
    import torch
    if dtype == "bf16":
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def as_f64(t) -> np.ndarray:
    """A device result widened exactly to float64."""
    import torch
    return t.to(torch.float64).cpu().numpy()


def paged_case(dtype, lens, n_q, n_kv, d, seed, n_layers=1, slack=3, max_blocks=None, poison=True):
    """Host pools [L, num_blocks, n_kv, 16, d], q, shuffled tables; unused rows NaN-poisoned."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nb = -(-lens.astype(np.int64) // W.BLOCK)
    num_blocks = int(nb.sum()) + slack
    if max_blocks is None:
        max_blocks = max(1, int(nb.max()) if len(nb) else 1)
    tables = W.shuffled_tables(lens, num_blocks, seed, max_blocks=max_blocks)
    kp = W.normal_values(rng, (n_layers, num_blocks, n_kv, W.BLOCK, d), dtype)
    vp = W.normal_values(rng, (n_layers, num_blocks, n_kv, W.BLOCK, d), dtype)
    if poison:
        for layer in range(n_layers):
            W.poison_unreferenced(kp[layer], tables, lens, dtype)
            W.poison_unreferenced(vp[layer], tables, lens, dtype)
    q = W.normal_values(rng, (len(lens), n_q, d), dtype)
    return q, kp, vp, tables, lens, num_blocks
