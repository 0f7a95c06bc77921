"""A paged KV cache on one GPU, its decode step and its chunked-prefill step, on top of the C ABI.

``PagedKVCache`` owns the all-layer K/V pools (torch device memory) and the host C block
manager. ``PrefillStep`` (at the end of this module) runs chunked prefill. ``DecodeBatch`` runs decode steps for a fixed list of sequences in the order the
method needs ("04 - Hacia PagedAttention (vista previa)", "La idea de PagedAttention", steps
3 and 5; "PagedAttention e continuous batching", "01 - Conceito", paragraph 6):

  1. host:   the block manager reserves one slot per sequence (taking a fresh block or
             copying a shared tail on write) and packs the block tables;
  2. H2D:    slots, tables, lengths and copy pairs go to the device in one upload (one pinned
             image per step, double-buffered on the host and on the device, on an upload stream:
             step i+1's upload overlaps step i's kernels). The upload is a kernel reading the
             pinned image (pkv_upload_metadata), not a copy-engine copy, so it never waits
             behind bulk host-to-device copies of other streams;
  3. device: copy-on-write block copies, then per layer the KV append and the paged decode
             attention -- copies before appends (else a copy would overwrite the new row),
             appends before attention (the new token attends to itself). By default the append
             and the attention of a layer are one kernel (pkv_paged_decode_append_attention).

All device work is in libpkv's kernels; this module only moves arguments.
"""
from __future__ import annotations

import ctypes
import os
import time

import numpy as np

from . import pkv

# PKV_CHECK=1: every planned step's metadata is validated on the host before it is uploaded (the
# kernels skip and flag bad values anyway; this names the offending entry before any launch).
CHECK_METADATA = os.environ.get("PKV_CHECK") == "1"


def validate_step_metadata(num_blocks: int, block_size: int, tables, lens, slots=None, pairs=None) -> None:
    """Host-side check of one step's device arguments; raises ValueError naming the first bad entry.

    tables [n, max_blocks] int32 and lens [n]: every block a sequence uses (the first ceil(len / 16)
    entries of its row) lies in [0, num_blocks) and len <= max_blocks * block_size; slots [n]: each in
    [0, num_blocks * block_size) or negative (skipped), no two equal, and each in the last block of its
    sequence's table at offset (len - 1) % block_size; pairs [p, 2]: source and destination ids in
    range, destinations distinct and disjoint from the sources (copy_blocks' contract).
    """
    tables = np.asarray(tables)
    lens = np.asarray(lens)
    n, mb = tables.shape
    if lens.shape != (n,):
        raise ValueError(f"lens has shape {lens.shape}, expected ({n},)")
    for s in range(n):
        ln = int(lens[s])
        if ln < 0 or ln > mb * block_size:
            raise ValueError(f"sequence {s}: length {ln} outside [0, {mb * block_size}]")
        used = tables[s, : -(-ln // block_size)]
        bad = np.nonzero((used < 0) | (used >= num_blocks))[0]
        if len(bad):
            i = int(bad[0])
            raise ValueError(f"sequence {s}: table entry {i} = {int(used[i])} outside [0, {num_blocks})")
    if slots is not None:
        slots = np.asarray(slots)
        live = slots[slots >= 0]
        if np.any(live >= num_blocks * block_size):
            raise ValueError(f"slot {int(live[live >= num_blocks * block_size][0])} beyond the pool")
        if len(np.unique(live)) != len(live):
            raise ValueError("two tokens share one slot")
        for s in range(min(n, len(slots))):
            if slots[s] < 0 or lens[s] <= 0:
                continue
            ln = int(lens[s])
            want = int(tables[s, (ln - 1) // block_size]) * block_size + (ln - 1) % block_size
            if int(slots[s]) != want:
                raise ValueError(f"sequence {s}: slot {int(slots[s])} is not position {ln - 1} of its table ({want})")
    if pairs is not None and len(pairs):
        pairs = np.asarray(pairs).reshape(-1, 2)
        if np.any((pairs < 0) | (pairs >= num_blocks)):
            raise ValueError("copy pair with a block id outside the pool")
        src, dst = set(pairs[:, 0].tolist()), pairs[:, 1].tolist()
        if len(set(dst)) != len(dst) or src & set(dst):
            raise ValueError("copy pairs: destinations repeat or overlap the sources")


class PagedKVCache:
    def __init__(self, desc: pkv.CacheDesc, free_order=None, device=None, init: str = "zeros", seed: int = 0):
        import torch
        self.desc = desc
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        dt = pkv.torch_dtype(desc.dtype_name)
        shape = pkv.pool_shape(desc)
        if init == "randn":
            g = torch.Generator(device=self.device)
            g.manual_seed(seed)
            self.k_pool = torch.randn(shape, dtype=dt, device=self.device, generator=g)
            self.v_pool = torch.randn(shape, dtype=dt, device=self.device, generator=g)
        else:
            self.k_pool = torch.zeros(shape, dtype=dt, device=self.device)
            self.v_pool = torch.zeros(shape, dtype=dt, device=self.device)
        self.mgr = pkv.BlockManager(desc.num_blocks, desc.block_size, free_order=free_order)

    def add_sequence(self, seq_id: int, n_prompt: int, reserve_tokens: int = 0) -> np.ndarray:
        rc, slots = self.mgr.add_seq(seq_id, n_prompt, reserve_tokens)
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, f"add_seq({seq_id}, {n_prompt})")
        return slots

    def fork(self, parent: int, child: int) -> None:
        rc = self.mgr.fork(parent, child)
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, f"fork({parent}, {child})")

    def free(self, seq_id: int) -> None:
        rc = self.mgr.free_seq(seq_id)
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, f"free_seq({seq_id})")

    def kv_bytes_per_token_layer(self) -> int:
        d = self.desc
        return 2 * d.n_kv_heads * d.head_dim * (4 if d.dtype_name == "f32" else 2)


class DecodeBatch:
    """Decode steps for a batch of n sequences whose tables are at most max_blocks wide."""

    def __init__(self, cache: PagedKVCache, seq_ids, max_blocks: int, stream=None, fused: bool = True):
        import torch
        self.cache = cache
        self.seq_ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        self._p_ids = self.seq_ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        self.n = len(self.seq_ids)
        self.max_blocks = int(max_blocks)
        self.stream = stream if stream is not None else torch.cuda.current_stream(cache.device)
        # fused: one kernel per layer appends the new rows and attends; else kv_append + decode
        self.fused = bool(fused)
        # overlap: each layer's fused launch may start while the previous layer's finishes
        self.overlap = True
        dev = cache.device
        n, mb = self.n, self.max_blocks
        # One int32 metadata image per step, [slots (int64) | tables | lens | CoW pairs], so the
        # upload is a single pkv_upload_metadata launch; the device image has fixed addresses across
        # steps.
        self._o_tab = 2 * n
        self._o_len = self._o_tab + n * mb
        self._o_pair = self._o_len + n
        self._meta_words = self._o_pair + 2 * max(n, 1)
        # two device copies of the image, filled on an upload stream: step i+1's metadata goes up
        # while step i's kernels run; a copy is refilled only after the kernels that read it are done
        self.up_stream = torch.cuda.Stream(dev)
        self._dev = []
        for _ in range(2):
            d_meta = torch.empty(self._meta_words, dtype=torch.int32, device=dev)
            slots, tables, lens, pairs = self._views(d_meta)
            self._dev.append(dict(meta=d_meta, slots=slots, tables=tables, lens=lens, pairs=pairs,
                                  uploaded=torch.cuda.Event(), read=torch.cuda.Event(), used=False))
        self.d_slots, self.d_tables, self.d_lens, self.d_pairs = (self._dev[0][k] for k in ("slots", "tables", "lens",
                                                                                             "pairs"))
        self.workspace = pkv.alloc_workspace(cache.desc, n, mb, device=dev)
        # two pinned staging images
        self._stage = []
        for _ in range(2):
            h_meta = torch.empty(self._meta_words, dtype=torch.int32).pin_memory()
            slots, tables, lens, pairs = self._views(h_meta)
            # numpy views of the pinned image and ctypes pointers into it, made once: planning a step
            # is two C calls writing straight into the staging image
            np_lens = lens.numpy()
            self._stage.append(dict(meta=h_meta, slots=slots, tables=tables, lens=lens, pairs=pairs,
                                    np_lens=np_lens,
                                    p_slots=slots.numpy().ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                    p_pairs=pairs.numpy().ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                    p_tables=tables.numpy().ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                    p_lens=np_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                    done=torch.cuda.Event(), used=False))
        self._turn = 0
        self.last_lens = np.zeros(n, dtype=np.int32)
        self.last_n_pairs = 0
        self.total_cow = 0
        self.manager_s = 0.0       # host time in the block manager (append + pack), waits excluded
        self.steps_planned = 0
        # validated per-layer launchers, one per device metadata image, for the step tensors they
        # were built for (kept alive here, so an identity match means the same tensors)
        self._launchers = [None, None]

    def _views(self, buf):
        n, mb = self.n, self.max_blocks
        import torch
        return (buf[: 2 * n].view(torch.int64), buf[self._o_tab: self._o_len].view(n, mb),
                buf[self._o_len: self._o_pair], buf[self._o_pair:].view(-1, 2))

    def order_longest_first(self) -> np.ndarray:
        """Reorder the batch's sequences by decreasing context length (ties keep their order) and
        return the new order (self.seq_ids). The decode grid launches its CTAs sequence by sequence
        in row order, so the longest partitions start first and the launch does not end on a long
        one that started late (measured on the ragged workload, lengths 5..8,192: 3.4 % more per
        step and per launch; on the GPT-style batch, lengths 64..2,048, 0.6 % less per step). Rows
        of q, k_new, v_new and out follow the new order."""
        rc, _, lens = self.cache.mgr.pack_tables(self.seq_ids, self.max_blocks)
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, "pack_tables")
        order = np.argsort(-lens.astype(np.int64), kind="stable")
        self.set_sequences(self.seq_ids[order])
        return self.seq_ids

    def set_sequences(self, seq_ids) -> None:
        ids = np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64))
        if len(ids) != self.n:
            raise ValueError("batch size is fixed")
        self.seq_ids = ids
        self._p_ids = ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))

    def plan(self) -> dict:
        """Host part of a step: reserve slots, collect CoW pairs, pack tables (pinned)."""
        st = self._stage[self._turn]
        st["buf"] = self._turn
        self._turn ^= 1
        if st["used"]:
            st["done"].synchronize()  # the GPU has consumed this staging set
        t0 = time.perf_counter()
        L = pkv.lib()
        h = self.cache.mgr._h
        n_cow, n_done = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = L.pkv_mgr_append_batch(h, self._p_ids, self.n, st["p_slots"], st["p_pairs"], ctypes.byref(n_cow),
                                    ctypes.byref(n_done))
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, f"append_batch stopped at sequence {int(self.seq_ids[n_done.value])}")
        npairs = int(n_cow.value)
        rc = L.pkv_mgr_pack_tables(h, self._p_ids, self.n, self.max_blocks, st["p_tables"], st["p_lens"])
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, "pack_tables (is max_blocks wide enough?)")
        st["npairs"] = npairs
        self.manager_s += time.perf_counter() - t0
        if CHECK_METADATA:
            validate_step_metadata(self.cache.desc.num_blocks, self.cache.desc.block_size, st["tables"].numpy(),
                                   st["np_lens"], st["slots"].numpy(), st["pairs"].numpy()[:npairs])
        self.steps_planned += 1
        self.last_lens = st["np_lens"].copy()
        self.last_n_pairs = npairs
        self.total_cow += npairs
        return st

    def upload(self, st: dict) -> None:
        words = self._o_pair + 2 * st["npairs"]  # only the pairs this step emitted
        dv = self._dev[st["buf"]]
        if dv["used"]:
            self.up_stream.wait_event(dv["read"])  # the kernels of two steps ago are done with it
        pkv.upload_metadata_ptr(dv["meta"].data_ptr(), st["meta"].data_ptr(), 4 * words, self.up_stream.cuda_stream)
        dv["uploaded"].record(self.up_stream)
        st["done"].record(self.up_stream)
        st["used"] = True

    def run_device(self, st: dict, q, k_new, v_new, out, scale: float, on_decode=None) -> None:
        """q/out [L, n, n_q, d]; k_new/v_new [L, n, n_kv, d] device tensors."""
        c = self.cache
        d = c.desc
        dv = self._dev[st["buf"]]
        self.stream.wait_event(dv["uploaded"])
        self.d_slots, self.d_tables, self.d_lens, self.d_pairs = dv["slots"], dv["tables"], dv["lens"], dv["pairs"]
        if st["npairs"]:
            pkv.pkv_copy_blocks(d, c.k_pool, c.v_pool, self.d_pairs[: st["npairs"]], stream=self.stream)
        if self.fused:  # the step's tensors checked once (and again only when they change); each
            # layer is then one C call
            key = (q, k_new, v_new, out, float(scale))
            hit = self._launchers[st["buf"]]
            if hit is not None and len(hit[0]) == len(key) and all(a is b for a, b in zip(hit[0][:4], key[:4])) \
                    and hit[0][4] == key[4]:
                launch = hit[1]
            else:
                launch = pkv.decode_append_launcher(d, q, k_new, v_new, c.k_pool, c.v_pool, self.d_tables,
                                                    self.d_lens, scale, out, self.workspace, stream=self.stream)
                self._launchers[st["buf"]] = (key, launch)
        for layer in range(d.n_layers):
            if on_decode is not None:
                on_decode(layer, "pre")  # before anything of this layer is launched
            if self.fused:
                if on_decode is not None:
                    on_decode(layer, "start")
                # layer l > 0 follows the previous layer's launch directly (no callback in between):
                # it may start while that one finishes (they share only the tables, lengths and the
                # workspace, which the kernel touches after the previous launch has completed)
                launch(layer, self.overlap and layer > 0 and on_decode is None)
            else:
                pkv.pkv_kv_append(d, layer, k_new[layer], v_new[layer], self.d_slots, c.k_pool, c.v_pool,
                                  stream=self.stream)
                if on_decode is not None:
                    on_decode(layer, "start")
                pkv.pkv_paged_decode_attention(d, layer, q[layer], c.k_pool, c.v_pool, self.d_tables, self.d_lens,
                                               scale, out[layer], self.workspace, stream=self.stream)
            if on_decode is not None:
                on_decode(layer, "end")
        dv["read"].record(self.stream)
        dv["used"] = True

    def step(self, q, k_new, v_new, out, scale: float, on_decode=None) -> dict:
        st = self.plan()
        self.upload(st)
        self.run_device(st, q, k_new, v_new, out, scale, on_decode)
        return st

    def kv_bytes_last_step(self) -> int:
        """Algorithmic KV bytes the last step's attention read: sum(ctx) * 2 * n_kv * d * e * L."""
        return int(self.last_lens.astype(np.int64).sum()) * self.cache.kv_bytes_per_token_layer() * \
            self.cache.desc.n_layers


class PrefillStep:
    """Chunked-prefill steps: each listed sequence gains a chunk of new tokens.

    "PagedAttention e continuous batching", "01 - Conceito", paragraph 5: long prompts are
    processed in slices so that they share steps with everyone else's decoding. One step:

      1. host:   a sequence's first chunk admits it (pkv_mgr_add_seq: blocks for the chunk
                 only); a later chunk extends it (pkv_mgr_extend, all or nothing, copying a
                 shared partial tail if there is one); the tables are packed;
      2. H2D:    slots, tables, lengths, query offsets and copy pairs in one upload (pinned,
                 double-buffered, through pkv_upload_metadata as in DecodeBatch);
      3. device: copy-on-write block copies, then the KV append of the chunk rows and the paged
                 prefill attention (the chunk attends causally to everything cached) of every
                 layer: without per-layer callbacks all appends go first and the attention
                 launches overlap (each may start while the previous layer's finishes).

    Capacity is fixed at construction: at most max_tokens chunk tokens and max_seqs sequences
    per step, tables at most max_blocks wide.
    """

    def __init__(self, cache: PagedKVCache, max_tokens: int, max_seqs: int, max_blocks: int, stream=None):
        import torch
        self.cache = cache
        self.overlap = True  # see step 3
        self.max_tokens, self.max_seqs, self.max_blocks = int(max_tokens), int(max_seqs), int(max_blocks)
        self.stream = stream if stream is not None else torch.cuda.current_stream(cache.device)
        T, S, mb = self.max_tokens, self.max_seqs, self.max_blocks
        # [slots int64 (2T words) | tables S*mb | lens S | query_start S+1 | pairs 2S]
        self._o_tab = 2 * T
        self._o_len = self._o_tab + S * mb
        self._o_qs = self._o_len + S
        self._o_pair = self._o_qs + S + 1
        self._words = self._o_pair + 2 * S
        self.d_meta = torch.empty(self._words, dtype=torch.int32, device=cache.device)
        self._stage = []
        for _ in range(2):
            h = torch.empty(self._words, dtype=torch.int32).pin_memory()
            self._stage.append(dict(meta=h, np=h.numpy(), done=torch.cuda.Event(), used=False))
        self._turn = 0
        self.manager_s = 0.0

    def _dev_views(self, n_seqs: int, n_tok: int):
        import torch
        m = self.d_meta
        S, mb = self.max_seqs, self.max_blocks
        return (m[: 2 * n_tok].view(torch.int64),
                m[self._o_tab: self._o_tab + S * mb].view(S, mb)[:n_seqs],
                m[self._o_len: self._o_len + n_seqs],
                m[self._o_qs: self._o_qs + n_seqs + 1],
                m[self._o_pair:].view(-1, 2))

    def plan(self, chunks) -> dict:
        """chunks: list of (seq_id, n_tokens, first) -- first=True admits the sequence."""
        n_seqs = len(chunks)
        n_tok = int(sum(c[1] for c in chunks))
        if n_seqs > self.max_seqs or n_tok > self.max_tokens or n_seqs == 0:
            raise ValueError("chunk set exceeds the step's capacity")
        st = self._stage[self._turn]
        self._turn ^= 1
        if st["used"]:
            st["done"].synchronize()
        t0 = time.perf_counter()
        meta = st["np"]
        slots = meta[: 2 * self.max_tokens].view(np.int64)
        qs = meta[self._o_qs: self._o_qs + n_seqs + 1]
        pairs = meta[self._o_pair:].reshape(-1, 2)
        mgr = self.cache.mgr
        npairs, pos, max_q = 0, 0, 0
        qs[0] = 0
        for i, (sid, n, first) in enumerate(chunks):
            n = int(n)
            if first:
                rc, got = mgr.add_seq(sid, n)
                if rc == pkv.PKV_OK:
                    slots[pos: pos + n] = got
                src = -1
            else:
                rc, _, src, dst = mgr.extend(sid, n, slots_out=slots[pos:])
            if rc != pkv.PKV_OK:
                raise pkv.PkvError(rc, f"prefill chunk of sequence {sid} ({n} tokens)")
            if src >= 0:
                pairs[npairs] = (src, dst)
                npairs += 1
            pos += n
            qs[i + 1] = pos
            max_q = max(max_q, n)
        ids = np.ascontiguousarray([c[0] for c in chunks], dtype=np.int64)
        tables = meta[self._o_tab: self._o_tab + n_seqs * self.max_blocks]
        lens = meta[self._o_len: self._o_len + n_seqs]
        rc, _, _ = mgr.pack_tables(ids, self.max_blocks, tables, lens)
        if rc != pkv.PKV_OK:
            raise pkv.PkvError(rc, "pack_tables (is max_blocks wide enough?)")
        self.manager_s += time.perf_counter() - t0
        st.update(n_seqs=n_seqs, n_tok=n_tok, npairs=npairs, max_q=max_q, lens=lens.copy(), qs=qs.copy())
        return st

    def upload(self, st: dict) -> None:
        pkv.upload_metadata_ptr(self.d_meta.data_ptr(), st["meta"].data_ptr(), 4 * self._words, self.stream.cuda_stream)
        st["done"].record(self.stream)
        st["used"] = True

    def run_device(self, st: dict, q, k_new, v_new, out, scale: float, on_attn=None) -> None:
        """q/out [L, T, n_q, d], k_new/v_new [L, T, n_kv, d] (T = the step's chunk tokens)."""
        c = self.cache
        d = c.desc
        slots, tables, lens, qs, pairs = self._dev_views(st["n_seqs"], st["n_tok"])
        if st["npairs"]:
            pkv.pkv_copy_blocks(d, c.k_pool, c.v_pool, pairs[: st["npairs"]], stream=self.stream)
        append = pkv.append_launcher(d, k_new, v_new, slots, c.k_pool, c.v_pool, stream=self.stream)
        attend = pkv.prefill_launcher(d, q, c.k_pool, c.v_pool, tables, lens, qs, st["max_q"], scale, out,
                                      stream=self.stream)
        if on_attn is None and self.overlap:
            # every layer's rows first, then the attention launches back to back: layer l > 0 may
            # start while layer l-1 finishes (it reads only what the appends above wrote), filling
            # the SMs the previous launch's last wave leaves idle
            for layer in range(d.n_layers):
                append(layer)
            for layer in range(d.n_layers):
                attend(layer, layer > 0)
            return
        for layer in range(d.n_layers):
            if on_attn is not None:
                on_attn(layer, "pre")  # before anything of this layer is launched
            append(layer)
            if on_attn is not None:
                on_attn(layer, "start")
            attend(layer)
            if on_attn is not None:
                on_attn(layer, "end")

    def step(self, chunks, q, k_new, v_new, out, scale: float, on_attn=None) -> dict:
        st = self.plan(chunks)
        self.upload(st)
        self.run_device(st, q, k_new, v_new, out, scale, on_attn)
        return st

    @staticmethod
    def attention_flops(st: dict, n_q: int, head_dim: int) -> float:
        """Causal attention flops of one layer: 4 * d * n_q * sum over chunk tokens of (position + 1)."""
        total = 0.0
        for s in range(st["n_seqs"]):
            n = int(st["qs"][s + 1] - st["qs"][s])
            c = int(st["lens"][s])
            # positions c-n .. c-1 see c-n+1 .. c keys
            total += n * (c - n) + n * (n + 1) / 2
        return 4.0 * head_dim * n_q * total


class StepExecutor:
    """Runs one continuous-batching iteration planned by scheduler.Scheduler on the device.

    The plan arrives complete (slots, tables, lengths, query offsets, copy pairs: every manager
    call has been made on the host). One packed metadata image goes up in one upload
    (pkv_upload_metadata); then the
    copy-on-write block copies, and per layer the chunk rows' append + paged prefill attention for
    the prefilling sequences and the fused append + paged decode attention for the decoding ones.
    Without per-kernel callbacks the chunk appends of every layer go first and the attention
    launches follow each other as programmatic dependents (see _run_overlapped).
    Capacities (decoders, chunk tokens, chunks, copy pairs per iteration; table width) are fixed
    at construction.
    """

    def __init__(self, cache: PagedKVCache, max_decode: int, max_tokens: int, max_chunks: int, max_blocks: int,
                 max_pairs: int | None = None, stream=None):
        import torch
        self.cache = cache
        self.D, self.T, self.S, self.mb = int(max_decode), int(max_tokens), int(max_chunks), int(max_blocks)
        self.P = int(max_pairs) if max_pairs is not None else self.D + self.S
        self.stream = stream if stream is not None else torch.cuda.current_stream(cache.device)
        self.overlap = True  # without callbacks, an iteration's launches follow each other as dependents
        D, T, S, mb, P = self.D, self.T, self.S, self.mb, self.P
        o = {}
        off = 0
        for name, words in (("dec_slots", 2 * D), ("pre_slots", 2 * T), ("dec_tables", D * mb), ("dec_lens", D),
                            ("pre_tables", S * mb), ("pre_lens", S), ("pre_qs", S + 1), ("pairs", 2 * P)):
            o[name] = (off, words)
            off += words + (words & 1)          # keep int64 fields 8-byte aligned
        self._off, self._words = o, off
        self.d_meta = torch.empty(off, dtype=torch.int32, device=cache.device)
        self._stage = []
        for _ in range(2):
            h = torch.empty(off, dtype=torch.int32).pin_memory()
            self._stage.append(dict(meta=h, np=h.numpy(), done=torch.cuda.Event(), used=False))
        self._turn = 0
        self.workspace = pkv.alloc_workspace(cache.desc, max(D, 1), mb, device=cache.device)

    def _host(self, np_meta, name, dtype=np.int32):
        off, words = self._off[name]
        v = np_meta[off: off + words]
        return v.view(np.int64) if dtype == np.int64 else v

    def _dev(self, name, n=None, shape=None, i64=False):
        import torch
        off, words = self._off[name]
        v = self.d_meta[off: off + words]
        if i64:
            v = v.view(torch.int64)
        if n is not None:
            v = v[:n]
        if shape is not None:
            v = v.view(*shape)
        return v

    def upload(self, plan) -> dict:
        n_dec, n_pre, n_tok, n_pairs = plan.n_dec, len(plan.pre_chunks), plan.n_pre_tokens, len(plan.pairs)
        if n_dec > self.D or n_tok > self.T or n_pre > self.S or n_pairs > self.P:
            raise ValueError("iteration exceeds the executor's capacity")
        st = self._stage[self._turn]
        self._turn ^= 1
        if st["used"]:
            st["done"].synchronize()
        m = st["np"]
        self._host(m, "dec_slots", np.int64)[:n_dec] = plan.dec_slots
        self._host(m, "pre_slots", np.int64)[:n_tok] = plan.pre_slots
        wd, wp = int(plan.dec_tables.shape[1]), int(plan.pre_tables.shape[1])
        if wd > self.mb or wp > self.mb:
            raise ValueError("plan tables wider than the executor's max_blocks")
        self._host(m, "dec_tables")[: n_dec * wd] = plan.dec_tables.reshape(-1)
        self._host(m, "dec_lens")[:n_dec] = plan.dec_lens
        self._host(m, "pre_tables")[: n_pre * wp] = plan.pre_tables.reshape(-1)
        self._host(m, "pre_lens")[:n_pre] = plan.pre_lens
        self._host(m, "pre_qs")[: n_pre + 1] = plan.pre_qs
        self._host(m, "pairs")[: 2 * n_pairs] = plan.pairs.reshape(-1)
        pkv.upload_metadata_ptr(self.d_meta.data_ptr(), st["meta"].data_ptr(),
                                self.d_meta.numel() * 4, self.stream.cuda_stream)
        st["done"].record(self.stream)
        st["used"] = True
        return dict(n_dec=n_dec, n_pre=n_pre, n_tok=n_tok, n_pairs=n_pairs, wd=wd, wp=wp,
                    max_q=max([n for _, n in plan.pre_chunks], default=0))

    def run(self, plan, dec_io, pre_io, scale: float, on_kernel=None) -> dict:
        """dec_io = (q [L, n_dec, n_q, d], k, v [L, n_dec, n_kv, d], out like q); pre_io the same with
        the iteration's chunk tokens in place of n_dec. Views of larger resident buffers are fine."""
        c = self.cache
        d = c.desc
        u = self.upload(plan)
        if u["n_pairs"]:
            pkv.pkv_copy_blocks(d, c.k_pool, c.v_pool, self._dev("pairs", 2 * u["n_pairs"], (-1, 2)),
                                stream=self.stream)
        append, attend, decode = self._launchers(u, dec_io, pre_io, scale)
        if on_kernel is None and self.overlap:
            self._run_overlapped(u, append, attend, decode)
            return u
        for layer in range(d.n_layers):
            if u["n_pre"]:
                append(layer)
                if on_kernel is not None:
                    on_kernel("prefill", layer, "start")
                attend(layer)
                if on_kernel is not None:
                    on_kernel("prefill", layer, "end")
            if u["n_dec"]:
                if on_kernel is not None:
                    on_kernel("decode", layer, "start")
                decode(layer)
                if on_kernel is not None:
                    on_kernel("decode", layer, "end")
        return u

    def _launchers(self, u, dec_io, pre_io, scale: float):
        """The iteration's per-layer launches (None where it has no such work), tensors checked once."""
        c = self.cache
        d = c.desc
        append = attend = decode = None
        if u["n_pre"]:
            q, k, v, out = pre_io
            append = pkv.append_launcher(d, k, v, self._dev("pre_slots", u["n_tok"], i64=True), c.k_pool, c.v_pool,
                                         stream=self.stream)
            attend = pkv.prefill_launcher(
                d, q, c.k_pool, c.v_pool, self._dev("pre_tables", u["n_pre"] * u["wp"], (-1, u["wp"])),
                self._dev("pre_lens", u["n_pre"]), self._dev("pre_qs", u["n_pre"] + 1), u["max_q"], scale, out,
                stream=self.stream)
        if u["n_dec"]:
            q, k, v, out = dec_io
            decode = pkv.decode_append_launcher(
                d, q, k, v, c.k_pool, c.v_pool, self._dev("dec_tables", u["n_dec"] * u["wd"], (-1, u["wd"])),
                self._dev("dec_lens", u["n_dec"]), scale, out, self.workspace, stream=self.stream)
        return append, attend, decode

    def _run_overlapped(self, u, append, attend, decode) -> None:
        """The iteration's chunk rows of every layer first, then per layer the prefill and the decode
        launch, each (after the first) a programmatic dependent of the one before: a launch reads
        only what the appends and copies above wrote (a decode sequence appends into its own last
        block, which no prefill reads), and touches its outputs and the decode workspace only after
        the previous launch has completed."""
        n_layers = self.cache.desc.n_layers
        if append is not None:
            for layer in range(n_layers):
                append(layer)
        first = True
        for layer in range(n_layers):
            if attend is not None:
                attend(layer, not first)
                first = False
            if decode is not None:
                decode(layer, not first)
                first = False


class StepCopyPipeline:
    """Whole-step host <-> device copies overlapped with other steps' kernels.

    Two device buffer sets alternate between steps: step i's inputs go up (on an upload stream)
    into one set while step i-1's kernels run on the other, and step i's outputs come down (on a
    download stream) while step i+1 runs. Nothing is recorded between a step's layer launches, so
    DecodeBatch can launch them back to back as programmatic dependents. Protocol per step:
    ``dev = upload(host_inputs)`` (may be issued while the previous step runs), ``begin()``, the
    step's kernels on ``compute_stream`` using ``dev``, ``end(host_outputs)``; ``finish()`` makes
    the compute stream wait until the last outputs are on the host.
    """

    def __init__(self, compute_stream, device, make_set):
        import torch
        self.compute = compute_stream
        self.sets = [make_set(), make_set()]  # dicts of device tensors, inputs and outputs
        self.h2d = torch.cuda.Stream(device)
        self.d2h = torch.cuda.Stream(device)
        self.uploaded = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.downloaded = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]
        self.next = 0  # the set the next upload fills
        self.cur = None

    def upload(self, host_inputs: dict) -> dict:
        """Queue the copies of one step's inputs (name -> pinned host tensor) into the next set."""
        import torch
        k = self.next
        dev = self.sets[k]
        with torch.cuda.stream(self.h2d):
            if self.used[k]:
                self.h2d.wait_event(self.done[k])  # the kernels of two steps ago are done with it
            for name, host in host_inputs.items():
                dev[name].copy_(host, non_blocking=True)
            self.uploaded[k].record(self.h2d)
        self.next ^= 1
        return dev

    def begin(self) -> dict:
        """The compute stream waits for the current set's inputs and for the download of its outputs
        from two steps ago; returns the set."""
        k = self.next ^ 1
        self.cur = k
        self.compute.wait_event(self.uploaded[k])
        if self.used[k]:
            self.compute.wait_event(self.downloaded[k])
        return self.sets[k]

    def end(self, host_outputs: dict) -> None:
        """Queue the copies of the step's outputs (name -> pinned host tensor) after its kernels."""
        import torch
        k = self.cur
        self.done[k].record(self.compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.done[k])
            for name, host in host_outputs.items():
                host.copy_(self.sets[k][name], non_blocking=True)
            self.downloaded[k].record(self.d2h)
        self.used[k] = True

    def finish(self) -> None:
        if self.cur is not None:
            self.compute.wait_event(self.downloaded[self.cur])
