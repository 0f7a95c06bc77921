"""Benchmark: paged decode attention on one GB300 (KV GB/s, decode tokens/s, % of HBM roofline).

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--config gpt|ragged|longdoc|prefix|prefill30k|serve|appendcopy] [--impl pkv|reference]

A step is one decode step of the whole hot path over one batch: the host block manager
reserves a slot per sequence (copy-on-write pairs included), the metadata goes to the device,
then copy_blocks, and per layer kv_append + paged decode attention. ``value`` is the KV bytes
the attention read per step (sum of context lengths x 2 x n_kv x head_dim x bytes x layers)
divided by the step time, with the step's inputs already in HBM; ``e2e`` is the same metric
with the per-step inputs (q, new K/V rows for every layer) copied from pinned host memory and
the outputs copied back inside the timed region.

The default run (--config gpt) measures the GPT-style batch for the line itself, then the
long-document, ragged and shared-prefix workloads at full size, each under "configs" with its
own value, per-launch roofline, e2e, clocks and cpu_baseline (--no-sub-configs skips them).
Every decode line also carries the read-only HBM bandwidth of the GPU ("read_peak": the library's
streaming-read probe over 4 GiB) and the fractions of it, beside the copy bandwidth.

--config prefill30k prints the chunked-prefill line instead: one 30,000-token prompt of the
long-document model prefilled in chunks of whole waves of the prefill grid (the number of waves
closest to 2,048 tokens: 2,432 on a GB300), ``value`` = causal attention TFLOP/s.
--config appendcopy times the two copy kernels of the path alone: per step one copy_blocks of 200
copy-on-write pairs over all layers and one kv_append per layer for a batch of 64 tokens;
``value`` = bytes read + written per step / step time.

Every input is synthetic and seeded (see paged_kv_cache_258_gb300/workloads.py). Multi-GPU
(torchrun) runs one independent replica per rank (weak scaling: sequences shard across ranks
with no data-path collective); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

from paged_kv_cache_258_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s & tokens/s at 1 GB300; % of HBM roofline"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------------------------
# distributed helpers (host logic; tested with gloo ranks on the CPU)

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_over_ranks(x: float, op: str, device=None) -> float:
    """max or sum of a float over ranks (identity on one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.15)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
                pw.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(device_index)


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return json.loads(p.read_text())
        except ValueError:
            pass
    return {}


# ---------------------------------------------------------------------------------------------
# workloads

def build_workload(name: str, warmup: int, steps: int, seed_offset: int = 0, layers: int | None = None):
    """(workload, description, churn log or None). ``layers`` overrides the layer count only
    (every layer's launch is identical, so a 2-layer case profiles the same kernel launch)."""
    wl, desc, churn = _build_workload(name, warmup, steps, seed_offset)
    if layers is not None and layers != wl.n_layers:
        wl.n_layers = int(layers)
        desc += f" [reduced to {layers} layers]"
    return wl, desc, churn


def _build_workload(name: str, warmup: int, steps: int, seed_offset: int = 0):
    extra = warmup + 3 * steps + 2 * W.BLOCK  # warm-up, the value pass, the roofline pass, e2e
    if name == "gpt":
        wl = W.gpt(seed=W.BASE_SEED + 1 + seed_offset, extra_tokens_per_seq=extra)
        desc = "gpt: 32 layers x 32 heads x head_dim 128 fp16 (512 KiB/token), batch 64, block 16, " \
               "ctx = min(U{64..512} + Geom(1/500), 2048)"
    elif name == "ragged":
        wl = W.ragged(seed=W.BASE_SEED + 2 + seed_offset, extra_tokens_per_seq=extra)
        desc = "ragged: 1 layer, 32 heads x head_dim 128 fp16, 32 sequences, ctx log-uniform [5, 8192] incl. " \
               "60/200/1500, block 16, shuffled free list"
    elif name == "longdoc":
        wl = W.longdoc(seed=W.BASE_SEED + 3 + seed_offset, extra_tokens_per_seq=extra)
        desc = "longdoc: 16 layers, GQA 16 q / 4 kv heads x head_dim 256 bf16 (64 KiB/token), " \
               "10 sequences x 32,768 tokens, block 16, split-K"
    elif name == "prefix":
        churn = W.prefix_churn(seed=W.BASE_SEED + 4 + seed_offset)
        wl = W.Workload("prefix", "f16", 1, 32, 32, 128, np.zeros(200, dtype=np.int32), churn.num_blocks,
                        churn.seed)
        desc = "prefix: 1 layer, 32 heads x head_dim 128 fp16, 200 sequences forked from 8 roots sharing a " \
               "1024+t token prompt, 1 token/sequence/step, 5% replaced per step, CoW on first divergent write"
        return wl, desc, churn
    else:
        raise ValueError(name)
    return wl, desc, None


# Workloads whose batch the engine orders longest first (row order is the engine's choice; q and
# out are synthetic): the ragged mix (5 .. 8,192 tokens) gains 3.4 % per step and per launch when its
# longest partitions start first; the GPT-style mix loses 0.6 % per step, so it keeps its order.
ORDER_LONGEST_FIRST = ("ragged",)


def setup_gpu_case(name: str, warmup: int, steps: int, device, seed_offset: int = 0, layers: int | None = None,
                   placement: str = "shuffled"):
    import torch
    from paged_kv_cache_258_gb300 import pkv
    from paged_kv_cache_258_gb300.engine import DecodeBatch, PagedKVCache

    wl, wdesc, churn = build_workload(name, warmup, steps, seed_offset, layers)
    desc = pkv.make_desc(wl.dtype, wl.n_layers, wl.num_blocks, wl.n_q_heads, wl.n_kv_heads, wl.head_dim)
    # shuffled: the free list is a seeded permutation, so a sequence's blocks lie anywhere in the pool;
    # contiguous: blocks are handed out in id order, so each sequence's blocks are adjacent
    order = W.free_order(wl.num_blocks, wl.seed) if placement == "shuffled" else None
    cache = PagedKVCache(desc, free_order=order, device=device, init="randn",
                         seed=wl.seed)
    extra = warmup + 3 * steps + 2 * W.BLOCK  # warm-up, the value pass, the roofline pass, e2e
    if churn is None:
        for s, n in enumerate(wl.context_lens):
            cache.add_sequence(s, int(n) - 1)   # the first step appends the token that makes ctx
        ids = list(range(wl.n_seqs))
        max_blocks = int(-(-(int(wl.context_lens.max()) + extra) // W.BLOCK))
    else:
        roots = [10 ** 6 + g for g in range(churn.n_groups)]
        for g, r in enumerate(roots):
            cache.add_sequence(r, churn.group_prompt[g])
        for m, g in enumerate(churn.member_group):
            cache.fork(roots[churn.member_group[m]], m)
        ids = list(range(len(churn.member_group)))
        max_blocks = int(-(-(max(churn.group_prompt) + extra) // W.BLOCK))
    batch = DecodeBatch(cache, ids, max_blocks)
    if churn is None and name in ORDER_LONGEST_FIRST:
        ids = [int(x) for x in batch.order_longest_first()]
    n = len(ids)
    dt = pkv.torch_dtype(wl.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + 7)
    L = wl.n_layers
    q = torch.randn((L, n, wl.n_q_heads, wl.head_dim), dtype=dt, device=device, generator=g)
    k_new = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), dtype=dt, device=device, generator=g)
    v_new = torch.randn((L, n, wl.n_kv_heads, wl.head_dim), dtype=dt, device=device, generator=g)
    out = torch.empty_like(q)
    state = {"churn": churn, "step": 0, "live": list(ids), "roots": [10 ** 6 + i for i in range(8)]}
    return wl, wdesc, cache, batch, (q, k_new, v_new, out), state


def apply_churn(cache, batch, state):
    churn = state["churn"]
    if churn is None or state["step"] >= len(churn.steps):
        state["step"] += 1
        return
    live = state["live"]
    for old, new, g in churn.steps[state["step"]]:
        cache.free(old)
        cache.fork(state["roots"][g], new)
        live[live.index(old)] = new
    batch.set_sequences(live)
    state["step"] += 1


# ---------------------------------------------------------------------------------------------
# GPU arm

def measure_read_peak(device, gib: float = 4.0, repeats: int = 10) -> dict:
    """Read-only HBM bandwidth of this GPU: the library's streaming-read probe over a buffer far
    larger than L2, timed with CUDA events launch by launch; best and median of the repeats."""
    import torch
    from paged_kv_cache_258_gb300 import pkv
    n = int(gib * 2 ** 30) // 4
    buf = torch.ones(n, dtype=torch.int32, device=device)
    fold = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        pkv.pkv_hbm_read_probe(buf, fold, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(repeats)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        pkv.pkv_hbm_read_probe(buf, fold, stream)
        b.record(stream)
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    nbytes = n * 4
    del buf
    torch.cuda.empty_cache()
    return {"best_gbs": round(nbytes / (ms[0] * 1e-3) / 1e9, 1),
            "median_gbs": round(nbytes / (ms[len(ms) // 2] * 1e-3) / 1e9, 1),
            "bytes": nbytes, "repeats": repeats,
            "how": f"pkv_hbm_read_probe: one coalesced 16-byte streaming load per word of a {gib:g} GiB buffer, "
                   f"CUDA events per launch"}


def measure_decode(args, config: str, device, rank: int, ws: int, read_peak: dict | None,
                   cpu: bool, cpu_budget: float) -> dict:
    """One decode workload at full size on this rank: the value pass (steps alone), the roofline
    pass (an event pair around every decode launch), the e2e pass, and on rank 0 of one GPU the
    oracle's cpu baseline. Returns the measurements; the pools are released when it returns."""
    import torch
    from paged_kv_cache_258_gb300 import pkv

    wl, wdesc, cache, batch, (q, k_new, v_new, out), state = setup_gpu_case(
        config, args.warmup, args.steps, device, seed_offset=rank, layers=args.layers,
        placement=args.placement)
    stream = batch.stream
    scale = wl.scale

    for _ in range(args.warmup):
        batch.step(q, k_new, v_new, out, scale)
        apply_churn(cache, batch, state)
    flags = pkv.pkv_get_device_status(stream)
    if flags:
        raise RuntimeError(f"device status flags {flags} during warm-up ({config})")

    # ---- timed region: inputs resident in HBM ----
    L = wl.n_layers
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps * L)]
    layer_bytes = []
    cursor = {"i": 0}

    def on_decode(layer, when):
        if when == "pre":
            return
        e = ev_pairs[cursor["i"]]
        if when == "start":
            e[0].record(stream)
        else:
            e[1].record(stream)
            cursor["i"] += 1

    sampler = ClockSampler(gpu_uuid(device.index))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = pkv.pkv_launch_count()
    kv_bytes = 0
    cow_pairs = 0
    t0.record(stream)
    for _ in range(args.steps):  # value: the steps alone (a timing event per launch would add a gap)
        st = batch.plan()
        batch.upload(st)
        batch.run_device(st, q, k_new, v_new, out, scale)
        kv_bytes += batch.kv_bytes_last_step()
        cow_pairs += st["npairs"]
        apply_churn(cache, batch, state)
    t1.record(stream)
    for _ in range(args.steps):  # roofline: the same steps again, each decode launch between two events
        st = batch.plan()
        batch.upload(st)
        batch.run_device(st, q, k_new, v_new, out, scale, on_decode)
        b = batch.kv_bytes_last_step()
        layer_bytes.extend([b // L] * L)
        apply_churn(cache, batch, state)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = (pkv.pkv_launch_count() - launches0) // 2  # per pass
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = reduce_over_ranks(elapsed_ms, "max", device)
    total_bytes = reduce_over_ranks(kv_bytes, "sum", device)
    total_seqs = reduce_over_ranks(batch.n * args.steps, "sum", device)
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError(f"device status flags set during the timed region ({config})")

    durs = [a.elapsed_time(b) for a, b in ev_pairs]
    achieved_gbs = sum(layer_bytes) / (sum(durs) * 1e-3) / 1e9

    # ---- e2e: per-step inputs from pinned host memory, outputs back to pinned host memory ----
    e2e = run_e2e(args, batch, cache, state, (q, k_new, v_new, out), scale, device)

    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    value = total_bytes / (elapsed_ms * 1e-3) / 1e9
    res = {
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(elapsed_ms / args.steps, 4),
        "dtype": wl.dtype,  # the operands of the QK^T and PV products (fp32 storage runs on CUDA cores)
        "config": {
            "workload": wdesc,
            "kv_dtype": wl.dtype,
            "n_seqs_per_gpu": batch.n,
            "layers": L,
            "q_heads": wl.n_q_heads,
            "kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim,
            "block_size": W.BLOCK,
            "kv_gib_per_step": round(kv_bytes / args.steps / 2 ** 30, 3),
            "l2": "no flush: every step reads more KV than the 129 MB L2 holds",
            "parallelism": f"replicas x{ws} (sequences shard by rank, no collective)",
            "placement": args.placement,
        },
        "tokens_per_s": round(total_seqs / (elapsed_ms * 1e-3), 1),
        "hbm_frac_of_measured": round(value / hbm_peak, 4),
        "hbm_frac_of_nominal_7900": round(value / NOMINAL_HBM_GBS, 4),
        "roofline": {
            "kernel": ("paged_decode_mma_kernel" if wl.dtype != "f32" else "paged_decode_kernel")
                      + " (split-K partitions merged inside the same launch)",
            "bound": "hbm",
            "achieved": round(achieved_gbs, 2),
            "peak": hbm_peak,
            "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)",
            "unit": "GB/s",
            "frac": round(achieved_gbs / hbm_peak, 4),
            "traffic": traffic_per_launch(config, sum(layer_bytes) / len(layer_bytes)),
            "launch_ms_mean": round(sum(durs) / len(durs), 5),
            "algorithmic_bytes_per_launch": int(sum(layer_bytes) / len(layer_bytes)),
        },
        "e2e": e2e,
        "gpu_launches": int(launches),
        "host_manager_us_per_step": round(batch.manager_s / max(batch.steps_planned, 1) * 1e6, 1),
        "cow_pairs_timed": int(cow_pairs),
        "clocks": clocks,
    }
    if read_peak:
        rp = read_peak["best_gbs"]
        res["hbm_frac_of_read_peak"] = round(value / rp, 4)
        res["roofline"]["read_peak_gbs"] = rp
        res["roofline"]["frac_of_read_peak"] = round(achieved_gbs / rp, 4)
    rf = res["roofline"]
    if rf["traffic"] is not None:
        # the same launches on the bytes DRAM actually moved (the shared-prefix workload reads its
        # shared blocks from L2 after the first reader, so its logical GB/s exceeds any HBM figure)
        rf["dram_gbs"] = round(rf["traffic"] / (rf["launch_ms_mean"] * 1e-3) / 1e9, 2)
        rf["frac_on_dram_bytes"] = round(rf["dram_gbs"] / hbm_peak, 4)
        if read_peak:
            rf["frac_on_dram_bytes_of_read_peak"] = round(rf["dram_gbs"] / read_peak["best_gbs"], 4)
    if cpu:
        res["cpu_baseline"] = cpu_baseline(cache, batch, wl, budget_s=cpu_budget)
    del cache, batch, q, k_new, v_new, out, state
    return res


def measure_dense(args, config: str, device, rank: int, read_peak: dict | None) -> dict:
    """The same decode kernels over a dense (batch, heads, max length, head_dim) cache with the same
    context lengths ("Lo que funciona en la Fase 22" keeps such a cache; the identity walk replaces
    the table). A step = one pkv_dense_decode_attention per layer, chained as in the paged step;
    value = KV bytes read / step time; roofline = each launch alone between CUDA events."""
    import torch
    from paged_kv_cache_258_gb300 import pkv

    wl, wdesc, churn = build_workload(config, args.warmup, args.steps, rank, args.layers)
    if churn is not None:
        raise ValueError("the dense comparison needs a fixed batch (gpt, ragged, longdoc)")
    L, B, n_kv, d = wl.n_layers, wl.n_seqs, wl.n_kv_heads, wl.head_dim
    lens = wl.context_lens.astype(np.int32)
    if config in ORDER_LONGEST_FIRST:  # the same row order as the paged batch
        lens = np.sort(lens)[::-1].copy()
    s_max = int(-(-int(lens.max()) // W.BLOCK) * W.BLOCK)
    desc = pkv.make_desc(wl.dtype, L, 1, wl.n_q_heads, n_kv, d)
    dt = pkv.torch_dtype(wl.dtype)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + 23)
    shape = pkv.dense_cache_shape(desc, B, s_max)
    k_cache = torch.randn(shape, dtype=dt, device=device, generator=g)
    v_cache = torch.randn(shape, dtype=dt, device=device, generator=g)
    q = torch.randn((L, B, wl.n_q_heads, d), dtype=dt, device=device, generator=g)
    out = torch.empty_like(q)
    l_t = torch.from_numpy(lens).to(device)
    ws_t = pkv.alloc_workspace(desc, B, s_max // W.BLOCK, device=device)
    stream = torch.cuda.current_stream(device)
    step_bytes = int(lens.astype(np.int64).sum()) * 2 * n_kv * d * wl.elem_bytes * L

    def step(events=None):
        for layer in range(L):
            if events is not None:
                events[layer][0].record(stream)
            pkv.pkv_dense_decode_attention(desc, layer, q[layer], k_cache, v_cache, l_t, wl.scale, out[layer], ws_t,
                                           stream, overlap_previous=events is None and layer > 0)
            if events is not None:
                events[layer][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError(f"device status flags set during the dense pass ({config})")
    ms = t0.elapsed_time(t1)
    durs = [a.elapsed_time(b) for row in evs for a, b in row]
    per_launch = step_bytes / L / (sum(durs) / len(durs) * 1e-3) / 1e9
    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    res = {"value": round(step_bytes * args.steps / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "ms_per_step": round(ms / args.steps, 4),
           "layout": f"dense [{L}][{B}][{n_kv}][{s_max}][{d}] per K and V, identity walk",
           "roofline": {"achieved": round(per_launch, 2), "peak": hbm_peak, "unit": "GB/s",
                        "frac": round(per_launch / hbm_peak, 4), "launch_ms_mean": round(sum(durs) / len(durs), 5)}}
    if read_peak:
        res["roofline"]["frac_of_read_peak"] = round(per_launch / read_peak["best_gbs"], 4)
    del k_cache, v_cache, q, out, ws_t
    return res


def indirection(paged: dict, dense: dict) -> dict:
    """The constant factor of the table walk: 1 - paged / dense, per step and per launch."""
    return {"step": round(1.0 - paged["value"] / dense["value"], 4),
            "per_launch": round(1.0 - paged["roofline"]["achieved"] / dense["roofline"]["achieved"], 4),
            "note": "fraction of the dense cache's bandwidth lost to the block-table walk and scattered placement"}


# the target workloads measured beside the headline one in the default run (one line, keyed objects)
SUB_CONFIGS = ("longdoc", "ragged", "prefix")
DENSE_CONFIGS = ("gpt", "longdoc")  # the dense-cache comparison of the default run
SHORT_STEPS = 200                   # timed steps of the one-layer workloads in the default run
PREFIX_CHURN_STEPS = 256            # steps of the shared-prefix workload's churn log


def run_gpu(args) -> dict | None:
    import gc

    import torch
    from paged_kv_cache_258_gb300 import pkv

    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pkv.lib()
    read_peak = measure_read_peak(device)
    cpu = ws == 1 and not args.no_cpu_baseline
    dense_for = set(DENSE_CONFIGS) if args.dense == "auto" else ({args.config} if args.dense == "on" else set())

    def one_with(a, name, budget):
        r = measure_decode(a, name, device, rank, ws, read_peak, cpu, budget)
        if name in dense_for and a.placement == "shuffled":
            gc.collect()
            torch.cuda.empty_cache()
            r["dense"] = measure_dense(a, name, device, rank, read_peak)
            r["indirection_overhead"] = indirection(r, r["dense"])
        return r

    def one(name, budget):
        return one_with(args, name, budget)

    res = one(args.config, args.cpu_budget)
    subs = {}
    if args.config == "gpt" and not args.no_sub_configs and args.layers is None:
        for name in SUB_CONFIGS:
            gc.collect()
            torch.cuda.empty_cache()
            # the one-layer workloads step in ~0.1-0.4 ms: time at least SHORT_STEPS of them, so that
            # the timed region is not a few milliseconds that one host hiccup would distort
            sub = argparse.Namespace(**vars(args))
            if name == "ragged":
                sub.steps = max(args.steps, SHORT_STEPS)
            elif name == "prefix":  # its churn log has 256 steps: warm-up + value + roofline + e2e passes
                sub.steps = max(args.steps, min(SHORT_STEPS, (PREFIX_CHURN_STEPS - args.warmup) // 3))
            subs[name] = one_with(sub, name, min(args.cpu_budget, 6.0))
            subs[name]["steps"] = sub.steps
            subs[name]["warmup"] = sub.warmup
    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": res["value"],
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": res["dtype"],
        "accumulate": "f32",
        "data": "synthetic (seeded N(0,1) K/V/q; shapes and length mixes of the pages' workloads)",
    }
    line.update({k: v for k, v in res.items() if k not in line})
    line["read_peak"] = read_peak
    if subs:
        line["configs"] = subs
    return line


# ---------------------------------------------------------------------------------------------
# chunked prefill of one long prompt ("01 - Conceito", paragraph 5: a 30,000-token prompt is
# processed in slices); the model is the long-document one (16 layers, 16 query / 4 KV heads x 256,
# bf16). The chunk size is not on the pages: the whole number of waves of the prefill grid closest
# to 2,048 tokens (pkv_prefill_wave_tokens: 2 x 1,216 = 2,432 tokens on a GB300, 76 CTA pairs of 64
# tokens per wave over 4 KV heads; 2,048-token chunks left 1.68 waves and ran 12 % slower per launch).

PREFILL_METRIC = "paged prefill attention TFLOP/s (causal) at 1 GB300; % of tensor roofline"
PREFILL = dict(n_layers=16, n_q=16, n_kv=4, d=256, dtype="bf16", prompt=30000, chunk_target=2048)


def prefill_chunks(prompt: int, chunk: int):
    return [(c0, min(chunk, prompt - c0)) for c0 in range(0, prompt, chunk)]


def setup_prefill_case(device, rank: int = 0, layers=None, placement: str = "shuffled"):
    """The prefill30k case as bench.py times it: pools, chunk stepper and resident inputs."""
    import torch
    from paged_kv_cache_258_gb300 import pkv
    from paged_kv_cache_258_gb300.engine import PagedKVCache, PrefillStep
    P = dict(PREFILL)
    if layers:
        P["n_layers"] = layers
    L, n_q, n_kv, d, prompt = P["n_layers"], P["n_q"], P["n_kv"], P["d"], P["prompt"]
    seed = W.BASE_SEED + 5 + rank
    P["seed"] = seed
    nb_seq = -(-prompt // W.BLOCK)
    num_blocks = int(nb_seq * 1.125) + 1
    desc = pkv.make_desc(P["dtype"], L, num_blocks, n_q, n_kv, d)
    chunk = P["chunk"] = pkv.wave_aligned_chunk(desc, P["chunk_target"])
    order = W.free_order(num_blocks, seed) if placement == "shuffled" else None
    P["free_order"] = order
    cache = PagedKVCache(desc, free_order=order, device=device)
    ps = PrefillStep(cache, max_tokens=chunk, max_seqs=1, max_blocks=nb_seq)
    dt = pkv.torch_dtype(P["dtype"])
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn((L, prompt, n_q, d), device=device, generator=g).to(dt)
    k_new = torch.randn((L, prompt, n_kv, d), device=device, generator=g).to(dt)
    v_new = torch.randn((L, prompt, n_kv, d), device=device, generator=g).to(dt)
    out = torch.empty_like(q)
    return P, cache, ps, (q, k_new, v_new, out), prefill_chunks(prompt, chunk)


def run_prefill_gpu(args) -> dict | None:
    import torch
    from paged_kv_cache_258_gb300 import pkv
    from paged_kv_cache_258_gb300.engine import PagedKVCache, PrefillStep

    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pkv.lib()
    P, cache, ps, (q, k_new, v_new, out), chunks = setup_prefill_case(device, rank, args.layers, args.placement)
    L, n_q, n_kv, d, prompt, chunk = P["n_layers"], P["n_q"], P["n_kv"], P["d"], P["prompt"], P["chunk"]
    stream = ps.stream
    scale = 1.0 / float(np.sqrt(d))
    seq = 1

    def one_step(on_attn=None):
        nonlocal seq
        flops = 0.0
        for i, (c0, n) in enumerate(chunks):
            st = ps.step([(seq, n, i == 0)], q[:, c0:c0 + n], k_new[:, c0:c0 + n], v_new[:, c0:c0 + n],
                         out[:, c0:c0 + n], scale, on_attn)
            flops += PrefillStep.attention_flops(st, n_q, d) * L
        cache.free(seq)       # host only: the next step admits the prompt again
        seq += 1
        return flops

    for _ in range(args.warmup):
        one_step()
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError("device status flags during warm-up")

    n_launch = args.steps * len(chunks) * L
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_launch)]
    cur = {"i": 0}

    def on_attn(layer, when):
        if when == "pre":
            return
        e = ev[cur["i"]]
        if when == "start":
            e[0].record(stream)
        else:
            e[1].record(stream)
            cur["i"] += 1

    sampler = ClockSampler(gpu_uuid(local))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = pkv.pkv_launch_count()
    flops = 0.0
    t0.record(stream)
    for _ in range(args.steps):  # value: the steps alone
        flops += one_step()
    t1.record(stream)
    for _ in range(args.steps):  # roofline: the same steps, each prefill launch between two events
        one_step(on_attn)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = (pkv.pkv_launch_count() - launches0) // 2  # per pass
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError("device status flags set during the timed region")
    ms = reduce_over_ranks(t0.elapsed_time(t1), "max", device)
    total_flops = reduce_over_ranks(flops, "sum", device)
    attn_ms = sum(a.elapsed_time(b) for a, b in ev)
    achieved = flops / (attn_ms * 1e-3) / 1e12
    # algorithmic bytes of a launch: its chunk's q rows read and output rows written, and the K/V rows
    # of every visible key read once (keys 0 .. c0 + n - 1 of the prompt)
    row_q, row_kv = n_q * d * 2, n_kv * d * 2
    alg_bytes = sum(2 * n * row_q + 2 * (c0 + n) * row_kv for c0, n in chunks) / len(chunks)
    traffic = traffic_per_launch("prefill30k", alg_bytes, "paged_prefill_prefill30k.traffic.json",
                                 PREFILL_SOURCES)

    # e2e: every chunk's q / new K / new V rows (all layers) from pinned host memory and its outputs
    # back, on copy streams beside the kernels. Each chunk has its own rows in the device buffers, so
    # a prompt's uploads are queued at once: chunk i's rows go up as soon as the previous prompt's
    # chunk i kernels are done with them, chunk i's kernels wait only for those rows (and for the
    # previous prompt's chunk i outputs to be down), and its outputs go down once its kernels are
    # done. Nothing is recorded between a chunk's launches, so the layer launches still overlap.
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k_new, v_new))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    prev = {"done": None, "down": None}

    def one_step_e2e():
        nonlocal seq
        flops = 0.0
        up, done, down = [], [], []
        with torch.cuda.stream(h2d_s):
            for i, (c0, n) in enumerate(chunks):
                if prev["done"] is not None:
                    h2d_s.wait_event(prev["done"][i])  # the previous prompt's chunk i has read these rows
                for l in range(L):
                    for dev_t, host_t in ((q, hq), (k_new, hk), (v_new, hv)):
                        dev_t[l, c0:c0 + n].copy_(host_t[l, c0:c0 + n], non_blocking=True)
                up.append(torch.cuda.Event())
                up[-1].record(h2d_s)
        for i, (c0, n) in enumerate(chunks):
            stream.wait_event(up[i])
            if prev["down"] is not None:
                stream.wait_event(prev["down"][i])  # the previous prompt's chunk i outputs are on the host
            st = ps.step([(seq, n, i == 0)], q[:, c0:c0 + n], k_new[:, c0:c0 + n], v_new[:, c0:c0 + n],
                         out[:, c0:c0 + n], scale)
            flops += PrefillStep.attention_flops(st, n_q, d) * L
            done.append(torch.cuda.Event())
            done[-1].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[-1])
                for l in range(L):
                    hout[l, c0:c0 + n].copy_(out[l, c0:c0 + n], non_blocking=True)
                down.append(torch.cuda.Event())
                down[-1].record(d2h_s)
        prev.update(done=done, down=down)
        cache.free(seq)  # host only: the next step admits the prompt again
        seq += 1
        return flops

    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_sampler = ClockSampler(gpu_uuid(local))  # the copies add power: the e2e pass has its own clocks
    e2e_sampler.start()
    e0.record(stream)
    h2d_s.wait_event(e0)  # no copy starts before the timed region
    e2e_flops = 0.0
    for _ in range(args.steps):
        e2e_flops += one_step_e2e()
    stream.wait_event(prev["down"][-1])  # the last prompt's outputs are on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_clocks = e2e_sampler.stop()
    e2e_ms = reduce_over_ranks(e0.elapsed_time(e1), "max", device)
    e2e_flops = reduce_over_ranks(e2e_flops, "sum", device)
    if rank != 0:
        return None
    peaks = measured_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
    peak_src = "measured bf16_tflops_sustained (cuBLAS bf16 GEMM, seconds-long loop)" \
        if "bf16_tflops_sustained" in peaks else "fallback 1.7 PFLOP/s sustained"
    value = total_flops / (ms * 1e-3) / 1e12
    elem = 2
    h2d = (q.numel() + k_new.numel() + v_new.numel()) * elem
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "data": "synthetic (seeded N(0,1) q and K/V rows)",
        "config": {"workload": f"prefill30k: one {prompt}-token prompt in {len(chunks)} chunks of {chunk} tokens, "
                               f"{L} layers x {n_q} q / {n_kv} kv heads x head_dim {d} bf16, block 16",
                   "step": "per chunk: manager admit/extend, one metadata upload, per layer kv_append + "
                           "paged prefill attention",
                   "l2": "no flush: each step streams 5.9 GB of new rows and 1 GiB of cache per layer set",
                   "parallelism": f"replicas x{ws} (one prompt per rank, no collective)",
                   "placement": args.placement},
        "prompt_tokens_per_s": round(prompt * args.steps * ws / (ms * 1e-3), 1),
        "roofline": {"kernel": "paged_prefill_umma_kernel (tcgen05, S and O in tensor memory, TMA K/V producers)",
                     "bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "peak_source": peak_src,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_note": "DRAM bytes per launch: a late chunk's ncu capture scaled by the mean "
                                     "launch's algorithmic bytes",
                     "algorithmic_bytes_per_launch": int(alg_bytes),
                     "launch_ms_mean": round(attn_ms / n_launch, 4),
                     "algorithmic_flops_per_launch": int(flops / n_launch)},
        "e2e": {"value": round(e2e_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out.numel() * elem),
                "ms_per_step": round(e2e_ms / args.steps, 3), "clocks": e2e_clocks},
        "gpu_launches": int(launches),
        "host_manager_us_per_step": round(ps.manager_s / max(1, (args.warmup + 2 * args.steps)) * 1e6, 1),
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_sample(cache, budget_s=args.cpu_budget, P=P, seed=P["seed"])
    return line


def prefill_cpu_sample(cache=None, budget_s: float = 12.0, P=None, seed: int = 0) -> dict:
    """The fp64 oracle's prefill, as it stands, on this host's cores: blocks of 64 queries of the
    prompt's last chunk (the costliest positions) on one layer, until the budget is spent."""
    import oracle
    P = P or PREFILL
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(seed + 17)
    prompt, n_q, n_kv, d, dtype = P["prompt"], P["n_q"], P["n_kv"], P["d"], P["dtype"]
    nb = -(-prompt // W.BLOCK)
    tables = W.shuffled_tables(np.array([prompt], dtype=np.int32), nb, seed)
    kp = W.normal_values(rng, (nb, n_kv, W.BLOCK, d), dtype)
    vp = W.normal_values(rng, (nb, n_kv, W.BLOCK, d), dtype)
    flops, el, done = 0.0, 0.0, 0
    chunk = P.get("chunk") or P["chunk_target"]  # the host sample needs no device: the nominal chunk
    last0 = prompt - (prompt % chunk or chunk)
    while el < budget_s and last0 + done + 64 <= prompt:
        c = last0 + done + 64                       # the cache holds positions 0 .. c-1
        q = W.normal_values(rng, (64, n_q, d), dtype)
        t0 = time.perf_counter()
        oracle.paged_prefill(dtype, q, kp, vp, tables, np.array([c], np.int32), np.array([0, 64], np.int32),
                             1.0 / np.sqrt(d), n_threads=threads)
        el += time.perf_counter() - t0
        flops += 4.0 * d * n_q * (64 * (c - 64) + 64 * 65 / 2)
        done += 64
    return {"value": round(flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} queries of the last chunk (positions {last0}..{last0 + done - 1}), 1 layer, "
                      f"{n_q} heads (fp64 C oracle, OpenMP over (sequence, head)); {el:.1f} s"}


def run_e2e(args, batch, cache, state, bufs, scale, device) -> dict:
    import torch
    q, k_new, v_new, out = bufs
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k_new, v_new))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    stream = batch.stream
    meta = batch.n * 8 + batch.n * batch.max_blocks * 4 + batch.n * 4
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv)) + meta
    d2h = hout.numel() * hout.element_size()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    kv = 0
    npairs = 0
    # step i's inputs go up while step i-1 computes and its outputs come down while step i+1 does
    # (engine.StepCopyPipeline); the layer launches of a step follow each other directly
    from paged_kv_cache_258_gb300.engine import StepCopyPipeline
    pipe = StepCopyPipeline(stream, device, lambda: {"q": torch.empty_like(q), "k": torch.empty_like(k_new),
                                                     "v": torch.empty_like(v_new), "out": torch.empty_like(out)})
    host_in = {"q": hq, "k": hk, "v": hv}
    sampler = ClockSampler(gpu_uuid(device.index))  # the copies add power: the e2e pass has its own clocks
    sampler.start()
    t0.record(stream)
    with torch.cuda.stream(stream):
        pipe.upload(host_in)
        for i in range(args.steps):
            dev = pipe.begin()
            st = batch.step(dev["q"], dev["k"], dev["v"], dev["out"], scale)
            pipe.end({"out": hout})
            if i + 1 < args.steps:
                pipe.upload(host_in)     # the next step's rows, while this step computes
            kv += batch.kv_bytes_last_step()
            npairs += st["npairs"]
            apply_churn(cache, batch, state)
        pipe.finish()                    # the last step's outputs are on the host
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    ms = reduce_over_ranks(t0.elapsed_time(t1), "max", device)
    kv = reduce_over_ranks(kv, "sum", device)
    return {"value": round(kv / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d + 8 * npairs // max(args.steps, 1)), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / args.steps, 4), "clocks": clocks}


DECODE_SOURCES = ("decode.cuh", "decode_mma.cuh", "common.cuh")
COPY_SOURCES = ("append_copy.cu", "common.cuh")
PREFILL_SOURCES = ("prefill_umma.cuh", "umma.cuh", "decode_mma.cuh", "common.cuh", "prefill_bf16.cu")


def traffic_per_launch(config: str, algorithmic: float, profile: str | None = None,
                       sources: tuple = DECODE_SOURCES):
    """DRAM bytes per launch from a committed ncu capture, if it matches the kernel as built now."""
    f = ROOT / "profiles" / (profile or f"paged_decode_{config}.traffic.json")
    if not f.exists():
        return None
    try:
        rec = json.loads(f.read_text())
    except ValueError:
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash(sources):
        return None  # the kernel changed since the counters were taken
    ratio = rec.get("dram_bytes_per_algorithmic_byte")
    return None if ratio is None else int(ratio * algorithmic)


def kernel_source_hash(sources: tuple = DECODE_SOURCES) -> str:
    """sha256 of the kernel sources' code: comments dropped and whitespace runs collapsed, so that a
    documentation edit does not void counters taken on the same code (string literals are kept)."""
    import hashlib
    import re
    token = re.compile(r'("(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\')|//[^\n]*|/\*.*?\*/', re.S)
    h = hashlib.sha256()
    csrc = ROOT / "paged_kv_cache_258_gb300" / "csrc"
    for name in sources:
        code = token.sub(lambda m: m.group(1) or " ", (csrc / name).read_text())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()


# ---------------------------------------------------------------------------------------------
# CPU oracle (reported baseline, and the reference arm)

def _host_pool(t, dtype: str) -> np.ndarray:
    import torch
    if dtype == "bf16":
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def cpu_baseline(cache, batch, wl, budget_s: float = 12.0) -> dict:
    """The fp64 oracle, as it stands, on this host's cores over whole layers of the same batch."""
    import oracle
    threads = os.cpu_count() or 1
    st = batch._stage[batch._turn ^ 1]
    tables = st["tables"].numpy().copy()
    lens = st["lens"].numpy().copy()
    dtype = wl.dtype
    q_all = None
    done_bytes, elapsed, layers = 0, 0.0, 0
    per_layer = int(lens.astype(np.int64).sum()) * cache.kv_bytes_per_token_layer()
    rng = np.random.default_rng(wl.seed + 11)
    for layer in range(wl.n_layers):
        kp = _host_pool(cache.k_pool[layer], dtype)
        vp = _host_pool(cache.v_pool[layer], dtype)
        q_all = W.normal_values(rng, (batch.n, wl.n_q_heads, wl.head_dim), dtype)
        t0 = time.perf_counter()
        oracle.paged_decode(dtype, q_all, kp, vp, tables, lens, wl.scale, n_threads=threads)
        elapsed += time.perf_counter() - t0
        done_bytes += per_layer
        layers += 1
        if elapsed >= budget_s:
            break
    return {"value": round(done_bytes / elapsed / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{layers} of {wl.n_layers} layers x all {batch.n} sequences x {wl.n_q_heads} heads "
                      f"(fp64 C oracle, OpenMP over (sequence, head)); {elapsed:.1f} s",
            "tokens_per_s": round(batch.n * layers / wl.n_layers / elapsed, 3)}


def run_reference(args) -> dict | None:
    """The reference arm: the fp64 CPU oracle timed on this host's cores, same config and metric."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl, wdesc, churn = build_workload(args.config, args.warmup, args.steps)
    rng = np.random.default_rng(wl.seed)
    threads = os.cpu_count() or 1
    if churn is not None:
        lens = np.array([churn.group_prompt[g] + 1 for g in churn.member_group], dtype=np.int32)
    else:
        lens = wl.context_lens.copy()
    # one layer's worth of the workload, sequences taken in order until the sample is ~0.3 s of work
    n_take = len(lens)
    if args.config == "longdoc":
        n_take = 1
    elif args.config in ("gpt", "prefix"):
        n_take = 16 if args.config == "gpt" else 32
    sel = lens[:n_take]
    nb = int(np.sum(-(-sel.astype(np.int64) // W.BLOCK)))
    tables = W.shuffled_tables(sel, nb, wl.seed)
    kp = W.normal_values(rng, (nb, wl.n_kv_heads, W.BLOCK, wl.head_dim), wl.dtype)
    vp = W.normal_values(rng, (nb, wl.n_kv_heads, W.BLOCK, wl.head_dim), wl.dtype)
    q = W.normal_values(rng, (n_take, wl.n_q_heads, wl.head_dim), wl.dtype)
    step_bytes = int(sel.astype(np.int64).sum()) * 2 * wl.n_kv_heads * wl.head_dim * wl.elem_bytes
    for _ in range(args.warmup):
        oracle.paged_decode(wl.dtype, q, kp, vp, tables, sel, wl.scale, n_threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_decode(wl.dtype, q, kp, vp, tables, sel, wl.scale, n_threads=threads)
    el = time.perf_counter() - t0
    value = step_bytes * args.steps / el / 1e9
    sample = f"per step: 1 layer x {n_take} of {wl.n_seqs if churn is None else len(lens)} sequences x " \
             f"{wl.n_q_heads} heads (fp64 C oracle, {threads} threads)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": wdesc, "kv_dtype": wl.dtype},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------------------
# continuous batching ("01 - Conceito", paragraphs 5-8): Poisson arrivals of two request classes on
# the GPT-style model of "Configurando as Constantes"; the loop synchronises every iteration to
# timestamp its tokens, as a serving loop does. Attention and cache management only: no model
# weights run, q and the new K/V rows are synthetic.

SERVE_METRIC = "continuous batching on the paged KV cache: generated tokens/s at 1 GB300 (attention + cache only)"
SERVE = dict(n_layers=32, n_q=32, n_kv=32, d=128, dtype="f16", num_blocks=16384, n_requests=192, rate=48.0,
             max_batch_tokens=2048, chunk=512, max_running=160, max_blocks=1024, seed=W.BASE_SEED + 6)


def serve_trace(P):
    from paged_kv_cache_258_gb300.scheduler import synthetic_trace
    reqs = synthetic_trace(P["n_requests"], seed=P["seed"], rate_per_s=P["rate"],
                           classes=[("chat", 0.85, 1), ("doc", 0.15, 0)])
    rng = np.random.default_rng(P["seed"] + 1)
    for r in reqs:
        if r.klass == "doc":                      # long documents: 2k..8k-token prompts
            r.prompt = int(rng.integers(2048, 8193))
    return reqs


def run_serve_gpu(args) -> dict | None:
    import torch
    from paged_kv_cache_258_gb300 import pkv
    from paged_kv_cache_258_gb300.engine import PagedKVCache, StepExecutor
    from paged_kv_cache_258_gb300.scheduler import Scheduler, serve

    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    P = dict(SERVE)
    if args.layers:
        P["n_layers"] = args.layers
    if args.rate:
        P["rate"] = float(args.rate)
    L, n_q, n_kv, d = P["n_layers"], P["n_q"], P["n_kv"], P["d"]
    desc = pkv.make_desc(P["dtype"], L, P["num_blocks"], n_q, n_kv, d)
    order = W.free_order(P["num_blocks"], P["seed"] + rank)
    cache = PagedKVCache(desc, free_order=order, device=device)
    D, T = P["max_running"], P["max_batch_tokens"]
    ex = StepExecutor(cache, max_decode=D, max_tokens=T, max_chunks=D, max_blocks=P["max_blocks"])
    stream = ex.stream
    dt = pkv.torch_dtype(P["dtype"])
    g = torch.Generator(device=device)
    g.manual_seed(P["seed"] + rank)
    dev_in = [torch.randn(shape, device=device, generator=g).to(dt)
              for shape in ((L, D, n_q, d), (L, D, n_kv, d), (L, D, n_kv, d), (L, T, n_q, d), (L, T, n_kv, d),
                            (L, T, n_kv, d))]
    d_out = torch.empty((L, D, n_q, d), dtype=dt, device=device)
    p_out = torch.empty((L, T, n_q, d), dtype=dt, device=device)
    # e2e buffers: an iteration's n rows of a tensor are one contiguous [L, n, heads, d] image at the
    # front of a flat buffer, so each tensor goes up (or comes down) in one copy
    flat_dev = [torch.empty(t.numel(), dtype=dt, device=device) for t in dev_in + [d_out, p_out]]
    flat_host = [t.reshape(-1).cpu().pin_memory() for t in dev_in]
    flat_host += [torch.empty(t.numel(), dtype=dt).pin_memory() for t in (d_out, p_out)]

    def rows(flat, like, n):
        return flat[: like.shape[0] * n * like[0, 0].numel()].view(like.shape[0], n, *like.shape[2:])
    scale = 1.0 / float(np.sqrt(d))
    kv_tok = 2 * n_kv * d * 2

    def one_run(copies: bool, timed_events: bool):
        sched = Scheduler(cache.mgr, max_batch_tokens=T, chunk=P["chunk"], max_running=D, max_blocks=P["max_blocks"])
        reqs = serve_trace(P)
        evs, dec_bytes, pre_flops = [], [0], [0.0]
        h2d, d2h = [0], [0]
        t_start = [None]

        def clock():
            return time.perf_counter() - t_start[0]

        def wait_until(t):
            dt_ = t - clock()
            if dt_ > 0:
                time.sleep(dt_)

        def on_kernel(kind, layer, when):
            if not timed_events or kind != "decode" or when == "pre":
                return
            if when == "start":
                evs.append([torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)])
                evs[-1][0].record(stream)
            else:
                evs[-1][1].record(stream)

        def execute(plan):
            nd, nt = plan.n_dec, plan.n_pre_tokens
            counts = (nd, nd, nd, nt, nt, nt, nd, nt)
            if copies:
                ins = [rows(fd, like, n) for fd, like, n in zip(flat_dev, dev_in + [d_out, p_out], counts)]
                with torch.cuda.stream(stream):
                    for i in range(6):
                        if counts[i]:
                            ins[i].copy_(rows(flat_host[i], dev_in[i], counts[i]), non_blocking=True)
                            h2d[0] += ins[i].numel() * 2
            else:
                ins = [t[:, :n] for t, n in zip(dev_in + [d_out, p_out], counts)]
            dq, dk, dv, pq, pk, pv, do, po = ins
            # without per-kernel events the iteration's launches follow each other as dependents
            ex.run(plan, (dq, dk, dv, do), (pq, pk, pv, po), scale, on_kernel if timed_events else None)
            if copies:
                with torch.cuda.stream(stream):
                    for j, (o, n) in enumerate(((do, nd), (po, nt))):
                        if n:
                            rows(flat_host[6 + j], o, n).copy_(o, non_blocking=True)
                            d2h[0] += o.numel() * 2
            stream.synchronize()                     # tokens of this iteration exist now
            dec_bytes[0] += int(plan.dec_lens.astype(np.int64).sum()) * kv_tok * L
            for i, (o, n) in enumerate(plan.pre_chunks):
                c = int(plan.pre_lens[i])
                pre_flops[0] += 4.0 * d * n_q * (n * (c - n) + n * (n + 1) / 2) * L

        torch.cuda.synchronize()
        barrier()
        t_start[0] = time.perf_counter()
        steps = serve(sched, reqs, execute, clock, wait_until)
        wall = clock()
        return sched, reqs, steps, wall, evs, dec_bytes[0], pre_flops[0], h2d[0], d2h[0]

    # warm-up: a short trace (kernels loaded, tensor maps cached, pinned buffers touched)
    saved = dict(P)
    P.update(n_requests=max(8, args.warmup * 4))
    for _ in range(1):
        one_run(False, False)
    P.clear()
    P.update(saved)
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError("device status flags during warm-up")
    sampler = ClockSampler(gpu_uuid(local))
    sampler.start()
    launches0 = pkv.pkv_launch_count()
    sched, reqs, steps, wall, _, _, pre_flops, _, _ = one_run(False, False)  # value: no events
    launches = pkv.pkv_launch_count() - launches0
    clocks = sampler.stop()
    torch.cuda.synchronize()
    if pkv.pkv_get_device_status(stream):
        raise RuntimeError("device status flags set during the timed run")
    # roofline: the same trace again with an event pair around every decode launch
    _, _, _, _, evs, dec_bytes, _, _, _ = one_run(False, True)
    dec_ms = sum(a.elapsed_time(b) for a, b in evs)
    m = sched.metrics()
    tokens = sum(r.generated for r in reqs if r.state == "done")
    wall_max = reduce_over_ranks(wall, "max", device)
    tokens_all = reduce_over_ranks(tokens, "sum", device)
    sched2, reqs2, steps2, wall2, _, _, _, h2d, d2h = one_run(True, False)
    wall2 = reduce_over_ranks(wall2, "max", device)
    tokens2 = reduce_over_ranks(sum(r.generated for r in reqs2 if r.state == "done"), "sum", device)
    if rank != 0:
        return None
    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    line = {
        "metric": SERVE_METRIC, "value": round(tokens_all / wall_max, 1), "unit": "tokens/s", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(wall_max / max(steps, 1) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": P["dtype"], "accumulate": "f32",
        "data": "synthetic (Poisson arrivals; seeded q and K/V rows; no model weights)",
        "config": {"workload": f"serve: {P['n_requests']} requests at {P['rate']}/s, 85% chat (prompt U{{64..512}}, "
                               f"response min(Geom(1/500), 2048), priority 1) / 15% doc (prompt U{{2048..8192}}, "
                               f"response U{{16..128}}, priority 0); GPT-style 32 layers x 32 heads x 128 fp16, "
                               f"pool {P['num_blocks']} blocks ({P['num_blocks'] * 16} tokens)",
                   "scheduler": f"max {T} tokens per iteration, prefill chunks <= {P['chunk']}, <= {D} running",
                   "step": "one scheduler iteration (plan on the C manager, one metadata upload, CoW copies, the "
                           "chunk appends of every layer, then per layer prefill attention and fused append + "
                           "decode attention launched as programmatic dependents, sync)",
                   "l2": "no flush: decode iterations read more KV than L2 holds",
                   "parallelism": f"replicas x{ws} (one trace per rank, no collective)"},
        "wall_s": round(wall_max, 3),
        "classes": m["classes"], "blocks": m["blocks"],
        "prefill_tflops": round(pre_flops / wall / 1e12, 2),
        "roofline": {"kernel": "paged_decode_mma_kernel (fused append) inside the serving loop", "bound": "hbm",
                     "achieved": round(achieved, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": None,
                     "launch_ms_mean": round(dec_ms / max(1, len(evs)), 4),
                     "algorithmic_bytes_per_launch": int(dec_bytes / max(1, len(evs)))},
        "e2e": {"value": round(tokens2 / wall2, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d / max(steps2, 1)),
                "d2h_bytes_per_step": int(d2h / max(steps2, 1)), "wall_s": round(wall2, 3)},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    return line


# ---------------------------------------------------------------------------------------------
# the copy kernels alone: copy-on-write block copies ("01 - Conceito", paragraph 6: 200 pairs, as
# when every member of the prefix-sharing workload first writes into its shared tail block) over the
# GPT-style model's 32 layers, and the per-layer KV append of a 64-token decode batch ("La idea de
# PagedAttention", step 3)

APPEND_COPY_METRIC = "KV append + copy-on-write block copy: GB/s moved (read + write) at 1 GB300; % of HBM roofline"
AC = dict(n_layers=32, n_q=32, n_kv=32, d=128, dtype="f16", num_blocks=2048, batch=64, pairs=200,
          seed=W.BASE_SEED + 7)


def append_copy_bytes(P) -> tuple[int, int]:
    """Bytes read + written per step by copy_blocks and by the layer loop of kv_append."""
    row = P["n_kv"] * P["d"] * 2  # one token's K (or V) row of one layer, fp16
    copy = P["pairs"] * P["n_layers"] * row * W.BLOCK * 2 * 2  # K and V, read and write
    append = P["batch"] * P["n_layers"] * row * 2 * 2
    return copy, append


def append_copy_inputs(P, n_steps: int):
    """Seeded per-step slots (distinct within a step) and the fixed copy pairs (disjoint src / dst)."""
    rng = np.random.default_rng(P["seed"])
    half = P["num_blocks"] // 2
    src = rng.permutation(half)[: P["pairs"]]
    dst = half + rng.permutation(half)[: P["pairs"]]
    pairs = np.stack([src, dst], axis=1).astype(np.int32)
    slots = np.stack([rng.permutation(P["num_blocks"] * W.BLOCK)[: P["batch"]] for _ in range(n_steps)])
    return pairs, slots.astype(np.int64)


def run_append_copy_gpu(args) -> dict | None:
    import torch
    from paged_kv_cache_258_gb300 import pkv

    ws, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pkv.lib()
    P = dict(AC, n_layers=args.layers) if args.layers else AC
    L = P["n_layers"]
    desc = pkv.make_desc(P["dtype"], L, P["num_blocks"], P["n_q"], P["n_kv"], P["d"])
    g = torch.Generator(device=device)
    g.manual_seed(P["seed"] + rank)
    kp = torch.empty(pkv.pool_shape(desc), dtype=torch.float16, device=device).normal_(generator=g)
    vp = torch.empty_like(kp).normal_(generator=g)
    k_new = torch.empty((L, P["batch"], P["n_kv"], P["d"]), dtype=torch.float16, device=device).normal_(generator=g)
    v_new = torch.empty_like(k_new).normal_(generator=g)
    n_steps = args.warmup + 3 * args.steps
    pairs_h, slots_h = append_copy_inputs(P, n_steps)
    pairs = torch.from_numpy(pairs_h).to(device)
    slots = torch.from_numpy(slots_h).to(device)
    stream = torch.cuda.current_stream()
    copy_b, append_b = append_copy_bytes(P)

    # The 32 appends of a step (~1-2 us of GPU work each) are replayed from a CUDA graph, as a
    # serving loop would issue them: launched one by one from Python they wait on the host. The
    # graph reads the step's slots from a fixed buffer that each step refills on the device.
    # Two sets of (rows, slots, graph): the e2e pass uploads step i+1's rows into one set while
    # step i's kernels read the other.
    sets = []
    cap = torch.cuda.Stream()
    for s_ in range(2):
        kn, vn = (k_new, v_new) if s_ == 0 else (torch.empty_like(k_new), torch.empty_like(v_new))
        sb = torch.empty(P["batch"], dtype=torch.int64, device=device)
        sb.copy_(slots[0])
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):  # one eager pass on the capture stream before capturing
            for layer in range(L):
                pkv.pkv_kv_append(desc, layer, kn[layer], vn[layer], sb, kp, vp)
        stream.wait_stream(cap)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            for layer in range(L):
                pkv.pkv_kv_append(desc, layer, kn[layer], vn[layer], sb, kp, vp)
        sets.append(dict(k=kn, v=vn, slots=sb, graph=gr, up=torch.cuda.Event(), free=None))
    torch.cuda.synchronize()

    def one_step(i, ev=None, host=None):
        st = sets[i % 2] if host is not None else sets[0]
        if host is not None:
            # the step's rows from pinned host memory on the copy stream, into the set the graph of
            # step i - 2 has finished reading; slots and pairs through the metadata-upload kernel,
            # which does not wait behind the row copies
            hk, hv, hsl, hpr, h2d_s = host
            with torch.cuda.stream(h2d_s):
                if st["free"] is not None:
                    h2d_s.wait_event(st["free"])
                st["k"].copy_(hk, non_blocking=True)
                st["v"].copy_(hv, non_blocking=True)
                st["up"].record(h2d_s)
            pkv.pkv_upload_metadata(st["slots"], hsl[i], stream=stream)
            pkv.pkv_upload_metadata(pairs, hpr, stream=stream)
        else:
            st["slots"].copy_(slots[i])
        if ev is not None:
            ev[0].record(stream)
        pkv.pkv_copy_blocks(desc, kp, vp, pairs)  # copies first, then the new rows (step order)
        if ev is not None:
            ev[1].record(stream)
        if host is not None:
            stream.wait_event(st["up"])
        st["graph"].replay()
        if ev is not None:
            ev[2].record(stream)
        if host is not None:
            st["free"] = torch.cuda.Event()
            st["free"].record(stream)

    for i in range(args.warmup):
        one_step(i)
    if pkv.pkv_get_device_status():
        raise RuntimeError("device status flags during warm-up")
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    sampler = ClockSampler(gpu_uuid(local))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    sampler.start()
    launches0 = pkv.pkv_launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for j in range(args.steps):  # value: the steps alone
        one_step(args.warmup + j)
    t1.record(stream)
    for j in range(args.steps):  # roofline: the same kind of steps with events around each kernel group
        one_step(args.warmup + args.steps + j, evs[j])
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    # copy_blocks launches counted by the library, plus the appends each graph replay runs
    launches = (pkv.pkv_launch_count() - launches0) // 2 + args.steps * L
    if pkv.pkv_get_device_status():
        raise RuntimeError("device status flags set during the timed region")
    ms = reduce_over_ranks(t0.elapsed_time(t1), "max", device)
    copy_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    append_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps

    # e2e: new rows, slots and pairs from pinned host memory each step; one destination block of
    # layer 0 read back (the copy's result) at the end of every step
    host = (k_new.cpu().pin_memory(), v_new.cpu().pin_memory(), torch.from_numpy(slots_h).pin_memory(),
            torch.from_numpy(pairs_h).pin_memory(), torch.cuda.Stream(device))
    back = torch.empty(kp[0, 0].shape, dtype=kp.dtype).pin_memory()
    dst0 = int(pairs_h[0, 1])
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    host[-1].wait_event(e0)  # no copy starts before the timed region
    for j in range(args.steps):
        one_step(args.warmup + 2 * args.steps + j, host=host)
        back.copy_(kp[0, dst0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_over_ranks(e0.elapsed_time(e1), "max", device)
    if rank != 0:
        return None
    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peak_src = "measured hbm_gbs (copy bandwidth, read + write bytes)" if "hbm_gbs" in peaks \
        else f"fallback {FALLBACK_HBM_GBS:.0f} GB/s"
    step_bytes = copy_b + append_b
    value = step_bytes * args.steps * ws / (ms * 1e-3) / 1e9
    achieved = copy_b / (copy_ms * 1e-3) / 1e9
    h2d = (k_new.numel() + v_new.numel()) * 2 + P["batch"] * 8 + pairs.numel() * 4
    line = {
        "metric": APPEND_COPY_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) pools and rows; seeded slots and pairs)",
        "config": {"workload": f"appendcopy: copy_blocks of {P['pairs']} copy-on-write pairs over {L} layers "
                               f"(K and V) + kv_append of a {P['batch']}-token batch into each of {L} layers; "
                               f"{P['n_kv']} kv heads x head_dim {P['d']} fp16, block 16, {P['num_blocks']} blocks",
                   "l2": "no flush: each step copies 1.68 GB of distinct blocks (larger than L2)",
                   "parallelism": f"replicas x{ws} (one pool per rank, no collective)"},
        "roofline": {"kernel": "copy_blocks_kernel (16-byte vector copies, grid pair x layer x K/V)",
                     "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic_per_launch("appendcopy", copy_b, "copy_blocks_appendcopy.traffic.json",
                                                   COPY_SOURCES),
                     "launch_ms_mean": round(copy_ms, 5), "algorithmic_bytes_per_launch": int(copy_b)},
        "append": {"kernel": "kv_append_kernel", "launches_per_step": L, "issued": "CUDA graph replay",
                   "us_per_launch": round(append_ms / L * 1e3, 3),
                   "gbs": round(append_b / (append_ms * 1e-3) / 1e9, 2),
                   "bytes_per_launch": int(append_b // L)},
        "e2e": {"value": round(step_bytes * args.steps * ws / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(back.numel() * 2),
                "ms_per_step": round(e2e_ms / args.steps, 4)},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = append_copy_cpu_sample(budget_s=args.cpu_budget)
    return line


_AC_HOST = {}


def append_copy_cpu_sample(budget_s: float = 10.0, layers: int = 2) -> dict:
    """The oracle's copy_blocks and kv_append (plain byte copies) on host pools of `layers` layers."""
    import oracle
    oracle.build()
    P = dict(AC, n_layers=layers)
    if layers not in _AC_HOST:  # host pools built once per process (their bits do not matter to a copy)
        rng = np.random.default_rng(P["seed"])
        shape = (layers, P["num_blocks"], P["n_kv"], W.BLOCK, P["d"])
        kp = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16).view(np.float16)
        vp = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16).view(np.float16)
        kn = rng.standard_normal((P["batch"], P["n_kv"], P["d"]), dtype=np.float32).astype(np.float16)
        vn = rng.standard_normal((P["batch"], P["n_kv"], P["d"]), dtype=np.float32).astype(np.float16)
        pairs, slots = append_copy_inputs(P, 64)
        _AC_HOST[layers] = (kp, vp, kn, vn, pairs, slots)
    kp, vp, kn, vn, pairs, slots = _AC_HOST[layers]
    copy_b, append_b = append_copy_bytes(P)
    done, el, steps = 0, 0.0, 0
    while el < budget_s and steps < 10_000:
        t0 = time.perf_counter()
        oracle.copy_blocks(kp, vp, pairs)
        for layer in range(layers):
            oracle.kv_append(kn, vn, slots[steps % len(slots)], kp[layer], vp[layer])
        el += time.perf_counter() - t0
        done += copy_b + append_b
        steps += 1
    return {"value": round(done / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{steps} steps of the same work on {layers} of {AC['n_layers']} layers "
                      f"(fp16 byte copies in the C oracle, one thread); {el:.1f} s"}


def run_append_copy_reference(args) -> dict | None:
    """Reference arm of the appendcopy line: the oracle's byte copies, as they stand, on the host."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    per_step = max(0.5, 60.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        append_copy_cpu_sample(budget_s=per_step / 4)
    t0 = time.perf_counter()
    samples = [append_copy_cpu_sample(budget_s=per_step) for _ in range(args.steps)]
    el = time.perf_counter() - t0
    value = statistics.median(s_["value"] for s_ in samples)
    cb = dict(samples[0])
    cb["value"] = value
    return {
        "impl": "reference", "metric": APPEND_COPY_METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded)",
        "config": {"workload": "appendcopy (bounded sample: 2 of 32 layers)"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_prefill_reference(args) -> dict | None:
    """Reference arm of the prefill line: the fp64 oracle, as it stands, on a bounded sample."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    per_step = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        prefill_cpu_sample(budget_s=per_step / 4, seed=W.BASE_SEED + 5)
    t0 = time.perf_counter()
    samples = [prefill_cpu_sample(budget_s=per_step, seed=W.BASE_SEED + 5) for _ in range(args.steps)]
    el = time.perf_counter() - t0
    value = statistics.median(s_["value"] for s_ in samples)
    cb = dict(samples[0])
    cb["value"] = value
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "prefill30k (bounded sample: queries of the last chunk, one layer)"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="gpt",
                    choices=["gpt", "ragged", "longdoc", "prefix", "prefill30k", "serve", "appendcopy"])
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="gpt only: skip the longdoc / ragged / prefix measurements of the default run")
    ap.add_argument("--dense", default="auto", choices=["auto", "on", "off"],
                    help="time the same kernels over a dense (B, H, S, d) cache beside the paged pool: "
                         "auto = gpt and longdoc, on = this config too, off = never")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling)")
    ap.add_argument("--placement", default="shuffled", choices=["shuffled", "contiguous"],
                    help="physical placement of each sequence's blocks (indirection-overhead study)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--rate", type=float, default=None,
                    help="serve: request arrivals per second (default 48; a very large rate submits all at once)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        if args.config == "prefill30k":
            line = run_prefill_reference(args)
        elif args.config == "appendcopy":
            line = run_append_copy_reference(args)
        elif args.config == "serve":
            line = {"impl": "reference", "unavailable": "the serving loop has no CPU restatement: its kernels' "
                                                       "reference arms are --config gpt and --config prefill30k"}
        else:
            line = run_reference(args)
    elif args.config == "prefill30k":
        line = run_prefill_gpu(args)
    elif args.config == "appendcopy":
        line = run_append_copy_gpu(args)
    elif args.config == "serve":
        line = run_serve_gpu(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
