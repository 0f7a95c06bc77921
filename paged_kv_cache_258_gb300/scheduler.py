"""Continuous batching on the paged KV cache: iteration-level scheduling, host side.

"PagedAttention e continuous batching", "01 - Conceito":
  * paragraph 5 -- the batch is revisited at every iteration boundary: finished or cancelled
    sequences leave, waiting ones enter, running ones advance one token; the scheduler weighs
    free blocks, a maximum of tokens per batch, priorities and the prefill/decode mix, and slices
    long prefills so that a newcomer's 30,000-token prompt does not stall everyone's next token;
  * paragraph 6 -- requests with the same prompt prefix share its blocks (here: a resident
    prefix root that requests fork from; copy-on-write on the first divergent write);
  * paragraph 7 -- admission reasons in countable blocks and refuses early, with a clear error,
    instead of failing in the middle of generation;
  * paragraph 8 -- block metrics, plus queue delay, time to first token and inter-token latency,
    reported per request class so that throughput cannot hide starvation.

Readings taken where the page is silent (each listed in the design notes):
  * a request is refused at submission when its prompt alone needs more blocks than the pool
    has; otherwise it waits until its whole prompt (plus ``headroom_blocks``) fits in the free
    blocks, then it is admitted and prefilled chunk by chunk;
  * each step first reserves one decode slot for every running, fully prefilled sequence; when
    the manager reports an append OOM the scheduler preempts the running request with the lowest
    priority and, among those, the latest arrival (its blocks return to the pool; it re-enters
    the queue and later recomputes its cache by prefill -- the tokens it already emitted stay
    emitted); then the remaining token budget goes to prefill chunks: requests already
    prefilling first (arrival order), then admissions in (priority, arrival) order;
  * a request emits its first token when its prompt is fully prefilled and one more token per
    decode step; it finishes after ``response`` tokens. No model runs: the new K/V rows and
    queries of each step are synthetic, so a "token" is one position of the cache.

Every manager call is made here, so a step's plan (slots, tables, lengths, query offsets, copy
pairs) is complete before the executor runs anything on the device.
"""
from __future__ import annotations

import math
from collections import deque
from dataclasses import dataclass, field

import numpy as np

from . import pkv


@dataclass
class Request:
    rid: int
    klass: str
    prompt: int                 # prompt tokens (including a shared prefix, if any)
    response: int               # tokens to emit (>= 1)
    arrival: float              # seconds on the scheduler's clock
    priority: int = 0           # larger = more important
    prefix: int | None = None   # id of a resident prefix root this request extends
    # runtime state
    state: str = "waiting"      # waiting | prefill | decode | done | rejected
    seq: int = -1               # sequence id in the block manager (a fresh one per admission)
    cached: int = 0             # positions in the cache
    alloc: int = 0              # positions with a reserved slot (cached + this step's chunk)
    target: int = 0             # positions the current prefill must reach
    generated: int = 0
    t_admit: float | None = None
    t_first: float | None = None
    token_times: list = field(default_factory=list)
    preemptions: int = 0
    error: str | None = None


@dataclass
class PrefixRoot:
    pid: int
    length: int
    seq: int
    ready: bool = False
    cached: int = 0


@dataclass
class StepPlan:
    """Everything one iteration runs. Arrays are host numpy; order matters (see StepExecutor)."""
    decode_reqs: list           # requests advancing one token
    dec_seq: np.ndarray         # int64 [n_dec]
    dec_slots: np.ndarray       # int64 [n_dec]
    dec_tables: np.ndarray      # int32 [n_dec, max_blocks]
    dec_lens: np.ndarray        # int32 [n_dec]
    pre_chunks: list            # (owner, n_tokens) owner = Request or PrefixRoot
    pre_slots: np.ndarray       # int64 [n_pre_tokens]
    pre_tables: np.ndarray      # int32 [n_pre, max_blocks]
    pre_lens: np.ndarray        # int32 [n_pre]
    pre_qs: np.ndarray          # int32 [n_pre + 1]
    pairs: np.ndarray           # int32 [n_pairs, 2] copy-on-write (src, dst), before any append
    preempted: list

    @property
    def n_dec(self) -> int:
        return len(self.dec_seq)

    @property
    def n_pre_tokens(self) -> int:
        return int(self.pre_qs[-1]) if len(self.pre_qs) else 0


class Scheduler:
    def __init__(self, mgr: pkv.BlockManager, max_batch_tokens: int = 2048, chunk: int = 512,
                 max_running: int = 256, max_blocks: int = 128, headroom_blocks: int = 1):
        self.mgr = mgr
        self.bs = mgr.block_size
        self.max_batch_tokens = int(max_batch_tokens)
        self.chunk = int(chunk)
        self.max_running = int(max_running)
        self.max_blocks = int(max_blocks)          # table width of the plans (caps context length)
        self.headroom = int(headroom_blocks)
        self.waiting: deque = deque()
        self.running: list = []                    # admitted: prefill or decode
        self.done: list = []
        self.rejected: list = []
        self.roots: dict = {}
        self._next_seq = 1 << 40                   # sequence ids of admissions (roots use their own range)
        self.preemptions = 0
        self.steps = 0
        self.prefix_forks = 0
        self.admissions = 0

    # ---- submission ---------------------------------------------------------------------
    def add_prefix(self, pid: int, length: int) -> None:
        """A shared prompt prefix of `length` tokens, prefilled once and kept resident."""
        if pid in self.roots:
            raise ValueError("prefix id in use")
        self.roots[pid] = PrefixRoot(pid, int(length), seq=-(pid + 1))

    def submit(self, r: Request) -> bool:
        """Queue a request, or refuse it at once if it can never fit ("refuse early")."""
        need = math.ceil((r.prompt + r.response) / self.bs)
        if r.response < 1 or r.prompt < 1:
            r.state, r.error = "rejected", "empty prompt or response"
        elif need > self.mgr.num_blocks - self.headroom or need > self.max_blocks:
            r.state = "rejected"
            r.error = f"needs {need} blocks; the pool has {self.mgr.num_blocks} and tables hold {self.max_blocks}"
        elif r.prefix is not None and (r.prefix not in self.roots or self.roots[r.prefix].length >= r.prompt):
            r.state, r.error = "rejected", "unknown prefix or prefix not shorter than the prompt"
        if r.state == "rejected":
            self.rejected.append(r)
            return False
        self.waiting.append(r)
        return True

    # ---- one iteration ------------------------------------------------------------------
    def _free_blocks(self) -> int:
        return self.mgr.stats()["free_blocks"]

    def _outstanding(self) -> int:
        """Blocks the admitted, still-prefilling requests will take before their prompts are in."""
        return sum(max(0, math.ceil(r.target / self.bs) - math.ceil(r.alloc / self.bs))
                   for r in self.running if r.state == "prefill")

    def _preempt_victim(self, exclude=()) -> Request | None:
        cands = [r for r in self.running if r not in exclude]
        if not cands:
            return None
        return min(cands, key=lambda r: (r.priority, -r.arrival, -r.rid))

    def _preempt(self, r: Request) -> None:
        rc = self.mgr.free_seq(r.seq)
        assert rc == pkv.PKV_OK
        self.running.remove(r)
        r.state = "waiting"
        r.cached = 0
        r.alloc = 0
        r.seq = -1
        r.preemptions += 1
        self.preemptions += 1
        # back at the head of its priority: it keeps its place ahead of later arrivals
        self.waiting.appendleft(r)

    def schedule(self, now: float) -> StepPlan:
        """Decide and reserve everything one iteration runs."""
        mgr = self.mgr
        self.steps += 1
        preempted = []
        pairs = []
        # 1. decode: one slot per running, fully prefilled request; preempt on append OOM. The
        # manager appends in order and stops at the first request it cannot serve (one C call for
        # the rest of the batch per attempt).
        dec = [r for r in self.running if r.state == "decode"]
        dec_slots = []
        i = 0
        while i < len(dec):
            rc, slots, new_pairs, n_done = mgr.append_batch([r.seq for r in dec[i:]])
            dec_slots.extend(slots.tolist())
            pairs.extend((int(s), int(d)) for s, d in new_pairs)
            i += n_done
            if rc == pkv.PKV_OK:
                continue
            if rc != pkv.PKV_ERR_NO_BLOCKS:
                raise pkv.PkvError(rc, "append_batch")
            victim = self._preempt_victim()
            # a victim that already took this step's slot gives it back with its blocks
            if victim in dec[:i]:
                j = dec.index(victim)
                del dec_slots[j]
                dec.remove(victim)
                i -= 1
            elif victim in dec:
                dec.remove(victim)
            self._preempt(victim)
            preempted.append(victim)
            # pairs of the victim's copy-on-write (if any) are dropped with it
            pairs = [p for p in pairs if mgr.refcount(p[1]) > 0]
        budget = self.max_batch_tokens - len(dec)
        # 2. prefill chunks: roots and requests already prefilling, then admissions
        chunks = []   # (owner, n, first)
        for root in self.roots.values():
            if budget <= 0:
                break
            if not root.ready and root.cached < root.length:
                n = min(self.chunk, budget, root.length - root.cached)
                if self._reserve_chunk(root.seq, root.cached == 0, n, pairs):
                    chunks.append((root, n))
                    budget -= n
        for r in [r for r in self.running if r.state == "prefill"]:
            if budget <= 0:
                break
            n = min(self.chunk, budget, r.target - r.cached)
            if n > 0 and self._reserve_chunk(r.seq, False, n, pairs):
                chunks.append((r, n))
                r.alloc = r.cached + n
                budget -= n
        order = sorted(self.waiting, key=lambda r: (-r.priority, r.arrival, r.rid))
        for r in order:
            if budget <= 0 or len(self.running) >= self.max_running:
                break
            if r.arrival > now:
                continue
            target = r.prompt + max(r.generated - 1, 0)   # a preempted request recomputes its cache
            need = math.ceil(target / self.bs) + self.headroom
            avail = self._free_blocks() - self._outstanding()
            if r.prefix is not None:
                root = self.roots[r.prefix]
                if not root.ready:
                    continue
                if need - root.length // self.bs > avail:
                    break   # blocks are the binding constraint: keep the queue order
                seq = self._new_seq()
                assert mgr.fork(root.seq, seq) == pkv.PKV_OK
                self.prefix_forks += 1
                cached = root.length
            else:
                if need > avail:
                    break
                seq = self._new_seq()
                cached = 0
            n = min(self.chunk, budget, target - cached)
            if not self._reserve_chunk(seq, cached == 0, n, pairs):
                if cached:
                    mgr.free_seq(seq)
                    self.prefix_forks -= 1
                break
            self.waiting.remove(r)
            r.seq, r.cached, r.alloc, r.target, r.state = seq, cached, cached + n, target, "prefill"
            self.admissions += 1
            if r.t_admit is None:
                r.t_admit = now
            self.running.append(r)
            chunks.append((r, n))
            budget -= n
        return self._pack(dec, dec_slots, chunks, pairs, preempted)

    def _new_seq(self) -> int:
        self._next_seq += 1
        return self._next_seq

    def _reserve_chunk(self, seq: int, first: bool, n: int, pairs: list) -> bool:
        """Blocks for the next n positions of seq (admitting it if first); slots follow from the tables."""
        if first:
            rc, _ = self.mgr.add_seq(seq, n)
            return rc == pkv.PKV_OK
        rc, _, src, dst = self.mgr.extend(seq, n)
        if rc != pkv.PKV_OK:
            return False
        if src >= 0:
            pairs.append((src, dst))
        return True

    def _width(self, ctxs) -> int:
        """Table width of a plan: the longest context's blocks, rounded up to 16 entries (the
        decode grid follows the width, so short iterations do not launch idle partitions)."""
        need = max((math.ceil(c / self.bs) for c in ctxs), default=1)
        return min(self.max_blocks, max(16, -(-need // 16) * 16))

    def _pack(self, dec, dec_slots, chunks, pairs, preempted) -> StepPlan:
        dec_seq = np.array([r.seq for r in dec], dtype=np.int64)
        rc, dec_tables, dec_lens = self.mgr.pack_tables(dec_seq, self._width([r.cached + 1 for r in dec]))
        assert rc == pkv.PKV_OK
        pre_seq = np.array([o.seq for o, _ in chunks], dtype=np.int64)
        rc, pre_tables, pre_lens = self.mgr.pack_tables(pre_seq, self._width([o.cached + n for o, n in chunks]))
        assert rc == pkv.PKV_OK
        qs = np.zeros(len(chunks) + 1, dtype=np.int32)
        qs[1:] = np.cumsum([n for _, n in chunks]) if chunks else []
        # slots of the chunk tokens: positions lens - n .. lens - 1 through the packed tables
        pre_slots = np.empty(int(qs[-1]), dtype=np.int64)
        for i, (o, n) in enumerate(chunks):
            pos = np.arange(int(pre_lens[i]) - n, int(pre_lens[i]))
            pre_slots[qs[i]: qs[i + 1]] = pre_tables[i, pos // self.bs].astype(np.int64) * self.bs + pos % self.bs
        return StepPlan(decode_reqs=dec, dec_seq=dec_seq, dec_slots=np.array(dec_slots, dtype=np.int64),
                        dec_tables=dec_tables, dec_lens=dec_lens, pre_chunks=chunks, pre_slots=pre_slots,
                        pre_tables=pre_tables, pre_lens=pre_lens, pre_qs=qs,
                        pairs=np.array(pairs, dtype=np.int32).reshape(-1, 2), preempted=preempted)

    def complete(self, plan: StepPlan, now: float) -> None:
        """Account for an executed iteration at time `now` (tokens, finishes, metrics)."""
        for r in plan.decode_reqs:
            r.cached += 1
            r.generated += 1
            r.token_times.append(now)
            if r.generated >= r.response:
                self._finish(r, now)
        for o, n in plan.pre_chunks:
            o.cached += n
            if isinstance(o, PrefixRoot):
                if o.cached >= o.length:
                    o.ready = True
                continue
            if o.cached >= o.target:
                o.state = "decode"
                if o.generated == 0:          # the prompt is in: the first token comes out now
                    o.generated = 1
                    o.t_first = now
                    o.token_times.append(now)
                    if o.generated >= o.response:
                        self._finish(o, now)

    def _finish(self, r: Request, now: float) -> None:
        assert self.mgr.free_seq(r.seq) == pkv.PKV_OK
        self.running.remove(r)
        r.state = "done"
        self.done.append(r)

    def idle(self) -> bool:
        return not self.waiting and not self.running and all(r.ready for r in self.roots.values())

    def break_stall(self) -> bool:
        """An iteration found nothing it could run while requests are admitted (every prefilling
        request is short of blocks): preempt one so the others can proceed."""
        victim = self._preempt_victim()
        if victim is None:
            return False
        self._preempt(victim)
        return True

    # ---- metrics ------------------------------------------------------------------------
    def metrics(self) -> dict:
        """Block metrics and per-class latency percentiles (seconds on the scheduler's clock)."""
        st = self.mgr.stats()
        out = {"blocks": {**st, "preemptions": self.preemptions, "prefix_forks": self.prefix_forks,
                          "prefix_hit_rate": self.prefix_forks / max(1, self.admissions)},
               "steps": self.steps, "done": len(self.done), "rejected": len(self.rejected), "classes": {}}
        classes = sorted({r.klass for r in self.done})
        for k in classes:
            rs = [r for r in self.done if r.klass == k]
            qd = [r.t_admit - r.arrival for r in rs]
            ttft = [r.t_first - r.arrival for r in rs]
            itl = [b - a for r in rs for a, b in zip(r.token_times, r.token_times[1:])]
            out["classes"][k] = {
                "n": len(rs), "tokens": int(sum(r.generated for r in rs)),
                "queue_delay_p50": _pct(qd, 50), "queue_delay_p99": _pct(qd, 99),
                "ttft_p50": _pct(ttft, 50), "ttft_p99": _pct(ttft, 99),
                "itl_p50": _pct(itl, 50), "itl_p99": _pct(itl, 99),
                "preempted": int(sum(r.preemptions for r in rs)),
            }
        return out


def _pct(xs, p):
    return float(np.percentile(xs, p)) if len(xs) else None


def synthetic_trace(n: int, seed: int, rate_per_s: float, classes=None) -> list:
    """Poisson arrivals; per class a prompt and response distribution and a priority.

    Default classes: "chat" (prompt U{64..512}, response min(Geom(1/500), 2048), the GPT-style
    mix of "Configurando as Constantes") and "doc" (a long prompt U{4096..16384}, short response
    U{16..128}, lower priority) -- a prefill-heavy class that must not starve chat.
    """
    rng = np.random.default_rng(seed)
    classes = classes or [("chat", 0.8, 1), ("doc", 0.2, 0)]
    names = [c[0] for c in classes]
    probs = np.array([c[1] for c in classes], dtype=float)
    prio = {c[0]: c[2] for c in classes}
    t = 0.0
    out = []
    for i in range(n):
        t += float(rng.exponential(1.0 / rate_per_s))
        k = names[int(rng.choice(len(names), p=probs / probs.sum()))]
        if k == "doc":
            prompt = int(rng.integers(4096, 16385))
            resp = int(rng.integers(16, 129))
        else:
            prompt = int(rng.integers(64, 513))
            resp = int(min(rng.geometric(1.0 / 500.0), 2048))
        out.append(Request(rid=i, klass=k, prompt=prompt, response=resp, arrival=t, priority=prio[k]))
    return out


def serve(sched: Scheduler, requests, execute, clock, wait_until, max_steps: int = 1_000_000) -> int:
    """Run requests to completion: submit each when the clock passes its arrival, then iterate
    schedule -> execute -> complete. `execute(plan)` runs the iteration (and must advance `clock`
    if the clock is virtual); `wait_until(t)` idles until time t. Returns the iterations run."""
    pending = sorted(requests, key=lambda r: (r.arrival, r.rid))
    i = 0
    steps = 0
    while steps < max_steps:
        now = clock()
        while i < len(pending) and pending[i].arrival <= now:
            sched.submit(pending[i])
            i += 1
        if sched.idle() and i == len(pending):
            return steps
        plan = sched.schedule(now)
        if plan.n_dec == 0 and not plan.pre_chunks:
            if sched.running and not any(r.state == "decode" for r in sched.running) and not plan.preempted:
                if sched.break_stall():
                    continue
            if i < len(pending):
                wait_until(pending[i].arrival)
                continue
            if not sched.running and not sched.waiting:
                return steps
            raise RuntimeError("no iteration can make progress")
        execute(plan)
        sched.complete(plan, clock())
        steps += 1
    raise RuntimeError("step limit reached")
