"""Prefetch / release scheduling of the forward and backward gathers: the
oracle's statement of the rules ([ZeRO-3 chapter] §5.1-5.3, §6.3, §7).
TEST INFRASTRUCTURE, like the rest of `oracle`.

A model is a list of modules, each using a list of parameters.  A pass
fetches modules in some order; each fetch is followed by the module's
compute and its release.  Readings of the pages (each a choice where the
pages only name the mechanism):

* Trace.  The first pass records the module order (RECORD); at the end of
  that pass the trace is COMPLETE and later passes prefetch from it.  A fetch
  that does not match the trace's next module invalidates the trace: no more
  prefetching in that pass, and the next pass records again (§5.1,
  trace_prologue; §7 first bullet).  A pass that ends early also invalidates.
* Fetch (§5.2 fetch_sub_module).  (1) The module's parameters that are not
  available and not in flight are gathered now, as one coalesced gather; (2)
  the compute waits for every gather that produces one of its parameters;
  (3) with a COMPLETE trace, prefetch: walk the parameter queue (every
  (position, parameter) use of the trace after the current position, in
  order), skipping parameters already available / in flight and persistent
  ones, gathering the others while the elements added so far are below
  min(prefetch_bucket_size, max_live_parameters - live elements), one
  coalesced gather per module of the trace reached (so a compute waits only
  for its own module's gather); a parameter that would not fit the arena
  ends the walk.  The
  walk resumes where it stopped at the next fetch (it never goes back
  before the next module's entries).
* Release (§5.3 release_sub_module, __params_to_release).  After the
  compute, each of the module's parameters is released unless it is
  persistent, or it is used again later in the trace (COMPLETE mode only)
  with a reuse distance — the elements of the parameter uses between now and
  that next use — of at most max_reuse_distance.
* End of a pass.  All gathered parameters are released: the optimizer step
  repartitions everything ([ZeRO-3 chapter] §6.3, _partition_all_parameters).
* Live elements count numel of the available or in-flight parameters
  (max_live_parameters, §5.3).  Persistent parameters are never gathered.
* Arena.  A gather takes one contiguous block of G*ps elements per
  parameter, laid out as zs_all_gather_coalesced lays them (running sums in
  ds_id order).  Free space is kept as segments tagged with the release that
  freed them (neighbours merge only when freed by the same release); a
  block may span adjacent segments and then waits for the latest of their
  releases; the placement with the oldest such release (never-used space
  first), then the lowest offset, is taken, so that a prefetch seldom waits
  for a recent compute.  A current fetch that does not fit is an error.

The log is a list of tuples:
  ("gather", op, module_pos, [(param, offset)...], wait_release)  wait_release
        is the index of the release event to wait for, or -1
  ("wait", module_pos, [op...])    the compute waits for these gathers
  ("release", module_pos, release_idx, [param...])
"""
from __future__ import annotations

from dataclasses import dataclass, field

from .plan import Plan


@dataclass
class SchedConfig:
    prefetch_bucket_size: int = 50_000_000
    max_live_parameters: int = 1_000_000_000
    max_reuse_distance: int = 1_000_000_000
    arena_elems: int = 0


class ArenaFull(Exception):
    pass


@dataclass
class Scheduler:
    plan: Plan
    modules: list                      # module id -> list of parameter indices
    cfg: SchedConfig
    trace: list = field(default_factory=list)
    complete: bool = False
    invalid: bool = False
    pos: int = 0
    queue_pos: int = 0                  # index into the queue of the current trace
    status: dict = field(default_factory=dict)    # param -> "inflight"
    offset: dict = field(default_factory=dict)    # param -> arena offset
    producer: dict = field(default_factory=dict)  # param -> gather op
    free: list = field(default_factory=list)      # [(off, size, release_idx)] sorted
    live: int = 0
    ops: int = 0
    releases: int = 0
    log: list = field(default_factory=list)
    recording: list = field(default_factory=list)

    def __post_init__(self):
        self.free = [(0, self.cfg.arena_elems, -1)] if self.cfg.arena_elems > 0 else []

    # ---------------------------------------------------------- helpers ---
    def _size(self, p):
        q = self.plan.params[p]
        return self.plan.group * q.ps

    def _gatherable(self, p):
        q = self.plan.params[p]
        return not q.persistent and q.ps > 0

    def _queue(self):
        return [(k, p) for k, m in enumerate(self.trace) for p in self.modules[m]]

    def _alloc(self, params):
        """One block for the params in ds_id order.  Free space is a sorted
        list of segments, each with the release that freed it; a block may
        span adjacent segments and waits for the latest release among them.
        The placement chosen has the oldest such release (never-used space
        first), then the lowest offset.  Returns (offsets, wait_release) or
        None."""
        srt = sorted(params, key=lambda i: self.plan.params[i].ds_id)
        total = sum(self._size(p) for p in srt)
        best = None
        n = len(self.free)
        for i in range(n):
            acc, wait = 0, -1
            for j in range(i, n):
                off_j, size_j, rel_j = self.free[j]
                if j > i and self.free[j - 1][0] + self.free[j - 1][1] != off_j:
                    break
                acc += size_j
                wait = max(wait, rel_j)
                if acc >= total:
                    cand = (wait, self.free[i][0], i, j, acc)
                    if best is None or cand[:2] < best[:2]:
                        best = cand
                    break
        if best is None:
            return None
        wait, off, i, j, acc = best
        rest = acc - total
        rel_j = self.free[j][2]
        self.free[i:j + 1] = [(off + total, rest, rel_j)] if rest > 0 else []
        offs, run = {}, off
        for p in srt:
            offs[p] = run
            run += self._size(p)
        return offs, wait

    def _free(self, p, rel):
        off, size = self.offset.pop(p), self._size(p)
        segs = sorted(self.free + [(off, size, rel)])
        merged = []
        for s in segs:            # merge neighbours freed by the same release
            if merged and merged[-1][0] + merged[-1][1] == s[0] and merged[-1][2] == s[2]:
                a = merged[-1]
                merged[-1] = (a[0], a[1] + s[1], a[2])
            else:
                merged.append(s)
        self.free = merged

    def _gather(self, params, module_pos, must_fit):
        if not params:
            return None
        got = self._alloc(params)
        if got is None:
            if must_fit:
                raise ArenaFull(params)
            return None
        offs, waits = got
        op = self.ops
        self.ops += 1
        srt = sorted(params, key=lambda i: self.plan.params[i].ds_id)
        for p in srt:
            self.status[p] = "inflight"
            self.offset[p] = offs[p]
            self.producer[p] = op
            self.live += self.plan.params[p].numel
        self.log.append(("gather", op, module_pos, [(p, offs[p]) for p in srt], waits))
        return op

    # ------------------------------------------------------------- API ----
    def fetch(self, m: int):
        pos = self.pos
        self.pos += 1
        if self.complete and not self.invalid:
            if pos >= len(self.trace) or self.trace[pos] != m:
                self.invalid = True
        if not self.complete and not self.invalid:
            self.recording.append(m)
        need = [p for p in dict.fromkeys(self.modules[m])
                if self._gatherable(p) and p not in self.status]
        self._gather(need, pos, True)
        ops = sorted({self.producer[p] for p in self.modules[m] if p in self.producer})
        self.log.append(("wait", pos, ops))
        if self.complete and not self.invalid:
            self._prefetch(pos)

    def _prefetch(self, pos):
        queue = self._queue()
        start = sum(len(self.modules[self.trace[k]]) for k in range(pos + 1))
        self.queue_pos = max(self.queue_pos, start)
        cap = min(self.cfg.prefetch_bucket_size, self.cfg.max_live_parameters - self.live)
        group, gpos, added = [], -1, 0
        while self.queue_pos < len(queue) and added < cap:
            k, p = queue[self.queue_pos]
            if not self._gatherable(p) or p in self.status or p in group:
                self.queue_pos += 1
                continue
            if group and k != gpos:          # one coalesced gather per module reached
                self._gather(group, pos, False)
                group = []
            if self._alloc_probe(group + [p]) is None:
                break
            group.append(p)
            gpos = k
            added += self.plan.params[p].numel
            self.queue_pos += 1
        self._gather(group, pos, False)

    def _alloc_probe(self, params):
        saved = list(self.free)
        got = self._alloc(params)
        self.free = saved
        return got

    def release(self, m: int):
        pos = self.pos - 1
        rel = self.releases
        self.releases += 1
        out = []
        for p in dict.fromkeys(self.modules[m]):
            if p not in self.status:
                continue
            if self.complete and not self.invalid and self._reused_soon(p, pos):
                continue
            self._drop(p, rel)
            out.append(p)
        self.log.append(("release", pos, rel, out))

    def _drop(self, p, rel):
        del self.status[p]
        self.producer.pop(p, None)
        self.live -= self.plan.params[p].numel
        self._free(p, rel)

    def _reused_soon(self, p, pos):
        dist = 0
        for k in range(pos + 1, len(self.trace)):
            ps = self.modules[self.trace[k]]
            if p in ps:
                return dist <= self.cfg.max_reuse_distance
            dist += sum(self.plan.params[q].numel for q in ps)
        return False

    def end_pass(self):
        rel = self.releases
        self.releases += 1
        out = sorted(self.status, key=lambda i: self.plan.params[i].ds_id)
        for p in out:
            self._drop(p, rel)
        self.log.append(("release", self.pos, rel, out))
        if self.complete and not self.invalid and self.pos != len(self.trace):
            self.invalid = True
        if not self.complete and not self.invalid:
            self.trace, self.complete = list(self.recording), True
        elif self.invalid:
            self.trace, self.complete, self.invalid = [], False, False
        self.recording = []
        self.pos = 0
        self.queue_pos = 0
