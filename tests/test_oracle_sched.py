"""Pins of the gather scheduler's oracle (oracle/sched.py): schedules
worked out by hand from the rules ([ZeRO-3 chapter] §5.1-5.3: trace
RECORD -> COMPLETE and its invalidation, fetch_sub_module's prefetch from
the parameter queue under prefetch_bucket_size and max_live_parameters,
release_sub_module's reuse distance; §6.3: the step repartitions every
parameter) and from the arena rule (a block waits for the latest release
of the space it takes; the placement with the oldest such release, then the
lowest offset, wins).  Each golden log below was derived on paper, step by
step, before it was compared with the oracle; mutants of the oracle must
fail one of them.

The model: N = 2, nothing persistent, numel 100, 200, 300, 400 (partition
sizes 50, 100, 150, 200, so each parameter takes numel elements of arena);
modules M0 = [p0], M1 = [p1, p2], M2 = [p3], M3 = [p0] (p0 used again at
the end, as a tied weight would be), fetched in the order 0, 1, 2, 3.

Log records: ("G", position, op, ((param, offset), ...), release waited)
for a gather, ("W", position, ops) for the compute's waits, ("R", position,
release index, params) for a release (position 4 = the end of the pass)."""
from __future__ import annotations

import pytest

from oracle import plan as oplan
from oracle import sched as osched

NUMEL = [100, 200, 300, 400]
MODS = [[0], [1, 2], [3], [0]]


def _plan():
    return oplan.build_partition(NUMEL, 2, threshold=0)


def _compact(log):
    out = []
    for e in log:
        if e[0] == "gather":
            _, op, pos, items, waits = e
            out.append(("G", pos, op, tuple((p, o) for p, o in items), waits))
        elif e[0] == "wait":
            out.append(("W", e[1], tuple(e[2])))
        else:
            out.append(("R", e[1], e[2], tuple(e[3])))
    return out


def _run(cfg, orders):
    s = osched.Scheduler(_plan(), MODS, osched.SchedConfig(**cfg))
    for order in orders:
        for m in order:
            s.fetch(m)
            s.release(m)
        s.end_pass()
    return s


SMALL_ARENA = dict(prefetch_bucket_size=1000, max_live_parameters=10**9, max_reuse_distance=0,
                   arena_elems=600)

# Worked by hand.  Pass 1 records the trace: no prefetch, every parameter
# released after its module.  The arena holds 600 elements, so later blocks
# reuse released space and wait for the release that freed it; a block may
# span two segments (op 2, op 5); equal waits go to the lower offset (op 2).
GOLDEN_SMALL_ARENA = [
    # pass 1 (RECORD)
    ("G", 0, 0, ((0, 0),), -1), ("W", 0, (0,)), ("R", 0, 0, (0,)),
    # [0,100) freed by release 0 vs never-used [100,600): the never-used wins
    ("G", 1, 1, ((1, 100), (2, 300)), -1), ("W", 1, (1,)), ("R", 1, 1, (1, 2)),
    # free: [0,100) rel 0, [100,600) rel 1 -> 400 at 0 (waits max(0,1) = 1)
    # or at 100 (waits 1): the lower offset
    ("G", 2, 2, ((3, 0),), 1), ("W", 2, (2,)), ("R", 2, 2, (3,)),
    # free: [0,400) rel 2, [400,600) rel 1 -> 100 at 400, waits 1
    ("G", 3, 3, ((0, 400),), 1), ("W", 3, (3,)), ("R", 3, 3, (0,)),
    ("R", 4, 4, ()),
    # pass 2 (COMPLETE): free [0,400) rel 2, [400,500) rel 3, [500,600) rel 1
    ("G", 0, 4, ((0, 500),), 1), ("W", 0, (4,)),
    # prefetch M1 (both parameters, one gather) into [0,500): waits 3; M2's
    # p3 does not fit the arena, which ends the walk
    ("G", 0, 5, ((1, 0), (2, 200)), 3),
    # p0 is used again at M3, 900 elements later > max_reuse_distance 0
    ("R", 0, 5, (0,)),
    # the walk resumes at p3, which still does not fit
    ("W", 1, (5,)), ("R", 1, 6, (1, 2)),
    # free: [0,500) rel 6, [500,600) rel 5: p3's fetch gathers it itself
    ("G", 2, 6, ((3, 0),), 6), ("W", 2, (6,)),
    # then prefetches M3's p0: [400,500) rel 6 vs [500,600) rel 5 -> 500
    ("G", 2, 7, ((0, 500),), 5), ("R", 2, 7, (3,)),
    ("W", 3, (7,)), ("R", 3, 8, (0,)),
    ("R", 4, 9, ()),
]

BIG = dict(prefetch_bucket_size=1000, max_live_parameters=10**9, max_reuse_distance=0,
           arena_elems=10000)


def test_golden_small_arena():
    s = _run(SMALL_ARENA, [[0, 1, 2, 3]] * 2)
    assert _compact(s.log) == GOLDEN_SMALL_ARENA


def _shape(log):
    """The log without arena offsets and waits."""
    out = []
    for e in _compact(log):
        if e[0] == "G":
            out.append(("G", e[1], e[2], tuple(p for p, _ in e[3])))
        else:
            out.append(e)
    return out


PASS1 = [("G", 0, 0, (0,)), ("W", 0, (0,)), ("R", 0, 0, (0,)),
         ("G", 1, 1, (1, 2)), ("W", 1, (1,)), ("R", 1, 1, (1, 2)),
         ("G", 2, 2, (3,)), ("W", 2, (2,)), ("R", 2, 2, (3,)),
         ("G", 3, 3, (0,)), ("W", 3, (3,)), ("R", 3, 3, (0,)),
         ("R", 4, 4, ())]


def test_golden_prefetch_one_gather_per_module():
    """A big arena: at M0's fetch the walk takes M1 (one gather of p1, p2)
    and M2 (a second gather); p0 at M3 is live then, so it is skipped and
    not taken again: M3's fetch gathers it itself."""
    s = _run(BIG, [[0, 1, 2, 3]] * 2)
    assert _shape(s.log) == PASS1 + [
        ("G", 0, 4, (0,)), ("W", 0, (4,)), ("G", 0, 5, (1, 2)), ("G", 0, 6, (3,)),
        ("R", 0, 5, (0,)),
        ("W", 1, (5,)), ("R", 1, 6, (1, 2)),
        ("W", 2, (6,)), ("R", 2, 7, (3,)),
        ("G", 3, 7, (0,)), ("W", 3, (7,)), ("R", 3, 8, (0,)),
        ("R", 4, 9, ())]
    # never-used space first: no gather of the big arena waits
    assert all(e[4] == -1 for e in _compact(s.log) if e[0] == "G")


def test_golden_max_live_parameters():
    """max_live_parameters 600.  At M0's fetch 100 elements are live, so the
    walk may add while below 500: p1 (200) and p2 (500 in all), then stops.
    At M1's fetch 500 are live (p1, p2): below 100 it takes p3 (the last one
    may cross the cap).  At M2's fetch p1, p2 are released: p0 for M3."""
    s = _run(dict(BIG, max_live_parameters=600), [[0, 1, 2, 3]] * 2)
    assert _shape(s.log) == PASS1 + [
        ("G", 0, 4, (0,)), ("W", 0, (4,)), ("G", 0, 5, (1, 2)), ("R", 0, 5, (0,)),
        ("W", 1, (5,)), ("G", 1, 6, (3,)), ("R", 1, 6, (1, 2)),
        ("W", 2, (6,)), ("G", 2, 7, (0,)), ("R", 2, 7, (3,)),
        ("W", 3, (7,)), ("R", 3, 8, (0,)),
        ("R", 4, 9, ())]


def test_golden_reuse_distance_keeps_a_parameter():
    """max_reuse_distance 900: p0's next use (M3) is 200 + 300 + 400 = 900
    elements of parameter uses away, so M0's release keeps it and M3 waits
    for the gather of pass 2's first fetch.  The recording pass releases
    everything (the distance rule needs a complete trace)."""
    s = _run(dict(BIG, max_reuse_distance=900), [[0, 1, 2, 3]] * 2)
    assert _shape(s.log) == PASS1 + [
        ("G", 0, 4, (0,)), ("W", 0, (4,)), ("G", 0, 5, (1, 2)), ("G", 0, 6, (3,)),
        ("R", 0, 5, ()),
        ("W", 1, (5,)), ("R", 1, 6, (1, 2)),
        ("W", 2, (6,)), ("R", 2, 7, (3,)),
        ("W", 3, (4,)), ("R", 3, 8, (0,)),
        ("R", 4, 9, ())]
    # one element less and p0 is released at M0 again
    s = _run(dict(BIG, max_reuse_distance=899), [[0, 1, 2, 3]] * 2)
    assert ("R", 0, 5, (0,)) in _shape(s.log)


def test_golden_trace_invalidation():
    """Pass 2 departs from the trace at its second fetch (M2 instead of M1):
    no prefetch from there on, and no reuse-distance rule; the end of the
    pass drops the trace, so pass 3 records again (no prefetch at all)."""
    s = _run(BIG, [[0, 1, 2, 3], [0, 2, 1, 3], [0, 1, 2, 3]])
    assert _shape(s.log) == PASS1 + [
        ("G", 0, 4, (0,)), ("W", 0, (4,)), ("G", 0, 5, (1, 2)), ("G", 0, 6, (3,)),
        ("R", 0, 5, (0,)),
        ("W", 1, (6,)), ("R", 1, 6, (3,)),
        ("W", 2, (5,)), ("R", 2, 7, (1, 2)),
        ("G", 3, 7, (0,)), ("W", 3, (7,)), ("R", 3, 8, (0,)),
        ("R", 4, 9, ()),
        # pass 3 records anew
        ("G", 0, 8, (0,)), ("W", 0, (8,)), ("R", 0, 10, (0,)),
        ("G", 1, 9, (1, 2)), ("W", 1, (9,)), ("R", 1, 11, (1, 2)),
        ("G", 2, 10, (3,)), ("W", 2, (10,)), ("R", 2, 12, (3,)),
        ("G", 3, 11, (0,)), ("W", 3, (11,)), ("R", 3, 13, (0,)),
        ("R", 4, 14, ())]


def test_end_of_pass_releases_what_is_kept():
    """A parameter kept by the reuse distance past its last use in the
    trace would stay live; the end of the pass releases it (the step
    repartitions every parameter)."""
    mods = [[0], [1], [0]]
    s = osched.Scheduler(_plan(), mods, osched.SchedConfig(**dict(BIG, max_reuse_distance=10**9)))
    for _ in range(2):
        for m in (0, 1, 2):
            s.fetch(m)
            s.release(m)
        s.end_pass()
    rel = [e for e in _compact(s.log) if e[0] == "R"]
    # pass 2: M0 keeps p0 (used again at position 2), M1 releases p1,
    # position 2 releases p0 (no later use), the end releases nothing left
    assert rel[-4:] == [("R", 0, 4, ()), ("R", 1, 5, (1,)), ("R", 2, 6, (0,)), ("R", 3, 7, ())]
    assert not s.status


def test_current_fetch_that_does_not_fit_is_an_error():
    s = osched.Scheduler(_plan(), MODS, osched.SchedConfig(**dict(SMALL_ARENA, arena_elems=450)))
    s.fetch(0)
    s.release(0)
    with pytest.raises(osched.ArenaFull):
        s.fetch(1)                      # p1 + p2 = 500 elements > 450


def test_library_reproduces_the_golden_logs():
    """The C++ scheduler (plan-only mode) gives the hand-derived logs."""
    zs = pytest.importorskip("zero_sharded_optimizer_bucket_gb300")
    from tests.test_sched_host import _oracle_records
    cfg_c = zs.zs_default_config(2)
    cfg_c.param_persistence_threshold = 0
    plan_c = zs.zs_build_partition(cfg_c, NUMEL)
    for cfg, orders in ((SMALL_ARENA, [[0, 1, 2, 3]] * 2),
                        (BIG, [[0, 1, 2, 3], [0, 2, 1, 3], [0, 1, 2, 3]]),
                        (dict(BIG, max_live_parameters=600), [[0, 1, 2, 3]] * 2)):
        c = zs.zs_sched_create(plan_c, MODS, cfg)
        for order in orders:
            for m in order:
                zs.zs_sched_fetch(c, m)
                zs.zs_sched_release(c, m)
            zs.zs_sched_end_pass(c)
        assert zs.zs_sched_log(c) == _oracle_records(_run(cfg, orders).log)


# ------------------------------------------------------------- mutants ---
def _mut_prefetch_ignores_max_live(orig):
    import dataclasses

    def bad(self, pos):
        keep = self.cfg
        self.cfg = dataclasses.replace(keep, max_live_parameters=10**18)
        try:
            orig(self, pos)
        finally:
            self.cfg = keep
    return bad


def _mut_release_ignores_reuse(orig):
    return lambda self, p, pos: False


def _mut_reuse_strict(orig):
    def bad(self, p, pos):
        dist = 0
        for k in range(pos + 1, len(self.trace)):
            ps = self.modules[self.trace[k]]
            if p in ps:
                return dist < self.cfg.max_reuse_distance
            dist += sum(self.plan.params[q].numel for q in ps)
        return False
    return bad


def _mut_no_invalidation(orig):
    def bad(self, m):
        orig(self, m)
        self.invalid = False
    return bad


def _mut_first_fit(orig):
    def bad(self, params):
        srt = sorted(params, key=lambda i: self.plan.params[i].ds_id)
        total = sum(self._size(p) for p in srt)
        for i in range(len(self.free)):
            acc, wait = 0, -1
            for j in range(i, len(self.free)):
                if j > i and self.free[j - 1][0] + self.free[j - 1][1] != self.free[j][0]:
                    break
                acc += self.free[j][1]
                wait = max(wait, self.free[j][2])
                if acc >= total:
                    off, rest, rel_j = self.free[i][0], acc - total, self.free[j][2]
                    self.free[i:j + 1] = [(off + total, rest, rel_j)] if rest > 0 else []
                    offs, run = {}, off
                    for p in srt:
                        offs[p] = run
                        run += self._size(p)
                    return offs, wait
        return None
    return bad


def _mut_merge_keeps_later_release(orig):
    def bad(self, p, rel):
        off, size = self.offset.pop(p), self._size(p)
        merged = []
        for s in sorted(self.free + [(off, size, rel)]):
            if merged and merged[-1][0] + merged[-1][1] == s[0]:
                a = merged[-1]
                merged[-1] = (a[0], a[1] + s[1], max(a[2], s[2]))
            else:
                merged.append(s)
        self.free = merged
    return bad


def _mut_one_prefetch_gather(orig):
    def bad(self, pos):
        queue = self._queue()
        start = sum(len(self.modules[self.trace[k]]) for k in range(pos + 1))
        self.queue_pos = max(self.queue_pos, start)
        cap = min(self.cfg.prefetch_bucket_size, self.cfg.max_live_parameters - self.live)
        group, added = [], 0
        while self.queue_pos < len(queue) and added < cap:
            k, p = queue[self.queue_pos]
            if not self._gatherable(p) or p in self.status or p in group:
                self.queue_pos += 1
                continue
            if self._alloc_probe(group + [p]) is None:
                break
            group.append(p)
            added += self.plan.params[p].numel
            self.queue_pos += 1
        self._gather(group, pos, False)
    return bad


def _mut_walk_restarts(orig):
    def bad(self, pos):
        self.queue_pos = 0
        orig(self, pos)
    return bad


# name: (Scheduler attribute replaced, factory(original) -> replacement, pin)
MUTANTS = {
    "prefetch ignores max_live_parameters": ("_prefetch", _mut_prefetch_ignores_max_live,
                                             test_golden_max_live_parameters),
    "release ignores the reuse distance": ("_reused_soon", _mut_release_ignores_reuse,
                                           test_golden_reuse_distance_keeps_a_parameter),
    "reuse distance compared with <": ("_reused_soon", _mut_reuse_strict,
                                       test_golden_reuse_distance_keeps_a_parameter),
    "no trace invalidation": ("fetch", _mut_no_invalidation, test_golden_trace_invalidation),
    "first-fit placement": ("_alloc", _mut_first_fit, test_golden_small_arena),
    "free segments merged keeping the later release": ("_free", _mut_merge_keeps_later_release,
                                                       test_golden_small_arena),
    "one prefetch gather for all modules": ("_prefetch", _mut_one_prefetch_gather,
                                            test_golden_prefetch_one_gather_per_module),
    "prefetch walk goes back": ("_prefetch", _mut_walk_restarts,
                                test_golden_prefetch_one_gather_per_module),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pin_catches_planted_scheduler_mistake(monkeypatch, name):
    attr, factory, pin = MUTANTS[name]
    monkeypatch.setattr(osched.Scheduler, attr, factory(getattr(osched.Scheduler, attr)))
    with pytest.raises(AssertionError):
        pin()
