"""Host logic of bench.py: the max-over-ranks aggregation of a replicated
run (gloo, world size 2, CPU), argument rules, and the oracle arm's JSON."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_setup()
    m = bench.max_over_ranks(10.0 + 5 * rank, w)
    bench.barrier(w)
    q.put((r, w, lr, m))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]


def test_warmup_rule():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.main(["--warmup", "2", "--steps", "1"]) == 2


def test_sample_is_bounded():
    sys.path.insert(0, ROOT)
    import bench
    from synth import workloads
    w = workloads.llama3_8b()
    idx = bench.oracle_sample(w)
    assert [w.names[i] for i in idx][0] == "layers.0.q_proj"
    assert sum(w.numel[i] for i in idx) == 218_112_000         # one whole decoder layer
    idx = bench.oracle_sample(w, target=50_000_000)
    assert all(w.numel[i] <= 50_000_000 for i in idx) and sum(w.numel[i] for i in idx) < 5e7
    w = workloads.many_small()
    assert 218_112_000 <= sum(w.numel[i] for i in bench.oracle_sample(w)) < 220_000_000


def test_split_elements_covers_every_element_once():
    sys.path.insert(0, ROOT)
    import bench
    rng = np.random.default_rng(3)
    for _ in range(50):
        numels = [int(x) for x in rng.integers(0, 1000, size=int(rng.integers(0, 12)))]
        P = int(rng.integers(1, 9))
        parts = bench.split_elements(numels, P)
        assert len(parts) == P
        flat = [n for part in parts for n in part]
        assert sum(flat) == sum(numels) and all(n >= 0 for n in flat)
        sizes = [sum(part) for part in parts]
        assert max(sizes, default=0) - min(sizes, default=0) <= 1
        # the pieces are the parameters cut at the part boundaries, in order
        cuts = np.cumsum([0] + [n for n in numels if n])
        edges = np.cumsum([0] + [n for n in flat if n])
        assert set(cuts.tolist()) <= set(edges.tolist())


def test_parallel_oracle_step_uses_the_global_norm():
    """The oracle's step on 2 host processes: the norm the parent forms from
    the processes' counts is the norm of both processes' reduced gradients
    together, computed here in one process from the same inputs."""
    sys.path.insert(0, ROOT)
    import bench
    from oracle import step as ostep
    from synth import workloads
    w = workloads.tiny(threshold=100)
    w.max_norm = 0.05
    idx = bench.oracle_sample(w)
    cl = bench.OracleCluster(w, idx, [None, None])
    try:
        got = cl.step()
    finally:
        cl.close()
    sq = 0.0
    counts = np.zeros(1 << 15, dtype=np.int64)
    for spec in bench.part_specs(w, idx, 2):
        plan, st, bufs = bench._oracle_part(spec)
        for b in range(len(plan.reduce_buckets)):
            ostep.reduce_scatter(plan, b, bufs[b], st)
        x = np.concatenate([ostep.to_f32(st.grad_shards).ravel(),
                            ostep.to_f32(st.persist_grads).ravel()]).astype(np.float64)
        sq += float(np.sum(x * x))
        counts += bench._part_counts(plan, st)
    ref = ostep.clip_from_sumsq(ostep.sumsq_from_counts(counts), w.max_norm)
    assert got[2] is False and got[1] < 1.0
    assert np.float32(got[0]).tobytes() == np.float32(ref[0]).tobytes()
    assert np.float32(got[1]).tobytes() == np.float32(ref[1]).tobytes()
    assert abs(float(got[0]) - np.sqrt(sq)) <= 1e-6 * np.sqrt(sq)


@pytest.mark.slow
def test_reference_arm_json_tiny():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    d = json.loads(out.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
