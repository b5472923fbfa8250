"""Host logic of bench.py: the max-over-ranks aggregation of a replicated
run (gloo, world size 2, CPU), argument rules, and the oracle arm's JSON."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

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
    idx = bench._sample_params(w)
    tot = sum(w.numel[i] for i in idx)
    assert 4_000_000 <= tot <= 16_000_000 and all(w.numel[i] <= 8_000_000 for i in idx)


@pytest.mark.slow
def test_reference_arm_json_tiny():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    d = json.loads(out.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
