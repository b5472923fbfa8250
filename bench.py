#!/usr/bin/env python3
"""Benchmark of the ZeRO-3 per-step shard data path (libzs) on GB300.

One step = reduce-scatter of every bucket of N virtual ranks (with the norm
partial sums) -> global norm and clip coefficient -> Adam(W) + bf16 cast of
every shard element -> the gathered parameters written into model flat
space; all gradients resident in HBM before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the CPU oracle, same metric

Prints one JSON line (rank 0).  With --gpus N > 1 (torchrun, one process
per GPU) every GPU runs its own complete replica of the workload: the path
has no exchange between GPUs (the N virtual ranks live in one GPU's HBM),
so the job's throughput is the sum of the replicas' and scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ZeRO-3 shard step: params/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
DEFAULT_WORKLOAD = "llama3_8b"
KERNELS_PER_STEP = 4   # reduce-scatter (all buckets), norm level 1, norm finish, Adam+gather


def _align8(x: int) -> int:
    return (x + 7) // 8 * 8


def load_workload(name: str):
    from synth import workloads
    return workloads.WORKLOADS[name]()


# ------------------------------------------------------------- device -----
class DeviceWorkload:
    """All buffers of one workload on one GPU, inputs resident.

    Gradients: rank k's buffer of bucket b is a view into one gradient pool
    filled by the synthetic generator (synth.gpu); pool_offsets lays the
    buffers out one after another and wraps when the pool is smaller than a
    whole step's gradients (the reuse distance is then the full pool, far
    above the 129 MB L2, so every read comes from HBM).
    """

    def __init__(self, w, device="cuda:0", max_norm=None, pool_elems=None, seed=None):
        import torch

        import zero_sharded_optimizer_bucket_gb300 as zs
        from synth import gpu as sg
        from synth import workloads as wl

        self.torch, self.zs, self.w = torch, zs, w
        self.dev = torch.device(device)
        self.seed = w.seed if seed is None else seed
        self.max_norm = w.max_norm if max_norm is None else max_norm
        cfg = zs.zs_default_config(w.n_ranks)
        cfg.param_persistence_threshold = w.persistence_threshold
        cfg.reduce_bucket_size = w.reduce_bucket_size
        cfg.prefetch_bucket_size = w.prefetch_bucket_size
        cfg.sub_group_size = w.sub_group_size
        self.fp16 = w.dtype == "fp16"
        cfg.dtype = zs.ZS_DTYPE_FP16 if self.fp16 else zs.ZS_DTYPE_BF16
        cfg.shard_group_size = w.shard_group_size
        self.plan = zs.zs_build_partition(cfg, w.numel, w.ds_id)
        info = self.info = zs.zs_plan_info(self.plan)
        N, S, Pn = info["n_ranks"], info["shard_elems"], info["persist_elems"]
        self.N = N
        R = info["shard_group_size"]     # rows of shard space (N unless HSDP)
        E = lambda n, dt: torch.empty(max(int(n), 8), dtype=dt, device=self.dev)
        self.table = E(info["device_table_bytes"], torch.uint8)
        zs.zs_plan_upload(self.plan, self.table, self.table.numel())
        self.gs, self.ps = E(R * S, torch.int16), E(R * S, torch.int16)
        self.master, self.m, self.v = (E(R * S, torch.float32) for _ in range(3))
        self.gP, self.pP = E(Pn, torch.int16), E(Pn, torch.int16)
        self.pm, self.pmm, self.pmv = (E(Pn, torch.float32) for _ in range(3))
        self.state = zs.make_state(grad_shards=self.gs, param_shards=self.ps, master=self.master,
                                   exp_avg=self.m, exp_avg_sq=self.v, persist_grads=self.gP,
                                   persist_params=self.pP, p_master=self.pm, p_exp_avg=self.pmm,
                                   p_exp_avg_sq=self.pmv)
        self.scratch = E(info["norm_scratch_elems"], torch.float64)
        self.d_norm = torch.zeros(8, dtype=torch.float32, device=self.dev)
        self.d_coef = torch.zeros(8, dtype=torch.float32, device=self.dev)
        self.d_flags = torch.zeros(8, dtype=torch.int32, device=self.dev)
        self.flat = E(info["flat_elems"], torch.int16)
        self.hp = w.hparams()
        self.t = 0
        # fp16: device-resident dynamic loss scale
        self.d_scale = torch.tensor([w.loss_scale, 0, 0, 0], dtype=torch.float32, device=self.dev)
        self.d_good = torch.zeros(4, dtype=torch.int32, device=self.dev)
        self.scaler = zs.make_loss_scaler(self.d_scale, self.d_good, 2.0, 1.0, w.scale_window)
        # weights: full fp32 parameters from the generator, partitioned once
        W = E(info["psi"], torch.float32)
        sg.fill_weight_f32(W, 0, self.seed, w.weight_sigma)
        zs.zs_partition(self.plan, W, self.state)
        torch.cuda.synchronize(self.dev)
        del W
        # gradient pool
        nb = info["n_reduce_buckets"]
        self.buf_elems = [zs.zs_bucket_info(self.plan, b)["buf_elems"] for b in range(nb)]
        total = sum(N * wl.pool_align(L) for L in self.buf_elems)
        if pool_elems is None:
            free = torch.cuda.mem_get_info(self.dev)[0]
            cap = max((free - (6 << 30)) // 2, 0)
            pool_elems = min(total, cap)
        need = (N + 1) * wl.pool_align(max(self.buf_elems, default=8))
        pool_elems = max(int(pool_elems), min(need, total) if total else 8)
        if total and pool_elems < total:
            pool_elems = max(pool_elems, need)
        self.pool = E(pool_elems, torch.int16)
        if self.fp16:
            sg.fill_grad_fp16(self.pool, 0, self.seed, w.fp16_log2_scale)
        else:
            sg.fill_grad_bf16(self.pool, 0, self.seed, w.grad_sigma, w.outlier_frac,
                              w.outlier_scale)
        self.pool_elems = self.pool.numel()
        self.offs = wl.pool_offsets(self.buf_elems, N, self.pool_elems) if nb else []
        base = self.pool.data_ptr()
        flat_ptrs = [base + 2 * o for row in self.offs for o in row]
        self.ptr_table = torch.tensor(flat_ptrs or [0], dtype=torch.int64, device=self.dev)
        torch.cuda.synchronize(self.dev)

    # host-side view of rank pointers of one bucket
    def bucket_ptrs(self, b):
        base = self.pool.data_ptr()
        return [base + 2 * o for o in self.offs[b]]

    def step(self, stream=None):
        self.t += 1
        if self.fp16:
            self.zs.zs_shard_step_scaled(self.plan, self.ptr_table, self.state, self.scratch,
                                         self.hp, self.t, self.max_norm, self.scaler, self.d_norm,
                                         self.d_coef, self.d_flags, self.flat, stream)
            return
        self.zs.zs_shard_step(self.plan, self.ptr_table, self.state, self.scratch, self.hp, self.t,
                              self.max_norm, self.d_norm, self.d_coef, self.d_flags, self.flat,
                              stream)

    def norm(self, recompute=False):
        if self.fp16:
            self.zs.zs_unscale_and_clip(self.plan, self.gs, self.gP, self.scratch, recompute,
                                        self.max_norm, self.scaler, self.d_norm, self.d_coef,
                                        self.d_flags)
        else:
            self.zs.zs_grad_norm(self.plan, self.gs, self.gP, self.scratch, recompute,
                                 self.max_norm, self.d_norm, self.d_coef, self.d_flags)

    def step_timed(self, ev):
        """The same step as step(), as its three calls with events between."""
        zs = self.zs
        self.t += 1
        ev[0].record()
        zs.zs_reduce_scatter_all(self.plan, self.ptr_table, self.gs, self.gP, self.scratch)
        ev[1].record()
        self.norm()
        ev[2].record()
        zs.zs_adam_gather(self.plan, self.hp, self.t, self.d_coef, self.d_flags, self.state,
                          self.flat)
        ev[3].record()

    def unfused_step(self):
        """The same step through the per-call API: zs_reduce_scatter per
        bucket, zs_grad_norm, zs_adam_step per sub-group, then
        zs_all_gather_coalesced per gather bucket into its place in model
        flat space.  Returns the number of kernel launches it made."""
        zs = self.zs
        if not hasattr(self, "_gathers"):
            self._bptrs = [self.bucket_ptrs(b) for b in range(len(self.buf_elems))]
            self._gathers = []
            for g in range(self.info["n_gather_buckets"]):
                gi = zs.zs_gather_bucket_info(self.plan, g)
                ps = [zs.zs_gather_bucket_param(self.plan, g, i) for i in range(gi["n_params"])]
                self._gathers.append((ps, self.flat.data_ptr() + 2 * gi["flat_offset"],
                                      gi["flat_elems"]))
        self.t += 1
        for b, ptrs in enumerate(self._bptrs):
            zs.zs_reduce_scatter(self.plan, b, ptrs, self.gs, self.gP, self.scratch)
        self.norm()
        for sg in range(self.info["n_sub_groups"]):
            zs.zs_adam_step(self.plan, sg, self.hp, self.t, self.d_coef, self.d_flags, self.state)
        launches = len(self._bptrs) + 2 + self.info["n_sub_groups"]
        for ps, base, n in self._gathers:
            zs.zs_all_gather_coalesced(self.plan, ps, self.ps, base, n)
            launches += (len(ps) + 127) // 128
        return launches

    def layer_ranges(self):
        """Runs of consecutive reduce buckets whose gradients one backward
        block produces together: the buckets whose first parameter lies in
        the same decoder layer (the embedding and the output head apart);
        lists without layers take runs of 32 buckets."""
        zs, w = self.zs, self.w
        nb = len(self.buf_elems)
        keys = []
        for b in range(nb):
            first = zs.zs_bucket_entry(self.plan, b, 0)[0]
            name = w.names[first]
            keys.append(name.split(".")[1] if name.startswith("layers.") else
                        name if any(n.startswith("layers.") for n in w.names) else b // 32)
        runs, a = [], 0
        for b in range(1, nb + 1):
            if b == nb or keys[b] != keys[a]:
                runs.append((a, b - a))
                a = b
        return runs

    def unfused_ranges_step(self):
        """unfused_step with the reduce-scatter issued as one
        zs_reduce_scatter_range per run of layer_ranges()."""
        zs = self.zs
        if not hasattr(self, "_runs"):
            self._runs = self.layer_ranges()
            self.unfused_step()          # sets up the gather lists
            self.t -= 1
        self.t += 1
        N = self.N
        for a, n in self._runs:
            zs.zs_reduce_scatter_range(self.plan, a, n, self.ptr_table[a * N:], self.gs, self.gP,
                                       self.scratch)
        self.norm()
        for sg in range(self.info["n_sub_groups"]):
            zs.zs_adam_step(self.plan, sg, self.hp, self.t, self.d_coef, self.d_flags, self.state)
        launches = len(self._runs) + 2 + self.info["n_sub_groups"]
        for ps, base, n in self._gathers:
            zs.zs_all_gather_coalesced(self.plan, ps, self.ps, base, n)
            launches += (len(ps) + 127) // 128
        return launches

    def algorithmic_bytes(self):
        """Bytes the method must move per step (padding excluded):
        reduce-scatter 2N + 2 per element; Adam + cast 28 per element plus
        2 for the gathered write of partitioned elements."""
        psi, N = self.info["psi"], self.N
        part = psi - self.info["persist_elems_logical"]
        rs = (2 * N + 2) * psi
        ag = 28 * psi + 2 * part
        norm = 8 * self.info["n_tiles"] * 2
        return {"reduce_scatter": rs, "norm": norm, "adam_gather": ag}


# ------------------------------------------------------------- clocks -----
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.proc, self.path, self.gpu_id = None, None, gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader", "-lms", "200"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1].split()[0]), float(parts[2].split()[0]), parts))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, p in rows for n, v in zip(names, p[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ----------------------------------------------------------- helpers ------
def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, when
    it was taken on the kernel's device sources (the entry's "sources") as
    they are now (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel)
    if not ent or not ent.get("sources"):
        return None
    try:
        if ent.get("sources_sha256") != sources_digest(ent["sources"]):
            return None
    except OSError:
        return None
    return ent.get("dram_bytes_per_launch")


def sources_digest(files):
    """sha256 over the named files of the package's csrc/, in sorted order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "zero_sharded_optimizer_bucket_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------ CPU baseline ------
# The oracle (oracle/, plain numpy, one process = one core) timed on the
# host.  One step of the path over a sample of the workload: the parameters
# of its first decoder layer (else its first parameters up to a bound).  On
# several cores the sample is cut into one element range per process; each
# process holds the oracle's plan and state of its ranges, so that a step is
#   phase 1: every process reduce-scatters its buckets (oracle.step
#            reduce_scatter) and returns the counts of its reduced values;
#   the parent adds the counts and forms the global norm and clip
#            coefficient (oracle.step sumsq_from_counts, clip_from_sumsq);
#   phase 2: every process runs Adam (oracle.step adam_step) and its gathers
#            (oracle.step gather_model).
# The same oracle functions in the same order as oracle.step.shard_step; the
# norm is global, as the pages require.  Gradients of a process come from a
# Philox pool of its own (synth.philox) that its rank buffers index with
# wrap-around, as the device workload's pool does.
ORACLE_POOL_ELEMS = 1 << 22
_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def oracle_sample(w, target=218_112_000):
    """Indices of the sampled parameters: the parameters of decoder layer 0
    (all parameters when the list has no layers), in order, leaving out any
    larger than `target` elements, until `target` elements are reached.
    The default takes a whole Llama-3-8B layer."""
    cand = [i for i, n in enumerate(w.names) if n.startswith("layers.0.")]
    if not cand:
        cand = list(range(len(w.numel)))
    idx, tot = [], 0
    for i in cand:
        if w.numel[i] <= target:
            idx.append(i)
            tot += w.numel[i]
            if tot >= target:
                break
    return idx


def split_elements(numels, parts):
    """Cut a list of parameter sizes into `parts` consecutive element ranges
    of near-equal size; returns, per part, the sizes of its pieces (a
    parameter cut between two parts becomes one piece in each)."""
    total = sum(numels)
    bounds = [total * (k + 1) // parts for k in range(parts)]
    out, cur, pos, k = [[] for _ in range(parts)], 0, 0, 0
    for n in numels:
        left = n
        while left > 0:
            take = min(left, bounds[k] - pos)
            if take > 0:
                out[k].append(take)
                pos += take
                left -= take
            if pos >= bounds[k] and k < parts - 1:
                k += 1
        if n == 0:
            out[k].append(0)
    return out


def cpu_info():
    """Host CPU: logical cores, the cores this process may run on, model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    try:
        allowed = sorted(os.sched_getaffinity(0))
    except AttributeError:
        allowed = list(range(os.cpu_count() or 1))
    return {"nproc": os.cpu_count(), "allowed": allowed, "cpu_model": model}


def _oracle_part(spec):
    """Plan, state and rank gradient buffers of one process's ranges.
    Weights and gradients are drawn from Philox pools of ORACLE_POOL_ELEMS
    values (the process's own counters) repeated to the length needed: the
    distributions of the workload at a bounded generation cost."""
    import numpy as np

    from oracle import plan as oplan
    from oracle import step as ostep
    from synth import philox
    from synth import workloads as wl
    plan = oplan.build_partition(spec["pieces"], spec["n_ranks"], threshold=spec["threshold"],
                                 reduce_bucket_size=spec["reduce_bucket_size"],
                                 prefetch_bucket_size=spec["prefetch_bucket_size"],
                                 sub_group_size=spec["sub_group_size"], dtype=spec["dtype"],
                                 shard_group_size=spec["group"] or None)
    P = spec["pool_elems"]
    n_w = max(1, min(plan.input_elems, P))
    W = philox.weight_f32(spec["seed"], spec["w_off"] + np.arange(n_w, dtype=np.uint64),
                          spec["weight_sigma"])
    st = ostep.partition(plan, np.resize(W, plan.input_elems))
    need = sum(plan.n_ranks * wl.pool_align(L) for L in plan.bucket_buf_elems)
    largest = wl.pool_align(max(plan.bucket_buf_elems, default=8))
    M = max(8, min(need, max(P, (plan.n_ranks + 1) * largest)))
    idx = spec["g_off"] + np.arange(min(M, P), dtype=np.uint64)
    if spec["dtype"] == "fp16":
        base = philox.grad_fp16(spec["seed"], 0, idx, spec["fp16_log2_scale"])
    else:
        base = philox.grad_bf16(spec["seed"], 0, idx, spec["grad_sigma"], spec["outlier_frac"],
                                spec["outlier_scale"])
    pool = np.resize(base, M)
    offs = wl.pool_offsets(plan.bucket_buf_elems, plan.n_ranks, M) if plan.bucket_buf_elems else []
    bufs = [[pool[o:o + L] for o in offs[b]] for b, L in enumerate(plan.bucket_buf_elems)]
    return plan, st, bufs


def _part_counts(plan, st):
    """Counts of the |x| bit patterns of a process's reduced gradients
    (shard and persistent space; padding is zero and adds nothing)."""
    import numpy as np
    c = np.bincount(st.grad_shards.ravel() & np.uint16(0x7FFF), minlength=1 << 15)
    c += np.bincount(st.persist_grads.ravel() & np.uint16(0x7FFF), minlength=1 << 15)
    return c.astype(np.int64)


def _oracle_worker(conn, spec):
    """One host process of the oracle's parallel step (see above)."""
    if spec.get("cpu") is not None:
        try:
            os.sched_setaffinity(0, {spec["cpu"]})
        except (AttributeError, OSError):
            pass
    from oracle import step as ostep
    plan, st, bufs = _oracle_part(spec)
    conn.send(("ready", plan.psi))
    while True:
        msg = conn.recv()
        if msg[0] == "rs":
            for b in range(len(plan.reduce_buckets)):
                ostep.reduce_scatter(plan, b, bufs[b], st)
            conn.send(("counts", _part_counts(plan, st)))
        elif msg[0] == "adam":
            _, coef, skip, t = msg
            ostep.adam_step(plan, -1, spec["hp"], t, coef, skip, st)
            ostep.gather_model(plan, st.param_shards)
            conn.send(("done", None))
        else:
            conn.send(("bye", None))
            return


def part_specs(w, sample_idx, parts):
    """What each of `parts` processes holds: its element ranges of the
    sampled parameters, the workload's settings, and the counter offsets of
    its weights and gradients."""
    numels = [w.numel[i] for i in sample_idx]
    specs, w_off, g_off = [], 0, 0
    for pieces in split_elements(numels, parts):
        specs.append(dict(pieces=pieces, n_ranks=w.n_ranks, threshold=w.persistence_threshold,
                          reduce_bucket_size=w.reduce_bucket_size,
                          prefetch_bucket_size=w.prefetch_bucket_size,
                          sub_group_size=w.sub_group_size, dtype=w.dtype,
                          group=w.shard_group_size, seed=w.seed, weight_sigma=w.weight_sigma,
                          grad_sigma=w.grad_sigma, outlier_frac=w.outlier_frac,
                          outlier_scale=w.outlier_scale, fp16_log2_scale=w.fp16_log2_scale,
                          hp=w.hparams(), w_off=w_off, g_off=g_off,
                          pool_elems=ORACLE_POOL_ELEMS, cpu=None))
        w_off += sum(pieces)
        g_off += ORACLE_POOL_ELEMS
    return specs


class OracleCluster:
    """The oracle's step on `cpus` host processes (spawned, one pinned to
    each listed core), each over one element range of the sampled
    parameters."""

    def __init__(self, w, sample_idx, cpus):
        import multiprocessing as mp

        self.cpus = list(cpus)
        self.w = w
        specs = part_specs(w, sample_idx, len(self.cpus))
        self.psi = sum(sum(sp["pieces"]) for sp in specs)
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        # one thread per process (the children inherit the environment)
        saved = {v: os.environ.get(v) for v in _THREAD_VARS}
        os.environ.update({v: "1" for v in _THREAD_VARS})
        try:
            for spec, cpu in zip(specs, self.cpus):
                a, b = ctx.Pipe()
                proc = ctx.Process(target=_oracle_worker, args=(b, dict(spec, cpu=cpu)),
                                   daemon=True)
                proc.start()
                self.conns.append(a)
                self.procs.append(proc)
        finally:
            for v, x in saved.items():
                if x is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = x
        for c in self.conns:
            tag, _ = c.recv()
            assert tag == "ready"
        self.t = 0
        self.scale = float(w.loss_scale) if w.dtype == "fp16" else 1.0

    def step(self):
        """One parallel oracle step; returns (norm, coef, skip)."""
        import numpy as np

        from oracle import step as ostep
        self.t += 1
        for c in self.conns:
            c.send(("rs",))
        counts = np.zeros(1 << 15, dtype=np.int64)
        for c in self.conns:
            counts += c.recv()[1]
        norm, coef, skip = ostep.clip_from_sumsq(ostep.sumsq_from_counts(counts, self.w.dtype),
                                                 self.w.max_norm, self.scale)
        for c in self.conns:
            c.send(("adam", coef, skip, self.t))
        for c in self.conns:
            c.recv()
        return norm, coef, skip

    def close(self):
        for c, p in zip(self.conns, self.procs):
            try:
                c.send(("stop",))
                c.recv()
            except (OSError, EOFError):
                pass
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()


def time_oracle(w, sample_idx, cpus, budget_s, min_steps=2, warmup=1):
    """Median seconds per parallel oracle step over at least min_steps
    steps and about budget_s seconds, after `warmup` untimed steps."""
    cl = OracleCluster(w, sample_idx, cpus)
    try:
        for _ in range(warmup):
            cl.step()
        times = []
        t_start = time.perf_counter()
        while len(times) < min_steps or time.perf_counter() - t_start < budget_s:
            t0 = time.perf_counter()
            cl.step()
            times.append(time.perf_counter() - t0)
        return cl.psi, times
    finally:
        cl.close()


def cpu_baseline(w, budget_s=12.0):
    """The oracle on the host: one core on a 1/16 slice of the sample, and
    every core this process may use on the whole sample."""
    info = cpu_info()
    idx = oracle_sample(w)
    cpus = info["allowed"]
    one_idx = idx
    psi_all, t_all = time_oracle(w, idx, cpus, budget_s)
    # one core: the same per-process share of the sample as one of the
    # all-core processes (a process holds psi / len(cpus) elements)
    sub = split_elements([w.numel[i] for i in one_idx], max(len(cpus), 1))[0]
    from synth import workloads as wl
    w1 = wl.Workload(w.name, w.n_ranks, [f"piece{i}" for i in range(len(sub))],
                     [(n,) for n in sub], **{k: getattr(w, k) for k in _WL_FIELDS})
    psi_1, t_1 = time_oracle(w1, list(range(len(sub))), cpus[:1], budget_s)
    per_all, per_1 = statistics.median(t_all), statistics.median(t_1)
    names = [w.names[i] for i in idx]
    what = ("decoder layer 0 (" + ", ".join(n.split(".")[-1] for n in names) + ")"
            if names and names[0].startswith("layers.0.") else f"{len(idx)} parameters")
    return {"value": psi_all / per_all, "unit": UNIT, "cores": len(cpus), "kind": "oracle",
            "sample": f"{what} of {w.name}: {psi_all} elements, N={w.n_ranks}; the whole oracle "
                      f"step (reduce-scatter, global norm, Adam, gathers) on {len(cpus)} "
                      f"processes, one element range each, median of {len(t_all)} steps "
                      f"({per_all:.3f} s)",
            "nproc": info["nproc"], "cpu_model": info["cpu_model"],
            "cores_all": {"value": psi_all / per_all, "cores": len(cpus), "psi": psi_all,
                          "s_per_step": per_all, "steps": len(t_all)},
            "cores_1": {"value": psi_1 / per_1, "cores": 1, "psi": psi_1, "s_per_step": per_1,
                        "steps": len(t_1),
                        "sample": f"the first of the {len(cpus)} element ranges ({psi_1} "
                                  f"elements) on one core"},
            "parallel_efficiency": (psi_all / per_all) / (len(cpus) * psi_1 / per_1)}


_WL_FIELDS = ("persistence_threshold", "reduce_bucket_size", "prefetch_bucket_size",
              "sub_group_size", "grad_sigma", "outlier_frac", "outlier_scale", "weight_sigma",
              "steps", "lr", "beta1", "beta2", "eps", "weight_decay", "adamw", "max_norm", "seed",
              "dtype", "fp16_log2_scale", "loss_scale", "scale_window", "shard_group_size")


# ------------------------------------------------------------- e2e --------
def run_e2e(dw, steps=2, warmup=1, host_pool_bytes=4 << 30, slots=4):
    """Same step through the C ABI with the gradients arriving from pinned
    host memory every step: per bucket one host->device copy of the N rank
    buffers into a ring of device slots (copy stream), zs_reduce_scatter on
    the compute stream as soon as its slot is filled, then zs_grad_norm and
    zs_adam_gather, and the norm and flag word read back to the host."""
    torch, zs = dw.torch, dw.zs
    from synth import workloads as wl
    N, nb = dw.N, len(dw.buf_elems)
    if nb == 0:
        return None
    sizes = [N * wl.pool_align(L) for L in dw.buf_elems]
    total = sum(sizes)
    H = min(total, max(host_pool_bytes // 2, 2 * max(sizes)))
    host = torch.empty(H, dtype=torch.int16, pin_memory=True)
    host.copy_(dw.pool[:min(H, dw.pool.numel())].cpu()) if H <= dw.pool.numel() else host.zero_()
    hoffs = [row[0] for row in wl.pool_offsets(sizes, 1, H)]
    smax = max(sizes)
    ring = torch.empty(slots * smax, dtype=torch.int16, device=dw.dev)
    cs = torch.cuda.Stream(device=dw.dev)
    comp = torch.cuda.current_stream(dw.dev)
    filled = [torch.cuda.Event() for _ in range(slots)]
    free = [torch.cuda.Event() for _ in range(slots)]
    # each step's result (norm bits, skip flags) is read back into its own
    # pinned row; the host does not wait for it inside the step, so the next
    # step's host->device copies overlap this step's update
    out = torch.empty((steps + warmup + 1, 2), dtype=torch.int32, pin_memory=True)
    h2d = sum(2 * N * L for L in dw.buf_elems)
    row = [0]
    used = [False] * slots

    def one_step():
        dw.t += 1
        for b in range(nb):
            s = b % slots
            n = sizes[b]          # the N rank buffers of the bucket, back to back
            if used[s]:           # the slot's last reader (this step or the last) is done
                cs.wait_event(free[s])
            with torch.cuda.stream(cs):
                ring[s * smax:s * smax + n].copy_(host[hoffs[b]:hoffs[b] + n], non_blocking=True)
                filled[s].record(cs)
            comp.wait_event(filled[s])
            base = ring.data_ptr() + 2 * s * smax
            ptrs = [base + 2 * k * wl.pool_align(dw.buf_elems[b]) for k in range(N)]
            zs.zs_reduce_scatter(dw.plan, b, ptrs, dw.gs, dw.gP, dw.scratch)
            free[s].record(comp)
            used[s] = True
        dw.norm()
        zs.zs_adam_gather(dw.plan, dw.hp, dw.t, dw.d_coef, dw.d_flags, dw.state, dw.flat)
        out[row[0], 0:1].copy_(dw.d_norm[0:1].view(torch.int32), non_blocking=True)
        out[row[0], 1:2].copy_(dw.d_flags[0:1], non_blocking=True)
        row[0] += 1

    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize(dw.dev)
    # this machine's own host->device rate (the link is shared with the rest of
    # the machine, so it varies): copies of the ring's size from the pinned
    # buffer, three before and three after the timed steps
    n_link = min(H, ring.numel())

    def link_rates():
        out = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cs)
            with torch.cuda.stream(cs):
                ring[:n_link].copy_(host[:n_link], non_blocking=True)
            b.record(cs)
            torch.cuda.synchronize(dw.dev)
            out.append(2 * n_link / (a.elapsed_time(b) * 1e-3) / 1e9)
        return out

    rates = link_rates()
    torch.cuda.synchronize(dw.dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    torch.cuda.synchronize(dw.dev)       # every step's result is on the host
    dt = (time.perf_counter() - t0) / steps
    flags = [int(out[i, 1]) for i in range(row[0])]
    rates += link_rates()
    link_gbs = max(rates)
    return {"value": dw.info["psi"] / dt, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": 8, "ms_per_step": dt * 1e3, "steps": steps,
            "h2d_gbs_achieved": h2d / dt / 1e9, "h2d_link_gbs_measured": link_gbs,
            "h2d_link_gbs_range": [min(rates), max(rates)],
            "skip_flags": flags,
            "path": "pinned host gradients -> per-bucket H2D ring -> zs_reduce_scatter; "
                    "zs_grad_norm; zs_adam_gather; norm+flags D2H"}


# ----------------------------------------------------------- arms ---------
def run_gpu(args):
    import torch
    rank, world, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    w = load_workload(args.workload)
    dw = DeviceWorkload(w, dev)
    for _ in range(args.warmup):
        dw.step()
    torch.cuda.synchronize(dev)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(_gpu_uuid(torch, dev))
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.25)
    for k in range(K):
        dw.step_timed(evs[k])
    torch.cuda.synchronize(dev)
    barrier(world)
    ck = clocks.stop()
    total_ms = evs[0][0].elapsed_time(evs[-1][3])
    step_ms = max_over_ranks(total_ms / K, world)
    per = {"reduce_scatter": [e[0].elapsed_time(e[1]) for e in evs],
           "norm": [e[1].elapsed_time(e[2]) for e in evs],
           "adam_gather": [e[2].elapsed_time(e[3]) for e in evs]}
    avg = {k: sum(v) / len(v) for k, v in per.items()}
    alg = dw.algorithmic_bytes()
    dom = max(("reduce_scatter", "adam_gather"), key=lambda k: avg[k])
    peak, peak_kind = peaks()
    achieved = alg[dom] / (avg[dom] * 1e-3) / 1e9
    psi = dw.info["psi"]
    value = world * psi / (step_ms * 1e-3)
    step_bytes = alg["reduce_scatter"] + alg["adam_gather"]
    flags = int(dw.d_flags[0].item())
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "storage": f"{w.dtype} gradients and parameters, f32 master / exp_avg / exp_avg_sq",
        "data": "synthetic (Philox4x32-10 gradients and weights; architecture shapes only)",
        "config": {"workload": w.name, "n_ranks": w.n_ranks, "psi": psi, "storage_dtype": w.dtype,
                   "shard_group_size": dw.info["shard_group_size"],
                   "n_params": w.n_params, "reduce_bucket_size": w.reduce_bucket_size,
                   "prefetch_bucket_size": w.prefetch_bucket_size,
                   "param_persistence_threshold": w.persistence_threshold,
                   "max_norm": dw.max_norm,
                   "l2": f"inputs larger than L2: {step_bytes / 1e9:.1f} GB moved per step, "
                         f"gradient pool {2 * dw.pool_elems / 1e9:.1f} GB",
                   "parallelism": "replicas" if world > 1 else "single GPU, N virtual ranks"},
        "hbm_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
        "hbm_frac_of_measured": step_bytes / (step_ms * 1e-3) / 1e9 / peak,
        "hbm_frac_of_nominal_7900": step_bytes / (step_ms * 1e-3) / 1e9 / 7900.0,
        "kernel_ms": avg,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(dom),
                     "algorithmic_bytes_per_launch": alg[dom]},
        "gpu_launches": KERNELS_PER_STEP * K,
        "clocks": ck,
        "skip_flags": flags,
    }
    # A3 on its own: the norm recomputed from the reduced gradients (2 bytes
    # read per element), as zs_grad_norm does without kept partials
    torch.cuda.synchronize(dev)
    n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KN = 5
    n0.record()
    for _ in range(KN):         # zs_grad_norm: no loss-scaler state to disturb
        dw.zs.zs_grad_norm(dw.plan, dw.gs, dw.gP, dw.scratch, True, dw.max_norm, dw.d_norm,
                           dw.d_coef, dw.d_flags)
    n1.record()
    torch.cuda.synchronize(dev)
    nms = n0.elapsed_time(n1) / KN
    res["norm_recompute"] = {"ms": nms, "gbs": 2 * dw.info["psi"] / (nms * 1e-3) / 1e9,
                             "launches": 3, "bytes_per_element": 2}
    # the same step through the per-call API, for comparison (not the value)
    dw.unfused_step()
    torch.cuda.synchronize(dev)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KU = max(2, K // 2)
    u0.record()
    for _ in range(KU):
        n_unfused = dw.unfused_step()
    u1.record()
    torch.cuda.synchronize(dev)
    res["unfused"] = {"ms_per_step": u0.elapsed_time(u1) / KU, "steps": KU,
                      "launches_per_step": n_unfused,
                      "calls": "zs_reduce_scatter per bucket, zs_grad_norm, zs_adam_step per "
                               "sub-group, zs_all_gather_coalesced per gather bucket"}
    dw.unfused_ranges_step()
    torch.cuda.synchronize(dev)
    u0.record()
    for _ in range(KU):
        n_ranged = dw.unfused_ranges_step()
    u1.record()
    torch.cuda.synchronize(dev)
    res["unfused_ranges"] = {"ms_per_step": u0.elapsed_time(u1) / KU, "steps": KU,
                             "launches_per_step": n_ranged, "ranges": len(dw._runs),
                             "calls": "zs_reduce_scatter_range per decoder layer's buckets, "
                                      "then as unfused"}
    res["unfused_bytes_per_elem"] = 2 * dw.N + 36
    # ZeRO-2 residency: no shard buffer, the parameters live in the replica
    st2 = dw.zs.make_state(grad_shards=dw.gs, param_shards=None, master=dw.master, exp_avg=dw.m,
                           exp_avg_sq=dw.v, persist_grads=dw.gP, persist_params=dw.pP,
                           p_master=dw.pm, p_exp_avg=dw.pmm, p_exp_avg_sq=dw.pmv)
    state3, dw.state = dw.state, st2
    dw.step()
    torch.cuda.synchronize(dev)
    u0.record()
    for _ in range(KU):
        dw.step()
    u1.record()
    torch.cuda.synchronize(dev)
    dw.state = state3
    z2 = u0.elapsed_time(u1) / KU
    res["zero2"] = {"ms_per_step": z2, "params_per_s": psi / (z2 * 1e-3),
                    "alg_bytes_per_elem": 2 * dw.N + 30,
                    "note": "same fused step, parameters kept only in the full replica"}
    if not args.no_e2e:
        res["e2e"] = run_e2e(dw, steps=args.e2e_steps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as it stands, on the host cores, same metric and workload:
    each step is the oracle's whole step (oracle.step functions, parallel
    over the host's cores as in cpu_baseline) on a bounded sample of the
    workload (its first decoder layer, else its first parameters)."""
    rank, world, _ = dist_setup()
    if rank != 0:
        return
    w = load_workload(args.workload)
    info = cpu_info()
    cpus = info["allowed"]
    idx = oracle_sample(w, target=args.reference_sample)
    cl = OracleCluster(w, idx, cpus)
    try:
        for _ in range(args.warmup):
            cl.step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            cl.step()
        dt = (time.perf_counter() - t0) / args.steps
    finally:
        cl.close()
    value = cl.psi / dt
    sample = (f"{len(idx)} parameters of {w.name} ({cl.psi} elements, N={w.n_ranks}): whole "
              f"oracle step per timed step on {len(cpus)} host processes, one element range "
              f"each (numpy float32)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": w.name, "n_ranks": w.n_ranks, "psi": w.psi,
                                        "sample_psi": cl.psi},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(cpus), "kind": "oracle",
                         "sample": sample, "nproc": info["nproc"], "cpu_model": info["cpu_model"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def llama_modules(w):
    """Modules of a Llama-shaped parameter list: the embedding, per layer an
    attention module (q, k, v, o, input norm) and an MLP module (gate, up,
    down, post-attention norm), then the final norm with the output head."""
    idx = {n: i for i, n in enumerate(w.names)}
    mods = [[idx["embed_tokens"]]] if "embed_tokens" in idx else []
    layers = sorted({int(n.split(".")[1]) for n in w.names if n.startswith("layers.")})
    for L in layers:
        a = [f"layers.{L}.{x}" for x in ("q_proj", "k_proj", "v_proj", "o_proj", "input_layernorm")]
        b = [f"layers.{L}.{x}" for x in ("gate_proj", "up_proj", "down_proj",
                                          "post_attention_layernorm")]
        mods.append([idx[n] for n in a])
        mods.append([idx[n] for n in b])
    tail = [idx[n] for n in ("norm", "lm_head") if n in idx]
    if tail:
        mods.append(tail)
    return mods


def run_gather_schedule(args):
    """Forward + backward gathers of the workload's modules through the
    gather scheduler, against a stand-in compute of ns_per_elem per element
    of each module: compute alone, gathers alone, both with prefetch, both
    without prefetch (prefetch_bucket_size 0)."""
    import torch

    import zero_sharded_optimizer_bucket_gb300 as zs
    from synth import gpu as sg
    dev = torch.device("cuda", 0)
    w = load_workload(args.workload)
    dw = DeviceWorkload(w, dev, pool_elems=1)
    mods = llama_modules(w)
    order = list(range(len(mods))) + list(reversed(range(len(mods))))
    G = dw.info["shard_group_size"]
    mod_elems = [sum(w.numel[p] for p in m) for m in mods]
    largest = max(sum(G * zs.zs_param_info(dw.plan, p)["partition_size"] for p in set(m))
                  for m in mods)
    base = dict(prefetch_bucket_size=w.prefetch_bucket_size, max_live_parameters=1_000_000_000,
                max_reuse_distance=1_000_000_000)
    arena_elems = base["max_live_parameters"] + 2 * largest
    arena = torch.empty(arena_elems, dtype=torch.int16, device=dev)
    sink = torch.zeros(4, device=dev)
    # optionally a high-priority gather stream (freed SM slots then go to
    # pending gather CTAs first, as collectives' streams are set up)
    gprio = -1 if args.gather_priority == "high" else 0
    comp, gath = torch.cuda.Stream(dev), torch.cuda.Stream(dev, priority=gprio)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.gather_compute == "gemm":
        # stand-in compute: bf16 GEMMs (cuBLAS through torch) of tokens x
        # 4096 by 4096 x 4096, as many per module as its parameters hold
        # 4096^2 blocks: 2 * tokens * numel flops, with the shared memory,
        # registers and tensor cores a real layer takes
        X = torch.randn(args.tokens, 4096, device=dev, dtype=torch.bfloat16)
        Wg = torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16) * 0.01
        Y = torch.empty(args.tokens, 4096, device=dev, dtype=torch.bfloat16)
        reps = [max(1, round(n / 4096 ** 2)) for n in mod_elems]

        def compute(m, count=None):
            with torch.cuda.stream(comp):
                for _ in range(count if count is not None else reps[m]):
                    torch.matmul(X, Wg, out=Y)
        probe_count = 100
        compute(None, 10)
    else:
        # stand-in compute: one warp per SM running a dependent FMA chain
        # takes time without taking the SMs' issue slots or memory bandwidth
        # (as tensor-core compute leaves them); calibrate its ns per step
        blocks, threads = 152, 32
        sg.busy(10000, blocks, sink, comp, threads)
        e0.record(comp)
        sg.busy(200000, blocks, sink, comp, threads)
        e1.record(comp)
        torch.cuda.synchronize(dev)
        ns_per_iter = e0.elapsed_time(e1) * 1e6 / 200000
        iters = [int(args.ns_per_elem * n / ns_per_iter) for n in mod_elems]

        def compute(m, count=None):
            sg.busy(count if count is not None else iters[m], blocks, sink, comp, threads)
        probe_count = 200000
    # concurrency probe: the same compute alone, then beside one large gather
    # on the other stream
    probe_params = [p for p in range(len(w.numel))
                    if not zs.zs_param_info(dw.plan, p)["persistent"]][:8]
    pr_elems = sum(G * zs.zs_param_info(dw.plan, p)["partition_size"] for p in probe_params)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(comp)
    compute(None, probe_count)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    alone = e0.elapsed_time(e1)
    e0.record(comp)
    compute(None, probe_count)
    e1.record(comp)
    e2.record(gath)
    zs.zs_all_gather_coalesced(dw.plan, probe_params, dw.ps, arena, pr_elems, gath)
    e3.record(gath)
    torch.cuda.synchronize(dev)
    probe = {"compute_ms_alone": alone, "compute_ms_beside_gather": e0.elapsed_time(e1),
             "gather_ms_beside_compute": e2.elapsed_time(e3)}

    def run(mode, cfg=None, passes=3, paced=False):
        """paced: the host waits for each module's compute before the next
        fetch (a loop that reads a value back every module), so only
        gathers issued ahead by prefetch can overlap a compute."""
        sched = zs.zs_sched_create(dw.plan, mods, dict(cfg, arena_elems=arena_elems),
                                   arena) if cfg else None
        times = []
        for k in range(passes):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a.record(comp)
            for m in order:
                if sched:
                    zs.zs_sched_fetch(sched, m, dw.ps, comp, gath)
                if mode != "gathers":
                    compute(m)
                if sched:
                    zs.zs_sched_release(sched, m, comp)
                if paced:
                    comp.synchronize()
            if sched:
                zs.zs_sched_end_pass(sched, comp)
            comp.wait_stream(gath)
            b.record(comp)
            torch.cuda.synchronize(dev)
            if k > 0:                   # pass 0 records the trace
                times.append(a.elapsed_time(b))
        st = zs.zs_sched_stats(sched) if sched else None
        return sum(times) / len(times), st

    clocks = ClockSampler(_gpu_uuid(torch, dev))
    clocks.start()
    t_comp, _ = run("compute")
    # gather grid caps: the whole GPU, then one and two CTAs per SM (room
    # left for the compute stream's blocks, as a collective's channels leave)
    by_ctas = {}
    for c in (0, 152, 304):
        cfg = dict(base, gather_ctas=c)
        by_ctas[str(c)] = {"gathers_only_ms": run("gathers", cfg)[0],
                           "prefetch_overlapped_ms": run("both", cfg)[0],
                           "no_prefetch_ms": run("both", dict(cfg, prefetch_bucket_size=0))[0]}
    best = min(by_ctas, key=lambda c: by_ctas[c]["prefetch_overlapped_ms"])
    base = dict(base, gather_ctas=int(best))
    t_gath, st_g = run("gathers", base)
    t_over, st = run("both", base)
    t_serial, _ = run("both", dict(base, prefetch_bucket_size=0))
    t_over2, _ = run("both", base)
    sweep = {}
    for pb in (200_000_000, 1_000_000_000):
        sweep[str(pb)] = run("both", dict(base, prefetch_bucket_size=pb))[0]
    paced = {"compute_only_ms": run("compute", paced=True)[0]}
    for pb in (0, w.prefetch_bucket_size, 200_000_000):
        paced["prefetch_" + str(pb) + "_ms"] = run("both", dict(base, prefetch_bucket_size=pb),
                                                   paced=True)[0]
    ck = clocks.stop()
    gathered = 2 * sum(w.numel[p] for m in mods for p in m if not zs.zs_param_info(dw.plan, p)["persistent"])
    res = {"mode": "gather_schedule", "workload": w.name, "modules": len(mods),
           "passes": "forward + backward, " + str(len(order)) + " fetches",
           "compute": (f"bf16 GEMMs, {args.tokens} tokens x 4096 x 4096, "
                       f"{sum(reps[m] for m in order)} per pass"
                       if args.gather_compute == "gemm"
                       else f"1 warp/SM FMA chain, {args.ns_per_elem} ns per element"),
           "gather_stream_priority": args.gather_priority,
           "compute_tflops": (2.0 * args.tokens * 4096 ** 2 * sum(reps[m] for m in order)
                              / (t_comp * 1e-3) / 1e12 if args.gather_compute == "gemm"
                              else None),
           "compute_only_ms": t_comp, "gathers_only_ms": t_gath, "prefetch_overlapped_ms": t_over,
           "prefetch_overlapped_repeat_ms": t_over2, "no_prefetch_ms": t_serial, "clocks": ck,
           "prefetch_bucket_sweep_ms": sweep, "concurrency_probe": probe,
           "by_gather_ctas": by_ctas, "host_paced": paced,
           "hidden_fraction_of_gather": (t_comp + t_gath - t_over) / t_gath,
           "gathers_only_gbs": 2 * 2 * gathered / (t_gath * 1e-3) / 1e9 if t_gath else None,
           "sched_stats": st, "config": dict(base, arena_elems=arena_elems)}
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="zs", choices=["zs", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of timed oracle steps per CPU-baseline leg")
    ap.add_argument("--reference-sample", type=int, default=50_000_000,
                    help="--impl reference: elements of the sampled parameters (bounded so "
                         "that a warm-up + timed run ends within minutes)")
    ap.add_argument("--gather-schedule", action="store_true",
                    help="measure the forward/backward gather scheduler instead of the step")
    ap.add_argument("--gather-compute", default="busy", choices=["busy", "gemm"],
                    help="gather-schedule mode: the stand-in compute of a module")
    ap.add_argument("--gather-priority", default="normal", choices=["high", "normal"],
                    help="gather-schedule mode: priority of the gather stream")
    ap.add_argument("--tokens", type=int, default=2048,
                    help="gather-schedule mode with --gather-compute gemm: GEMM rows")
    ap.add_argument("--ns-per-elem", type=float, default=0.002,
                    help="stand-in compute per parameter element and pass (gather-schedule "
                         "mode); 0.002 ns is 6 flops x ~570 tokens at 1.7 PFLOP/s")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "zs":
        print("bench.py: at least 3 warm-up steps are required", file=sys.stderr)
        return 2
    if args.impl == "reference":
        run_reference(args)
    elif args.gather_schedule:
        run_gather_schedule(args)
    else:
        run_gpu(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
