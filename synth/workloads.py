"""Parameter lists and settings of the synthetic workloads.

The shapes are those of the transformer workloads the ZeRO-3 pages talk
about (a Llama-style decoder layer, Llama-3-8B-shaped layers and model, many
small tensors), as architecture shapes only: no weights, no dataset.  Values
are drawn from `synth.philox`; nothing here computes any part of the
ZeRO-3 step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import philox


@dataclass
class Workload:
    name: str
    n_ranks: int
    names: list
    shapes: list
    persistence_threshold: int = 100_000
    reduce_bucket_size: int = 5_000_000
    prefetch_bucket_size: int = 50_000_000
    sub_group_size: int = 1_000_000_000
    grad_sigma: float = 1e-3
    outlier_frac: float = 0.0
    outlier_scale: float = 100.0
    weight_sigma: float = 0.02
    steps: int = 1
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    adamw: int = 1
    max_norm: float = 1.0
    seed: int = 0x5EED
    ds_id: list = field(default=None)
    dtype: str = "bf16"             # 16-bit storage: "bf16" | "fp16"
    fp16_log2_scale: int = -2       # fp16 gradients: floor(z/512) * 2^e (std ~52 = 1e-3 * 2^16)
    loss_scale: float = 65536.0     # fp16: initial dynamic loss scale
    scale_window: int = 1000
    shard_group_size: int = 0       # HSDP group size G (0: plain ZeRO-3 over all N)

    @property
    def numel(self) -> list:
        return [int(math.prod(s)) for s in self.shapes]

    @property
    def n_params(self) -> int:
        return len(self.shapes)

    @property
    def psi(self) -> int:
        return sum(self.numel)

    def config(self) -> dict:
        return dict(n_ranks=self.n_ranks,
                    param_persistence_threshold=self.persistence_threshold,
                    reduce_bucket_size=self.reduce_bucket_size,
                    prefetch_bucket_size=self.prefetch_bucket_size,
                    sub_group_size=self.sub_group_size)

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay, adamw=self.adamw,
                    bias_correction=1)


def _llama_layer(h: int, ffn: int, kv: int, prefix: str):
    names = [f"{prefix}.q_proj", f"{prefix}.k_proj", f"{prefix}.v_proj", f"{prefix}.o_proj",
             f"{prefix}.gate_proj", f"{prefix}.up_proj", f"{prefix}.down_proj",
             f"{prefix}.input_layernorm", f"{prefix}.post_attention_layernorm"]
    shapes = [(h, h), (kv, h), (kv, h), (h, h), (ffn, h), (ffn, h), (h, ffn), (h,), (h,)]
    return names, shapes


def tiny(threshold: int = 0) -> Workload:
    """Six small tensors, N=4, three AdamW steps (37,248 elements)."""
    shapes = [(64, 64), (64,), (256, 64), (256,), (64, 256), (64,)]
    names = ["fc1.weight", "fc1.bias", "fc2.weight", "fc2.bias", "fc3.weight", "fc3.bias"]
    return Workload("tiny", 4, names, shapes, persistence_threshold=threshold,
                    grad_sigma=1e-3, steps=3, seed=0x5EED0001)


def llama_layer() -> Workload:
    """One Llama-style decoder layer: hidden 4096, 32 heads, ffn 11008, N=8."""
    names, shapes = _llama_layer(4096, 11008, 4096, "layers.0")
    return Workload("llama_layer", 8, names, shapes, grad_sigma=1e-3, steps=1,
                    max_norm=1.0, seed=0x5EED0002)


def _many_small_shapes(n: int, seed: int):
    idx = np.arange(n, dtype=np.uint64)
    u = philox.uniform_u32(seed, philox.STREAM_SHAPE, 0, idx)
    d = philox.uniform_u32(seed, philox.STREAM_SHAPE, 1, idx)
    shapes = []
    for i in range(n):
        x = 2.0 + 4.0 * (int(u[i]) / 4294967296.0)
        numel = int(math.floor(10.0 ** x + 0.5))
        ndim = 1 + int(d[i]) % 3
        shapes.append(_factor(numel, ndim))
    return shapes


def _largest_divisor_at_most(n: int, lim: int) -> int:
    for a in range(max(1, lim), 0, -1):
        if n % a == 0:
            return a
    return 1


def _factor(n: int, ndim: int):
    if ndim == 1:
        return (n,)
    if ndim == 2:
        a = _largest_divisor_at_most(n, math.isqrt(n))
        return (a, n // a)
    a = _largest_divisor_at_most(n, int(round(n ** (1.0 / 3.0))))
    return (a,) + _factor(n // a, 2)


def many_small(n_params: int = 10_000, n_ranks: int = 64) -> Workload:
    """numel log-uniform in [1e2, 1e6], random 1-3D shapes, N=64, 5 steps."""
    seed = 0x5EED0003
    shapes = _many_small_shapes(n_params, seed)
    names = [f"t{i}" for i in range(n_params)]
    return Workload("many_small", n_ranks, names, shapes, grad_sigma=1e-2, steps=5,
                    seed=seed)


def llama3_layers(n_layers: int = 16) -> Workload:
    """16 Llama-3-8B-shaped layers (hidden 4096, 8 KV heads, ffn 14336), N=8,
    grads with 1% outliers x100 so that clipping is exercised."""
    names, shapes = [], []
    for i in range(n_layers):
        n, s = _llama_layer(4096, 14336, 1024, f"layers.{i}")
        names += n
        shapes += s
    return Workload("llama3_16_layers", 8, names, shapes, grad_sigma=1e-3,
                    outlier_frac=0.01, outlier_scale=100.0, steps=1, max_norm=1.0,
                    seed=0x5EED0004)


def llama3_8b() -> Workload:
    """Full Llama-3-8B-shaped parameter list (32 layers, vocab 128256), N=16."""
    names, shapes = ["embed_tokens"], [(128256, 4096)]
    for i in range(32):
        n, s = _llama_layer(4096, 14336, 1024, f"layers.{i}")
        names += n
        shapes += s
    names += ["norm", "lm_head"]
    shapes += [(4096,), (128256, 4096)]
    return Workload("llama3_8b", 16, names, shapes, grad_sigma=1e-3, steps=1,
                    max_norm=1.0, seed=0x5EED0005)


def llama3_attn() -> Workload:
    """One attention block of the Llama-3-8B shapes (q, k, v, o and the input
    norm, 41.9M elements), N=16: the small case for detailed profiles (a
    reduce-scatter launch still reads 1.3 GB, ten times the L2)."""
    n, s = _llama_layer(4096, 14336, 1024, "layers.0")
    keep = [0, 1, 2, 3, 7]
    return Workload("llama3_attn", 16, [n[i] for i in keep], [s[i] for i in keep],
                    grad_sigma=1e-3, steps=1, max_norm=1.0, seed=0x5EED0006)


def llama3_8b_fp16() -> Workload:
    """The Llama-3-8B-shaped list with fp16 gradients and parameters, the
    gradients scaled by a dynamic loss scale starting at 2^16."""
    w = llama3_8b()
    w.name, w.dtype, w.seed = "llama3_8b_fp16", "fp16", 0x5EED0007
    return w


def llama3_8b_hsdp() -> Workload:
    """The Llama-3-8B-shaped list, N=16 ranks as 2 replica groups of 8
    (HSDP: shard within a group, replicate across groups)."""
    w = llama3_8b()
    w.name, w.shard_group_size, w.seed = "llama3_8b_hsdp", 8, 0x5EED0008
    return w


def many_small_prof() -> Workload:
    """200 parameters drawn like many_small (log-uniform sizes, N=64): the
    small case for detailed profiles of that list (2.5 GB of rank gradients
    per step, twenty times the L2)."""
    w = many_small(200)
    w.name, w.steps = "many_small_prof", 1
    return w


def giant_param() -> Workload:
    """One parameter of 2^31 + 5 elements (past any 32-bit element index)
    beside two small ones, N=2: an edge case of the kernels' index
    arithmetic, about 50 GB on the device."""
    shapes = [[2 ** 31 + 5], [4100], [64]]
    names = ["giant", "small", "bias"]
    return Workload("giant_param", 2, names, shapes, grad_sigma=1e-3, steps=1, max_norm=1.0,
                    seed=0x5EED0009)


WORKLOADS = {
    "tiny": tiny,
    "llama_layer": llama_layer,
    "many_small": many_small,
    "llama3_16_layers": llama3_layers,
    "llama3_8b": llama3_8b,
    "llama3_attn": llama3_attn,
    "llama3_8b_fp16": llama3_8b_fp16,
    "llama3_8b_hsdp": llama3_8b_hsdp,
    "giant_param": giant_param,
    "many_small_prof": many_small_prof,
}


POOL_ALIGN = 64      # elements: every buffer starts on a 128-byte boundary


def pool_align(n: int) -> int:
    """n rounded up to the pool's buffer alignment (64 elements, 128 bytes,
    as separately allocated buffers are aligned at least)."""
    return (int(n) + POOL_ALIGN - 1) // POOL_ALIGN * POOL_ALIGN


def pool_offsets(bucket_buf_elems, n_ranks: int, pool_elems: int):
    """Element offsets into a gradient pool for every (bucket, rank) buffer.

    Bucket b of rank k reads `pool[off[b][k] : off[b][k] + bucket_buf_elems[b]]`.
    Buffers are laid one after another, each starting on a 128-byte
    boundary; when the pool is exhausted the layout restarts at 0, so a pool
    smaller than the whole step's gradients is reused with a reuse distance
    of the full pool.
    """
    offs = []
    run = 0
    total = sum(pool_align(L) for L in bucket_buf_elems) * n_ranks
    wraps = total > pool_elems
    for L in bucket_buf_elems:
        L8 = pool_align(L)
        if wraps and L8 * (n_ranks + 1) > pool_elems:
            # (N+1) buffers guarantee that the buffers of one bucket never
            # overlap when the layout wraps around in the middle of a bucket
            raise ValueError("gradient pool smaller than N+1 buffers of one bucket")
        row = []
        for _ in range(n_ranks):
            if run + L8 > pool_elems:
                run = 0
            row.append(run)
            run += L8
        offs.append(row)
    return offs
