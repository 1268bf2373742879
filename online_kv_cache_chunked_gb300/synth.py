"""Seeded synthetic workloads: the inputs both the CUDA path and the oracle consume.

This module holds no arithmetic of the method itself, only input generation.
Keys follow the pages' observations [Chelsea §二 关键观察 / §三 核心观察; CentroidKV
核心组件 观察结果]: key states are highly cosine-similar along the sequence and the
similarity decays monotonically and convexly with distance. An AR(1) process per
(layer, KV head) has E[cos] ~ rho^distance, which has exactly that shape:

    z_0 ~ N(0, I),  z_t = rho z_{t-1} + sqrt(1 - rho^2) eps_t,  k_t = mu_h + z_t,

with rho drawn per head, mu_h a per-head mean offset with N(0, std^2) entries, the
decode keys continuing the same chain, values V ~ N(0, 1), queries q ~ N(0, I) and
degrees N = 1. Layers fold into the batch dimension (one unit per (layer, sequence,
KV head)); statistics (rho, mu) are per (layer, KV head) and shared by the sequences.

Two generators implement the recipe: `make_numpy` (CPU, numpy PCG64, the same bits
on every platform; used for the small cases) and `make_device` (torch on the GPU,
a blocked scan of the recurrence; used for the large cases). Their random streams
differ; parity tests copy the device inputs back to the host for the oracle.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "bf16" | "f32"
    layers: int
    seqs: int
    h_kv: int
    h_q: int
    d: int
    n: tuple              # prefill length per sequence
    rho: tuple            # (lo, hi) of U(lo, hi), or (r, r)
    mu_std: float
    n1: int
    n2: int
    c: int
    R: float
    r_init: float
    dr: float
    r_min: float
    g: int
    steps: int            # decode steps (= Gamma in the budget)
    outlier_frac: float
    seed: int
    forced_round: bool = False  # run one round regardless of the trigger (the tiny case)
    budget_exact: bool = False  # each round merges only the oldest chunks needed to reach B
    # A shard of a larger workload (see shard()): this workload holds layers
    # [layer0, layer0 + layers), sequences [seq0, seq0 + seqs) and KV heads
    # [head0, head0 + h_kv) of one with layers_total x seqs_total x h_kv_total
    # (0 = the same as the shard's own count).
    layer0: int = 0
    seq0: int = 0
    head0: int = 0
    layers_total: int = 0
    seqs_total: int = 0
    h_kv_total: int = 0

    @property
    def global_shape(self):
        """(layers, sequences, KV heads) of the whole workload this one is part of."""
        return (self.layers_total or self.layers, self.seqs_total or self.seqs, self.h_kv_total or self.h_kv)

    @property
    def is_shard(self) -> bool:
        return self.global_shape != (self.layers, self.seqs, self.h_kv)

    @property
    def batch(self) -> int:
        return self.layers * self.seqs

    @property
    def cap(self) -> int:
        # prefill + every decode append, rounded up to a multiple of 64
        return int(math.ceil((max(self.n) + self.steps) / 64.0) * 64)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


def _ragged(seed, count, lo, hi):
    rng = np.random.default_rng(seed + 7)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, count))


WORKLOADS = {
    # fp32 correctness case: 2 KV heads x 1 q head, d=64, s=1024, rho=0.9, one forced round, one decode step
    "tiny_f32": Workload("tiny_f32", "f32", 1, 1, 2, 2, 64, (1024,), (0.9, 0.9), 0.0, 4, 16, 64, 0.2,
                         0.5, 0.0, 0.5, 64, 1, 0.0, 0, forced_round=True),
    # Llama-3.1-8B-shaped layer, 32 q / 8 KV heads, 16K prefill, 1000 decode steps
    "llama_16k": Workload("llama_16k", "bf16", 1, 1, 8, 32, 128, (16384,), (0.8, 0.97), 0.5, 16, 64, 256,
                          0.2, 0.5, 0.0, 0.5, 64, 1000, 0.0, 0),
    # same layer, 32K x batch 4, progressive r_j = max(0.5 - 0.05 j, 0.1), 4% outlier KV heads
    "llama_32k_b4": Workload("llama_32k_b4", "bf16", 1, 4, 8, 32, 128, (32768,) * 4, (0.8, 0.97), 0.5, 16,
                             64, 256, 0.2, 0.5, 0.05, 0.1, 64, 1000, 0.04, 0),
    # 32 independent Llama-3.1-8B-shaped layers, 64K context, batch 1
    "llama_64k_32l": Workload("llama_64k_32l", "bf16", 32, 1, 8, 32, 128, (65536,), (0.8, 0.97), 0.5, 16, 64,
                              256, 0.2, 0.5, 0.0, 0.5, 64, 1000, 0.0, 0),
    # Qwen2-7B-shaped layer, 28 q / 4 KV heads, 16 sequences with lengths U{8192..65536}
    "qwen2_ragged": Workload("qwen2_ragged", "bf16", 1, 16, 4, 28, 128, _ragged(0, 16, 8192, 65536),
                             (0.7, 0.97), 0.0, 16, 64, 256, 0.25, 0.5, 0.0, 0.5, 64, 512, 0.0, 0),
}


def scaled(w: Workload, **kw) -> Workload:
    """A copy with some fields replaced (smaller sizes for quick tests)."""
    return dataclasses.replace(w, **kw)


def head_stats(w: Workload):
    """Per (layer, KV head) rho [layers, h_kv] and mean offset mu [layers, h_kv, d] (float64),
    and the outlier-head mask [h_kv] (uint8), all from the workload seed. A shard gets
    its rows of the whole workload's statistics."""
    Lt, _, Ht = w.global_shape
    rng = np.random.default_rng(w.seed)
    lo, hi = w.rho
    rho = rng.uniform(lo, hi, (Lt, Ht)) if hi > lo else np.full((Lt, Ht), lo)
    mu = rng.normal(0.0, w.mu_std, (Lt, Ht, w.d)) if w.mu_std > 0 else np.zeros((Lt, Ht, w.d))
    mask = np.zeros(Ht, np.uint8)
    if w.outlier_frac > 0:
        k = max(1, int(round(w.outlier_frac * Ht)))
        mask[rng.choice(Ht, size=k, replace=False)] = 1
    ls, hs = slice(w.layer0, w.layer0 + w.layers), slice(w.head0, w.head0 + w.h_kv)
    return rho[ls, hs], mu[ls, hs], mask[hs]


def make_numpy(w: Workload):
    """All inputs on the host (float32 arrays; cast to the cache dtype by the caller).

    Returns dict with K, V: [batch, h_kv, n_max + steps, d] (keys of prefill and decode
    positions), q: [steps, batch, h_q, d], lengths [seqs], rho, mu, head_mask.
    """
    assert not w.is_shard, "make_numpy serves whole workloads; shards use make_device"
    rho, mu, mask = head_stats(w)
    rng = np.random.default_rng(w.seed + 1)
    B, H, d = w.batch, w.h_kv, w.d
    T = max(w.n) + w.steps
    r = np.repeat(rho[:, None, :], w.seqs, axis=1).reshape(B, H)[:, :, None]  # [B, H, 1]
    sig = np.sqrt(1.0 - r * r)
    K = np.empty((B, H, T, d), np.float32)
    z = rng.standard_normal((B, H, d))
    K[:, :, 0] = z
    for t in range(1, T):
        z = r * z + sig * rng.standard_normal((B, H, d))
        K[:, :, t] = z
    K += np.repeat(mu[:, None], w.seqs, axis=1).reshape(B, H, 1, d).astype(np.float32)
    V = rng.standard_normal((B, H, T, d)).astype(np.float32)
    q = rng.standard_normal((w.steps, B, w.h_q, d)).astype(np.float32)
    return dict(K=K, V=V, q=q, lengths=np.array(w.n, np.int64), rho=rho, mu=mu, head_mask=mask)


def _ar1_device(rho_u: torch.Tensor, T: int, d: int, gen: torch.Generator, block: int = 256):
    """AR(1) chains on the device, one per unit: [U, T, d] float32 (blocked linear scan)."""
    U = rho_u.numel()
    nb = (T + block - 1) // block
    dev = rho_u.device
    eps = torch.randn((U, nb * block, d), generator=gen, device=dev, dtype=torch.float32)
    eps[:, 0] = 0.0
    rho = rho_u.view(U, 1, 1).to(torch.float32)
    sig = torch.sqrt(1.0 - rho * rho)
    idx = torch.arange(block, device=dev, dtype=torch.float32)
    expo = (idx.view(-1, 1) - idx.view(1, -1)).clamp(min=0)
    tri = torch.tril(torch.ones(block, block, device=dev))
    Tm = torch.where(tri > 0, rho ** expo.view(1, block, block), torch.zeros((), device=dev)) * tri
    z0 = torch.randn((U, d), generator=gen, device=dev, dtype=torch.float32)
    out = torch.empty((U, nb * block, d), device=dev, dtype=torch.float32)
    powers = rho.view(U, 1, 1) ** (idx + 1).view(1, block, 1)  # rho^(i+1)
    carry = z0 / rho.view(U, 1)  # so that block 0 starts from z0 at t=0
    for k in range(nb):
        e = eps[:, k * block:(k + 1) * block] * sig
        wsum = torch.bmm(Tm, e)
        blk = powers * carry.view(U, 1, d) + wsum
        out[:, k * block:(k + 1) * block] = blk
        carry = blk[:, -1]
    return out[:, :T]


def _group_seed(w: Workload, layer: int, seq: int) -> int:
    """Seed of the inputs of one (layer, sequence) of the whole workload."""
    return (w.seed * 1_000_003 + 7919 * layer + seq + 1) % (2 ** 63)


def make_device(w: Workload, device="cuda"):
    """All inputs generated on the device in the cache dtype.

    Every (layer, sequence) draws its inputs (all KV heads of the whole workload,
    their decode keys and values, its query heads) from a generator seeded by its
    global indices, so a shard of a workload (shard()) gets exactly the inputs
    the whole workload has at its units.

    Returns dict with K, V: [batch, h_kv, cap, d] (prefill rows filled, N=1, len=n per
    sequence), k_dec, v_dec: [steps, batch, h_kv, d], q: [steps, batch, h_q, d],
    lengths [seqs] (host), head_mask (device uint8 [h_kv]).
    """
    _, _, Ht = w.global_shape
    G = w.h_q // w.h_kv
    rho_all, mu_all, mask = _global_rows(w)
    B, H, d, cap = w.batch, w.h_kv, w.d, w.cap
    dt = w.torch_dtype
    K = torch.zeros((B, H, cap, d), dtype=dt, device=device)
    V = torch.zeros((B, H, cap, d), dtype=dt, device=device)
    k_dec = torch.empty((w.steps, B, H, d), dtype=dt, device=device)
    v_dec = torch.empty((w.steps, B, H, d), dtype=dt, device=device)
    q = torch.empty((w.steps, B, w.h_q, d), dtype=dt, device=device)
    lengths = np.array(w.n, np.int64)
    hs = slice(w.head0, w.head0 + H)
    for l in range(w.layers):
        rho_l = torch.from_numpy(rho_all[l]).to(device)                  # [Ht]
        mu_l = torch.from_numpy(mu_all[l]).to(device, torch.float32)     # [Ht, d]
        for sq in range(w.seqs):
            b = l * w.seqs + sq
            gen = torch.Generator(device=device)
            gen.manual_seed(_group_seed(w, w.layer0 + l, w.seq0 + sq))
            n = int(lengths[sq])
            T = n + w.steps  # this sequence's prefill and decode positions
            z = _ar1_device(rho_l, T, d, gen) + mu_l.view(Ht, 1, d)
            v = torch.randn((Ht, T, d), generator=gen, device=device, dtype=torch.float32)
            qg = torch.randn((w.steps, Ht * G, d), generator=gen, device=device, dtype=torch.float32)
            K[b, :, :n] = z[hs, :n].to(dt)
            V[b, :, :n] = v[hs, :n].to(dt)
            k_dec[:, b] = z[hs, n:n + w.steps].transpose(0, 1).to(dt)
            v_dec[:, b] = v[hs, n:n + w.steps].transpose(0, 1).to(dt)
            q[:, b] = qg[:, w.head0 * G:(w.head0 + H) * G].to(dt)
            del z, v, qg
    N = torch.zeros((B, H, cap), dtype=torch.int32, device=device)
    length = torch.zeros((B, H), dtype=torch.int32, device=device)
    for b in range(B):
        n = int(lengths[b % w.seqs])
        N[b, :, :n] = 1
        length[b, :] = n
    return dict(K=K, V=V, N=N, len=length, k_dec=k_dec, v_dec=v_dec, q=q, lengths=lengths,
                head_mask=torch.from_numpy(mask).to(device))


def _global_rows(w: Workload):
    """rho [layers, Ht] and mu [layers, Ht, d] over all KV heads of the whole workload
    for this workload's layers, and this workload's outlier mask [h_kv]."""
    whole_heads = dataclasses.replace(w, head0=0, h_kv=w.global_shape[2], h_q=w.h_q // w.h_kv * w.global_shape[2])
    rho, mu, _ = head_stats(whole_heads)
    _, _, mask = head_stats(w)
    return rho, mu, mask


def shard(w: Workload, rank: int, world: int, mode: str = "weak") -> Workload:
    """Rank `rank`'s part when `world` ranks (one GPU each) run a workload.

    The path has no exchange between (layer, sequence, KV head) units, so ranks
    share nothing. "weak": the whole job is `world` copies of w's shape side by
    side in the sequence dimension (sequences seqs * world), each rank running its
    own seqs sequences with their own inputs -- per-GPU work stays fixed as ranks
    are added. "strong": w's own units are split, by sequences, layers or KV heads
    (the first of these that `world` divides), so the whole job stays fixed.
    """
    if world == 1:
        return w
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world {world}")
    if w.is_shard:
        raise ValueError("already a shard")
    tag = f"{w.name}[{mode} {rank}/{world}]"
    if mode == "weak":
        return dataclasses.replace(w, seq0=rank * w.seqs, seqs_total=world * w.seqs, name=tag)
    if mode != "strong":
        raise ValueError(f"unknown shard mode {mode!r}")
    if w.seqs % world == 0:
        k = w.seqs // world
        return dataclasses.replace(w, seq0=rank * k, seqs=k, seqs_total=w.seqs, n=tuple(w.n[rank * k:(rank + 1) * k]),
                                   name=tag)
    if w.layers % world == 0:
        k = w.layers // world
        return dataclasses.replace(w, layer0=rank * k, layers=k, layers_total=w.layers, name=tag)
    if w.h_kv % world == 0:
        k = w.h_kv // world
        return dataclasses.replace(w, head0=rank * k, h_kv=k, h_q=w.h_q // world, h_kv_total=w.h_kv, name=tag)
    raise ValueError(f"{w.name}: {world} ranks divide neither its sequences, layers nor KV heads")


def shard_axis(w: Workload) -> str:
    """Which dimension a shard cuts ("sequences", "layers", "kv heads" or "none")."""
    L, S, H = w.global_shape
    if S != w.seqs:
        return "sequences"
    if L != w.layers:
        return "layers"
    if H != w.h_kv:
        return "kv heads"
    return "none"


def units(w: Workload):
    """Global (layer, sequence, KV head) of every unit, in the cache's unit order."""
    return [(w.layer0 + b // w.seqs, w.seq0 + b % w.seqs, w.head0 + h) for b in range(w.batch) for h in range(w.h_kv)]


def cache_from_numpy(w: Workload, data, device="cuda"):
    """Device cache tensors from make_numpy's arrays (prefill rows, N=1, len=n)."""
    B, H, d, cap = w.batch, w.h_kv, w.d, w.cap
    dt = w.torch_dtype
    K = torch.zeros((B, H, cap, d), dtype=dt)
    V = torch.zeros((B, H, cap, d), dtype=dt)
    N = torch.zeros((B, H, cap), dtype=torch.int32)
    L = torch.zeros((B, H), dtype=torch.int32)
    k_dec = torch.empty((w.steps, B, H, d), dtype=dt)
    v_dec = torch.empty((w.steps, B, H, d), dtype=dt)
    for b in range(B):
        n = int(w.n[b % w.seqs])
        K[b, :, :n] = torch.from_numpy(data["K"][b, :, :n]).to(dt)
        V[b, :, :n] = torch.from_numpy(data["V"][b, :, :n]).to(dt)
        N[b, :, :n] = 1
        L[b] = n
        k_dec[:, b] = torch.from_numpy(np.moveaxis(data["K"][b, :, n:n + w.steps], 1, 0)).to(dt)
        v_dec[:, b] = torch.from_numpy(np.moveaxis(data["V"][b, :, n:n + w.steps], 1, 0)).to(dt)
    q = torch.from_numpy(data["q"]).to(dt)
    out = dict(K=K, V=V, N=N, len=L, k_dec=k_dec, v_dec=v_dec, q=q, lengths=data["lengths"],
               head_mask=torch.from_numpy(data["head_mask"]))
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in out.items()}
