"""Benchmark: CSM compression throughput and degree-aware decode-attention HBM bandwidth.

One step is one pass of the whole hot path over the workload (default: 32
independent Llama-3.1-8B-shaped layers, 8 KV / 32 q heads, d=128, bf16, 64K
prefill, 1000 decode steps):
  restore the prefill cache (device copy from a pristine replica),
  the CSM rounds the trigger fires after prefill,
  1000 x [append the step's k, v; log-N decode attention; triggered CSM rounds].
CSM and attention calls are bracketed by CUDA events on the launching stream.

value         = CSM KV tokens compressed per second of CSM device time (a token is
                one row of one layer's cache of one sequence, all its KV heads);
decode_attn   = algorithmic bytes of the attention calls / their device time;
roofline      = the attention call (the dominant kernel) against measured HBM peak;
e2e           = the same CSM metric through the C ABI from pinned host buffers
                (H2D of the prefill cache, the prefill round, D2H of the compacted
                cache), plus attention decode steps from host buffers;
cpu_baseline  = the fp64 oracle on the host cores on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSM KV tokens compressed/s; log-N decode-attn HBM GB/s (% of peak), 1×GB300"
FALLBACK_HBM_GBS = 6800.0


CSM_KERNELS = {"auto": 0, "simt": 1, "split": 3}
L2_BYTES = 128 << 20  # GB300 L2 is about 129 MB


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def row_bytes(w):
    e = 2 if w.dtype == "bf16" else 4
    return 2 * w.d * e + 4


def csm_call_stats(w, rd, head_mask):
    """Tokens and algorithmic bytes of one CSM call (per the round's sequences). A
    token is one row of one layer's cache (all its KV heads), so a shard that holds
    some of the KV heads counts that fraction of each token."""
    rb = row_bytes(w)
    active_heads = w.h_kv - int(np.asarray(head_mask).sum())
    head_frac = w.h_kv / w.global_shape[2]
    tokens = 0
    nbytes = 0
    for k, s in enumerate(rd.s_before):
        mid = max(0, s - w.n1 - w.n2)
        ch = mid // w.c
        if rd.limits and rd.limits[k] > 0:  # budget-exact round: only the oldest chunks
            ch = min(ch, rd.limits[k])
        tail = s - (w.n1 + ch * w.c) if ch else 0
        tokens += s * w.layers * head_frac
        per_head = ch * w.c * rb + ch * (w.c - rd.m) * rb + 2 * tail * rb
        nbytes += per_head * active_heads * w.layers
    return tokens, nbytes


def attn_bytes(w, lengths_units):
    e = 2 if w.dtype == "bf16" else 4
    return int(lengths_units.sum()) * row_bytes(w) + w.batch * w.h_q * w.d * e * 2


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "online_kv_cache_chunked_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel, key, w):
    """ncu DRAM bytes (per launch or per step) of a kernel, if taken on the current source
    and on this workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    try:
        ok = rec.get("source_sha") == source_sha(rec.get("files", []))
    except OSError:
        ok = False
    ok = ok and rec.get("workload_name") == w.name and not w.budget_exact
    return rec.get(key) if ok else None


class Clocks:
    """Samples nvidia-smi during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples go to a temporary file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"csmkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample(w, units=16, threads=None, decode=False):
    """The fp64 oracle's prefill CSM round on a bounded sample of the workload's units
    (the first 2 layers' 16 KV heads, generated with the same recipe); tokens/s."""
    import oracle
    from online_kv_cache_chunked_gb300 import synth

    layers = max(1, units // w.h_kv)
    ws = synth.scaled(w, layers=layers, seqs=1, n=(w.n[0],), steps=1, name=w.name + "_sample", layer0=0, seq0=0,
                      head0=0, layers_total=0, seqs_total=0, h_kv_total=0)
    data = synth.make_numpy(ws)
    BH = ws.batch * ws.h_kv
    n = ws.n[0]
    cap = ws.cap
    K = np.zeros((BH, cap, ws.d))
    V = np.zeros((BH, cap, ws.d))
    K[:, :n] = data["K"].reshape(BH, -1, ws.d)[:, :n]
    V[:, :n] = data["V"].reshape(BH, -1, ws.d)[:, :n]
    if ws.dtype == "bf16":  # the oracle sees exactly the stored bf16 values
        import torch
        K = torch.from_numpy(K).to(torch.bfloat16).to(torch.float64).numpy()
        V = torch.from_numpy(V).to(torch.bfloat16).to(torch.float64).numpy()
    N = np.ones((BH, cap), np.int32)
    L = np.full(BH, n, np.int32)
    m = oracle.edges_per_chunk(w.r_init, w.c)
    nth = oracle.max_threads() if threads is None else threads
    t0 = time.perf_counter()
    out = oracle.csm_round(K, V, N, L, ws.n1, ws.n2, ws.c, m, nthreads=nth)
    dt = time.perf_counter() - t0
    tokens = n * layers  # tokens per (layer, sequence) cache, all KV heads
    res = dict(value=tokens / dt, unit="tokens/s", cores=nth, seconds=dt,
               sample=f"prefill CSM round (s={n}, c={w.c}, m={m}) of {BH} (layer, KV head) units "
                      f"= {layers} layers x {w.h_kv} heads of the {w.layers}-layer stack, fp64 oracle")
    if decode:
        # one decode step's log-N attention over the compressed sample (the first layer's
        # heads, G query heads each), in the same algorithmic bytes as the GPU metric
        h = w.h_kv
        Kc = out["K"][:h].reshape(1, h, cap, ws.d)
        Vc = out["V"][:h].reshape(1, h, cap, ws.d)
        Nc = out["N"][:h].reshape(1, h, cap)
        Lc = out["len"][:h].reshape(1, h)
        q = np.random.default_rng(0).standard_normal((1, w.h_q, ws.d))
        t0 = time.perf_counter()
        oracle.decode_attn_logn(q, Kc, Vc, Nc, Lc, w.h_q, nthreads=nth)
        da = time.perf_counter() - t0
        nbytes = int(Lc.sum()) * row_bytes(w) + w.h_q * ws.d * (2 if w.dtype == "bf16" else 4) * 2
        res["decode"] = {"value": nbytes / da / 1e9, "unit": "GB/s", "seconds": da,
                         "sample": f"one decode step of log-N attention over {h} compressed KV heads "
                                   f"({int(Lc[0, 0])} tokens each), {w.h_q} query heads, fp64 oracle"}
    return res


def near_tie_check(w, K0, V0, N0, L0, head_mask, p, units=16):
    """The first round's merge decisions on a sample of units against the oracle: the
    GPU compresses a copy of the sample's pristine caches (units are independent, so
    its decisions are the ones the timed run makes), the oracle runs the same round on
    the same stored values, and compare.check_round counts decisions that differ only
    within the 1e-5 near-tie margin (allowed, logged) and any that differ beyond it
    (failures). Part of the CPU-baseline leg: the oracle runs here only."""
    import torch

    import oracle
    from oracle import compare
    from online_kv_cache_chunked_gb300 import binding as B

    rd = p.rounds[0]
    if rd.step != 0:
        return None
    layers = max(1, min(w.layers, units // w.h_kv))  # whole layers of the first sequence's rows
    rows = [l * w.seqs for l in range(layers)]  # batch index of (layer l, sequence 0)
    K, V, N, L = (t[rows].clone() for t in (K0, V0, N0, L0))
    hm = torch.from_numpy(np.asarray(head_mask, np.uint8)).cuda() if int(np.asarray(head_mask).sum()) else None
    cache = B.cache_desc(K)
    m = B.csm_edges_per_chunk(rd.r, w.c)
    maxch = max(1, B.csm_max_chunks(cache, w.n1, w.n2, w.c))
    BHs = K.shape[0] * K.shape[1]
    match = torch.full((BHs, maxch, w.c // 2), -2, dtype=torch.int32, device="cuda")
    ws = B.new_workspace(B.csm_workspace_bytes(cache, w.n1, w.n2, w.c))
    pre_len = L.cpu().numpy().reshape(BHs)
    top = int(pre_len.max())
    preK = K[:, :, :top].cpu().to(torch.float64).numpy().reshape(BHs, top, w.d)
    preV = V[:, :, :top].cpu().to(torch.float64).numpy().reshape(BHs, top, w.d)
    preN = N[:, :, :top].cpu().numpy().reshape(BHs, top)
    B.csm_compress_ex(K, V, N, L, w.n1, w.n2, w.c, rd.r, head_mask=hm, match_out=match, workspace=ws)
    torch.cuda.synchronize()
    gm = match.cpu().numpy()
    skip = np.array([int(np.asarray(head_mask)[u % w.h_kv]) for u in range(BHs)], np.uint8)
    free = oracle.csm_round(preK, preV, preN, pre_len, w.n1, w.n2, w.c, m, skip=skip)
    n_chunks = np.array([0 if skip[u] else oracle.num_chunks(int(pre_len[u]), w.n1, w.n2, w.c) for u in range(BHs)])
    log = []
    dev, fails = compare.check_round(preK, free, gm, n_chunks, m, w.n1, w.c, log=log)
    return {"units": int(BHs), "chunks": int(n_chunks.sum()), "deviating_chunks": int(dev),
            "near_tie_decisions": len(log), "failures": len(fails), "records": log[:8],
            "what": "first round's merge decisions (GPU) on the first sequence's caches of the first "
                    f"{layers} layer(s) against the fp64 oracle on the same values; deviations allowed only "
                    "within a 1e-5 similarity margin"}


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def aggregate(local, world, dist_mod=None):
    """Whole-job numbers: units summed over ranks, times max over ranks."""
    if world == 1:
        return dict(local)
    import torch

    keys_sum = ["tokens", "attn_bytes", "steps_done"]
    keys_max = ["elapsed_s", "csm_s", "attn_s"]
    v_sum = torch.tensor([float(local[k]) for k in keys_sum], dtype=torch.float64)
    v_max = torch.tensor([float(local[k]) for k in keys_max], dtype=torch.float64)
    dm = dist_mod
    if dm is None:
        import torch.distributed as dm
    dev = "cuda" if dm.get_backend() == "nccl" else "cpu"
    v_sum, v_max = v_sum.to(dev), v_max.to(dev)
    dm.all_reduce(v_sum, op=dm.ReduceOp.SUM)
    dm.all_reduce(v_max, op=dm.ReduceOp.MAX)
    out = dict(local)
    out.update({k: float(x) for k, x in zip(keys_sum, v_sum.cpu().tolist())})
    out.update({k: float(x) for k, x in zip(keys_max, v_max.cpu().tolist())})
    return out


def run_reference(args):
    """The oracle as it stands, timed on the host cores (the reference arm)."""
    from online_kv_cache_chunked_gb300 import synth

    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    w = workload_of(args)
    for _ in range(args.warmup):
        oracle_sample(w, units=args.ref_units)
    vals, secs = [], []
    for _ in range(args.steps):
        r = oracle_sample(w, units=args.ref_units)
        vals.append(r["value"])
        secs.append(r["seconds"])
    tokens_per_step = r["value"] * r["seconds"]
    value = tokens_per_step * len(secs) / sum(secs)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * sum(secs) / len(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def workload_of(args):
    from online_kv_cache_chunked_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if getattr(args, "layers", None):  # a smaller or larger stack of the same layer shape
        w = synth.scaled(w, layers=int(args.layers), name=f"{w.name}[{int(args.layers)} layers]")
    return synth.scaled(w, budget_exact=True) if getattr(args, "budget_exact", False) else w


def config_of(w, world=1):
    L, S, H = w.global_shape
    par = "1 GPU"
    if world > 1:
        par = (f"{world} ranks, one GPU each; (layer, sequence, KV head) units sharded by "
               f"{synth_axis(w)} (per rank: {w.layers} layers x {w.seqs} sequences x {w.h_kv} KV heads); "
               "no collective on the data path")
    return {"workload": w.name, "layers": w.layers, "sequences": w.seqs, "kv_heads": w.h_kv, "q_heads": w.h_q,
            "head_dim": w.d, "prefill_tokens": list(w.n) if len(set(w.n)) > 1 else w.n[0],
            "decode_steps": w.steps, "cache_dtype": w.dtype, "n1": w.n1, "n2": w.n2, "c": w.c, "R": w.R,
            "r_init": w.r_init, "delta_r": w.dr, "r_min": w.r_min, "g": w.g, "outlier_frac": w.outlier_frac,
            "budget_exact": w.budget_exact,
            "whole_job": {"layers": L, "sequences": S, "kv_heads": H},
            "parallelism": par,
            "l2": "inputs larger than L2: each decode step reads ~1.1 GB of cache, each prefill round ~13 GB"}


def synth_axis(w):
    from online_kv_cache_chunked_gb300 import synth
    return synth.shard_axis(w)


def run_gpu(args):
    import torch

    from online_kv_cache_chunked_gb300 import _build
    from online_kv_cache_chunked_gb300 import binding as B
    from online_kv_cache_chunked_gb300 import synth
    from online_kv_cache_chunked_gb300.pipeline import Pipeline

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    if not os.path.exists(_build.OUT):
        _build.build()
    B.load()
    # each rank runs its own shard of the job's units (no exchange between ranks)
    w = synth.shard(workload_of(args), rank, world, args.shard)
    stream = torch.cuda.current_stream()
    d = synth.make_device(w)
    K0, V0, N0, L0 = (d[k].clone() for k in ("K", "V", "N", "len"))
    kv = None
    if args.paged:  # the same cache in pages of args.page_rows rows scattered over one pool per array
        from online_kv_cache_chunked_gb300 import paged as PG
        kv = PG.to_paged(d["K"], d["V"], d["N"], args.page_rows, spare_pages=64, seed=w.seed)
        kv0 = tuple(t.clone() for t in (kv.K, kv.V, kv.N))
    p = Pipeline(w, d, stream=None, csm_kernel=CSM_KERNELS[args.csm_kernel], paged=kv)
    head_mask = d["head_mask"].cpu().numpy()
    rounds = p.rounds

    # host mirror of every unit's length at each attention call
    from online_kv_cache_chunked_gb300.pipeline import plan  # noqa: F401
    comp = np.array(w.n, np.int64)
    attn_len = []
    ri = 0
    for step in range(0, w.steps + 1):
        if step > 0:
            comp += 1
            lens = np.zeros((w.batch, w.h_kv), np.int64)
            for b in range(w.batch):
                i = b % w.seqs
                lens[b] = np.where(head_mask.astype(bool), w.n[i] + step, comp[i])
            attn_len.append(lens)
        while ri < len(rounds) and rounds[ri].step == step:
            for i, sa in zip(rounds[ri].seqs, rounds[ri].s_after):
                comp[i] = sa
            ri += 1
    attn_bytes_step = sum(attn_bytes(w, x) for x in attn_len)
    csm_stats = [csm_call_stats(w, rd, head_mask) for rd in rounds]
    csm_tokens_step = sum(t for t, _ in csm_stats)
    csm_bytes_step = sum(b_ for _, b_ in csm_stats)

    # per-call device timing: events recorded by the native loop around every call
    n_pre = sum(1 for rd in rounds if rd.step == 0)
    ev_pre = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_pre)]
    ev_att = [torch.cuda.Event(enable_timing=True) for _ in range(2 * w.steps)]
    ev_csm = [torch.cuda.Event(enable_timing=True) for _ in range(2 * (len(rounds) - n_pre))]
    for e in ev_pre + ev_att + ev_csm:  # torch creates events lazily, on first record
        e.record(stream)
    flush = None
    if args.l2_flush == "on" or (args.l2_flush == "auto" and attn_bytes_step / w.steps < 2 * L2_BYTES):
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    pre_marks = []

    def hook(kind, what, before):
        e = ev_pre[len(pre_marks)]
        e.record(stream)
        pre_marks.append(e)

    def one_step(timed):
        pairs = ((kv.K, kv0[0]), (kv.V, kv0[1]), (kv.N, kv0[2])) if kv is not None else (
            (d["K"], K0), (d["V"], V0), (d["N"], N0))
        for dst, src in pairs + ((d["len"], L0),):
            dst.copy_(src, non_blocking=True)
        pre_marks.clear()
        p.run_native(hook=hook if timed else None, attn_events=ev_att if timed else None,
                     csm_events=ev_csm if timed else None, l2_flush=flush)

    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    csm_ms = attn_ms = 0.0
    attn_calls = 0
    round_ms = [0.0] * len(rounds)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        torch.cuda.synchronize()
        t_start.record(stream)
        for _ in range(args.steps):
            one_step(True)
            torch.cuda.synchronize()
            for k, e in enumerate(ev_pre[0::2] + ev_csm[0::2]):
                e1 = (ev_pre[1::2] + ev_csm[1::2])[k]
                dt = e.elapsed_time(e1)
                round_ms[k] += dt / args.steps
                csm_ms += dt
            for k in range(0, len(ev_att), 2):
                attn_ms += ev_att[k].elapsed_time(ev_att[k + 1])
                attn_calls += 1
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    for ws in (p.ws_csm, p.ws_app, p.ws_att):
        st = B.csmkv_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {st}: {B.status_str(st)}")
    if not np.array_equal(d["len"].cpu().numpy(), attn_len[-1]):
        raise RuntimeError("device lengths disagree with the host schedule")

    local_res = dict(tokens=csm_tokens_step * args.steps, attn_bytes=attn_bytes_step * args.steps,
                     steps_done=args.steps, elapsed_s=elapsed_ms / 1e3, csm_s=csm_ms / 1e3, attn_s=attn_ms / 1e3)
    agg = aggregate(local_res, world)

    # ---- end to end through the C ABI from pinned host buffers
    if rank != 0:
        e2e = None
    elif kv is not None:
        e2e = e2e_measure_paged(w, d, kv, kv0, L0, p, rounds, args)
    else:
        e2e = e2e_measure(w, d, K0, V0, N0, L0, p, rounds, args)
    clocks = clk.summary()
    if rank != 0:
        return 0
    prefill = prefill_measure(w, d, K0, V0, L0, args) if kv is None and not args.no_prefill else None
    hbm, kind = peaks()
    attn_gbs = agg["attn_bytes"] / agg["attn_s"] / 1e9
    per_launch_bytes = attn_bytes_step / w.steps
    avg_launch_s = (attn_ms / 1e3) / max(1, attn_calls)
    csm_gbs = csm_bytes_step * args.steps / (csm_ms / 1e3) / 1e9
    cpu = oracle_sample(w, units=args.cpu_units, decode=True) if not args.no_cpu_baseline else None
    near = near_tie_check(w, K0, V0, N0, L0, head_mask, p) if not args.no_cpu_baseline else None
    line = {
        "metric": METRIC,
        "value": agg["tokens"] / agg["csm_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "strong" if (world > 1 and args.shard == "strong") else "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded AR(1) keys, N(0,1) values, N(0,I) queries; no model weights)",
        "config": dict(config_of(w, world), l2=("a 2xL2 buffer is read before every attention call" if flush is not None
                                          else "every attention call reads more than 2xL2 of cache"),
                       csm_kernel=args.csm_kernel,
                       layout=(f"paged: {args.page_rows}-row pages scattered over a pool (block table per "
                               "(sequence, KV head))" if kv is not None else "dense")),
        "decode_attn": {"value": attn_gbs, "unit": "GB/s", "frac_of_measured_peak": attn_gbs / hbm,
                        "frac_of_nominal_7900": attn_gbs / 7900.0, "calls_timed": attn_calls,
                        "avg_call_us": 1e6 * avg_launch_s},
        "roofline": {"bound": "hbm", "achieved": per_launch_bytes / avg_launch_s / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": per_launch_bytes / avg_launch_s / 1e9 / hbm,
                     "traffic": traffic_record("decode_attn", "bytes_per_launch", w) if kv is None else None, "kernel": "decode_step_logn (append + log-N attention over token splits, then the merge of the splits; one call, two kernels)",
                     "peak_kind": kind, "bytes_per_launch": per_launch_bytes},
        "roofline_csm": {"bound": "hbm", "achieved": csm_gbs, "peak": hbm, "unit": "GB/s", "frac": csm_gbs / hbm,
                         "traffic": traffic_record("csm_compress", "bytes_per_step", w) if kv is None else None, "kernel": "csm_compress",
                         "csm_kernel": args.csm_kernel,
                         "peak_kind": kind, "bytes_per_step": csm_bytes_step},
        "csm": {"tokens_per_step": csm_tokens_step, "head_tokens_per_s": agg["tokens"] * (w.h_kv - int(head_mask.sum())) / agg["csm_s"],
                "ms_per_step": csm_ms / args.steps, "rounds_per_step": len(rounds),
                "rounds": [{"step": rd.step, "m": rd.m, "s_before": int(rd.s_before[0]), "ms": round_ms[k],
                            "gbs": csm_stats[k][1] / (round_ms[k] / 1e3) / 1e9}
                           for k, rd in enumerate(rounds)]},
        "e2e": e2e,
        "prefill": prefill,
        # per decode step: the split kernel and the merge kernel (+ a planning prologue
        # beyond 512 units) and the L2 eviction read when enabled; per round: prologue +
        # main kernel
        "gpu_launches": args.steps * (2 * len(rounds) + ((2 if w.batch * w.h_kv <= 512 else 3)
                                                          + (1 if flush is not None else 0)) * w.steps),
        "clocks": clocks,
    }
    if near is not None:
        line["near_ties"] = near
    if cpu is not None:
        line["cpu_baseline"] = {"value": cpu["value"], "unit": "tokens/s", "cores": cpu["cores"], "kind": "oracle",
                                "sample": cpu["sample"], "seconds": cpu["seconds"], "decode": cpu.get("decode")}
    print(json.dumps(line))
    return 0


def prefill_measure(w, d, K0, V0, L0, args, reps=3):
    """The prompt's attention with the first CSM round fused into it, on one layer of the
    workload (its sequences and all their heads): prefill_attn_csm (attention, and the
    compressed prompt written to a second cache), prefill_attn (attention alone) and the
    standalone round on the same prompt, timed with CUDA events; FLOPs are the causal
    attention's 4 d sum_i (i + 1) per query head."""
    import torch

    from online_kv_cache_chunked_gb300 import binding as B

    if w.dtype != "bf16" or w.d != 128 or w.c != 256:
        return {"unavailable": "the fused prefill kernel covers bf16, head_dim 128, c = 256"}
    rows = slice(0, w.seqs)  # layer 0 of every sequence
    K, V = K0[rows].contiguous(), V0[rows].contiguous()
    lens = L0[rows][:, 0].to(torch.int32).contiguous()
    n = int(lens.max())
    g = torch.Generator(device=K.device).manual_seed(1234)
    q = torch.randn(w.seqs, w.h_q, n, w.d, device=K.device, generator=g).to(torch.bfloat16)
    out = torch.empty_like(q)
    Ko, Vo = torch.empty_like(K), torch.empty_like(V)
    No = torch.empty(K.shape[:3], dtype=torch.int32, device=K.device)
    Lo = torch.empty(K.shape[:2], dtype=torch.int32, device=K.device)
    ws = B.new_workspace(B.prefill_workspace_bytes(), K.device)
    hm = d["head_mask"]
    stream = torch.cuda.current_stream()

    def timed(fn):
        fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        return float(np.median(ts))

    t_fused = timed(lambda: B.prefill_attn_csm(q, K, V, n, out, Ko, Vo, No, Lo, w.n1, w.n2, w.c, w.r_init, ws,
                                               seq_len=lens, head_mask=hm))
    t_attn = timed(lambda: B.prefill_attn(q, K, V, n, out, ws, seq_len=lens))
    st = B.csmkv_device_status(ws)
    # the same round by csm_compress on a copy of the prompt (N = 1, len = s)
    Kc, Vc = K.clone(), V.clone()
    Nc = torch.ones_like(No)
    Lc = lens[:, None].expand(-1, w.h_kv).contiguous()
    wsc = B.new_workspace(B.csm_workspace_bytes(B.cache_desc(Kc), w.n1, w.n2, w.c), K.device)

    def restore():
        Kc.copy_(K)
        Vc.copy_(V)
        Nc.fill_(1)
        Lc.copy_(lens[:, None].expand(-1, w.h_kv))
    t_restore = timed(restore)
    t_round = timed(lambda: (restore(), B.csm_compress(Kc, Vc, Nc, Lc, w.n1, w.n2, w.c, w.r_init, head_mask=hm,
                                                       workspace=wsc))) - t_restore
    same = bool(torch.equal(Lo, Lc))
    if same:
        for u in range(w.seqs):
            for h in range(w.h_kv):
                s_ = int(Lc[u, h])
                same = (same and torch.equal(Ko[u, h, :s_], Kc[u, h, :s_]) and torch.equal(Vo[u, h, :s_], Vc[u, h, :s_])
                        and torch.equal(No[u, h, :s_], Nc[u, h, :s_]))
    flops = 4.0 * w.d * w.h_q * float(sum(int(x) * (int(x) + 1) / 2 for x in lens.tolist()))
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(pk.get("bf16_tflops", 1900.0))
    tf = flops / t_fused / 1e12
    del q, out, Ko, Vo, Kc, Vc
    torch.cuda.empty_cache()
    return {"workload": f"layer 0 of {w.name}: {w.seqs} sequence(s) of up to {n} prompt rows, {w.h_q} query / "
                        f"{w.h_kv} KV heads, first round r = {w.r_init}",
            "value": tf, "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_kind": "measured (cuBLAS bf16 burst)" if pk else "fallback",
                         "kernel": "prefill_attn_csm (tcgen05 QK^T and PV, TMEM accumulators)"},
            "ms_fused": t_fused * 1e3, "ms_attention_only": t_attn * 1e3,
            "attention_only_tflops": flops / t_attn / 1e12,
            "fused_round_extra_ms": (t_fused - t_attn) * 1e3, "standalone_round_ms": t_round * 1e3,
            "second_cache_equals_standalone_round": same, "device_status": st}


def e2e_measure_paged(w, d, kv, kv0, L0, p, rounds, args):
    """The paged layout end to end: H2D of the pools and the lengths from pinned host
    buffers, the prefill round(s) through the paged entry point, D2H of the pools."""
    import torch

    from online_kv_cache_chunked_gb300 import binding as B

    host = [t.cpu().pin_memory() for t in kv0] + [L0.cpu().pin_memory()]
    back = [torch.empty_like(t, device="cpu").pin_memory() for t in (kv.K, kv.V, kv.N)]
    dev = [kv.K, kv.V, kv.N, d["len"]]
    stream = torch.cuda.current_stream()
    pre_k = [k for k, rd in enumerate(rounds) if rd.step == 0]
    tokens = sum(csm_call_stats(w, rounds[k], d["head_mask"].cpu().numpy())[0] for k in pre_k)
    times = []
    for it in range(args.warmup + max(1, args.steps)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for dst, src in zip(dev, host):
            dst.copy_(src, non_blocking=True)
        p.compress_at(0)
        for dst, src in zip(back, (kv.K, kv.V, kv.N)):
            dst.copy_(src, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in back)
    return {"value": tokens / float(np.median(times)), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "what": "paged layout: H2D of the pools, the prefill round(s) "
            "through the paged entry point, D2H of the pools (one stream, not pipelined)"}


def host_link(reps=3, nb=256 << 20):
    """The host link's copy rates in this process (pinned buffers of 256 MB, copy engines):
    upload alone, download alone, and both at once on two streams; GB/s, best of a few."""
    import torch

    dv = torch.empty(nb, dtype=torch.uint8, device="cuda")
    u8 = torch.ones(nb, dtype=torch.uint8).pin_memory()
    d8 = torch.empty(nb, dtype=torch.uint8).pin_memory()
    half = nb // 2
    s_up, s_dn = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, nbytes):
        best = 0.0
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
        return best

    def both():
        cur = torch.cuda.current_stream()
        s_up.wait_stream(cur)
        s_dn.wait_stream(cur)
        with torch.cuda.stream(s_up):
            dv[:half].copy_(u8[:half], non_blocking=True)
        with torch.cuda.stream(s_dn):
            d8[half:2 * half].copy_(dv[half:2 * half], non_blocking=True)
        cur.wait_stream(s_up)
        cur.wait_stream(s_dn)

    return {"h2d_gbs": timed(lambda: dv.copy_(u8, non_blocking=True), nb),
            "d2h_gbs": timed(lambda: d8.copy_(dv, non_blocking=True), nb),
            "both_gbs": timed(both, 2 * half), "bytes": int(nb)}


def e2e_groups(batch, h_kv, fin, want):
    """The end-to-end leg's groups and downloads. A group is a range of cache rows
    with all their KV heads or, with fewer rows than `want` groups, one row's range
    of KV heads: (row0, row1, head0, head1). Each group's download is made of runs
    of consecutive caches of one row with the same final length fin[row, head]:
    (group, first unit, end unit, rows, offset in rows of the host buffers), every
    run in its own contiguous stretch. Returns (groups, runs, total rows)."""
    if batch >= want:
        bounds = [(g * batch // want, (g + 1) * batch // want, 0, h_kv) for g in range(want)]
    else:
        hs = min(h_kv, -(-want // batch))
        bounds = [(b, b + 1, j * h_kv // hs, (j + 1) * h_kv // hs) for b in range(batch) for j in range(hs)]
    runs = []
    off = 0
    for g, (b0, b1, h0, h1) in enumerate(bounds):
        for b in range(b0, b1):
            h = h0
            while h < h1:
                e = h + 1
                while e < h1 and fin[b, e] == fin[b, h]:
                    e += 1
                L = int(fin[b, h])
                runs.append((g, b * h_kv + h, b * h_kv + e, L, off))
                off += (e - h) * L
                h = e
    return bounds, runs, off


def e2e_measure(w, d, K0, V0, N0, L0, p, rounds, args):
    """CSM end to end from pinned host buffers: H2D of the prefill cache, the prefill
    round(s), D2H of the compacted rows (pipelined over groups of layers on separate
    streams); and attention decode steps from host buffers."""
    import torch

    from online_kv_cache_chunked_gb300 import binding as B

    hK = torch.empty_like(K0, device="cpu").pin_memory()
    hV = torch.empty_like(V0, device="cpu").pin_memory()
    hN = torch.empty_like(N0, device="cpu").pin_memory()
    hL = torch.empty_like(L0, device="cpu").pin_memory()
    hK.copy_(K0)
    hV.copy_(V0)
    hN.copy_(N0)
    hL.copy_(L0)
    pre = [rd for rd in rounds if rd.step == 0]
    BH = w.batch * w.h_kv
    # rows every cache holds after the prefill round(s): its sequence's compressed
    # length, or the prompt length for a KV head the mask leaves out
    comp0 = np.array(w.n, np.int64)
    for rd in pre:
        for i, sa in zip(rd.seqs, rd.s_after):
            comp0[i] = sa
    hmask = d["head_mask"].cpu().numpy().astype(bool)
    fin = np.array([np.where(hmask, w.n[b % w.seqs], comp0[b % w.seqs]) for b in range(w.batch)], np.int64)
    stream = torch.cuda.current_stream()
    tokens = sum(csm_call_stats(w, rd, d["head_mask"].cpu().numpy())[0] for rd in pre)
    # Pipelined by groups of caches: group g's upload, its prefill round(s) and its
    # download run on three streams, so one group's transfers overlap another's
    # compression and the two copy directions overlap (a second upload stream was
    # slower: the uploads share the host link). Smaller groups shorten the download
    # of the last group, which nothing overlaps. A group is a range of cache rows
    # (layers x sequences) with all their KV heads or, when there are fewer rows
    # than groups wanted, one row's range of KV heads (every (row, KV head) cache is
    # compressed on its own, and such a slice is contiguous). A group costs a dozen
    # copies and two kernels: groups upload at least 64 MB, but there are at least 8
    # when the iteration runs as a CUDA graph (below) -- the host then no longer
    # issues every call (measured: 32K x 4 best at 8 groups of 70 MB, 0.82 of the
    # link, 0.77 at 32; the 16K layer 0.62 at 8 groups of 9 MB, 0.52 at one).
    h2d_all = sum(t.numel() * t.element_size() for t in (hK, hV, hN, hL))
    want = max(0 if args.e2e_eager else 8, h2d_all // (64 << 20))
    want = max(1, min(args.e2e_groups, want))
    bounds, runs, off = e2e_groups(w.batch, w.h_kv, fin, want)
    G = len(bounds)
    oK = torch.empty((off, w.d), dtype=K0.dtype).pin_memory()
    oV = torch.empty((off, w.d), dtype=V0.dtype).pin_memory()
    oN = torch.empty((off,), dtype=torch.int32).pin_memory()
    dK, dV, dN = d["K"].view(BH, -1, w.d), d["V"].view(BH, -1, w.d), d["N"].view(BH, -1)
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    pre_k = [k for k, rd in enumerate(rounds) if rd.step == 0]

    def issue():
        """One iteration: every group's upload, prefill round(s) and download, forked
        from the current stream onto the three streams and joined back into it."""
        cur = torch.cuda.current_stream()
        ev0 = torch.cuda.Event()
        ev0.record(cur)
        for st_ in (s_in, s_cmp, s_out):
            st_.wait_event(ev0)
        for g, (b0, b1, h0, h1) in enumerate(bounds):
            ev_in, ev_c = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                for key, host in (("K", hK), ("V", hV), ("N", hN), ("len", hL)):
                    d[key][b0:b1, h0:h1].copy_(host[b0:b1, h0:h1], non_blocking=True)
                ev_in.record(s_in)
            s_cmp.wait_event(ev_in)
            for k in pre_k:
                rd = rounds[k]
                mask = p.masks[k]
                lim = p.limits[k]
                B.csm_compress_ex(d["K"][b0:b1, h0:h1], d["V"][b0:b1, h0:h1], d["N"][b0:b1, h0:h1],
                                  d["len"][b0:b1, h0:h1], w.n1, w.n2, w.c, rd.r,
                                  None if p.head_mask is None else p.head_mask[h0:h1],
                                  None if mask is None else mask[b0:b1],
                                  seq_max_chunks=None if lim is None else lim[b0:b1], workspace=p.ws_csm,
                                  stream=s_cmp)
            ev_c.record(s_cmp)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                for _, u0, u1, L, o in (r_ for r_ in runs if r_[0] == g):
                    n_ = (u1 - u0) * L
                    oK[o:o + n_].view(u1 - u0, L, w.d).copy_(dK[u0:u1, :L], non_blocking=True)
                    oV[o:o + n_].view(u1 - u0, L, w.d).copy_(dV[u0:u1, :L], non_blocking=True)
                    oN[o:o + n_].view(u1 - u0, L).copy_(dN[u0:u1, :L], non_blocking=True)
        for st_ in (s_in, s_cmp, s_out):
            cur.wait_stream(st_)

    # The iteration is captured once in a CUDA graph and replayed: every replay
    # still uploads, compresses and downloads every group, without the host's
    # per-call cost (a dozen copy and launch calls per group). Eager issue if the
    # capture fails.
    graph = None
    if not args.e2e_eager:
        try:
            issue()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
                issue()
            torch.cuda.synchronize()
        except RuntimeError as exc:
            print(f"e2e: CUDA graph capture failed ({exc}); issuing eagerly", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
    times = []
    for it in range(args.warmup + max(1, args.steps)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            issue()
        e1.record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            times.append(e0.elapsed_time(e1) / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in (hK, hV, hN, hL))
    d2h = sum(t.numel() * t.element_size() for t in (oK, oV, oN))
    t_e2e = float(np.median(times))
    # untimed: the grouped result equals one call over the whole cache, byte for byte
    for key, src in (("K", K0), ("V", V0), ("N", N0), ("len", L0)):
        d[key].copy_(src)
    for k in pre_k:
        mask, lim = p.masks[k], p.limits[k]
        B.csm_compress_ex(d["K"], d["V"], d["N"], d["len"], w.n1, w.n2, w.c, rounds[k].r, p.head_mask, mask,
                          seq_max_chunks=lim, workspace=p.ws_csm)
    torch.cuda.synchronize()
    if not np.array_equal(d["len"].cpu().numpy(), fin):
        raise RuntimeError("end-to-end leg: lengths after the prefill round disagree with the host schedule")
    def bits(t):
        return t.view(torch.int16 if t.element_size() == 2 else torch.int32)

    for _, u0, u1, L, o in runs:
        n_ = (u1 - u0) * L
        same = (torch.equal(bits(oK[o:o + n_].view(u1 - u0, L, w.d)), bits(dK[u0:u1, :L].cpu()))
                and torch.equal(bits(oV[o:o + n_].view(u1 - u0, L, w.d)), bits(dV[u0:u1, :L].cpu()))
                and torch.equal(oN[o:o + n_].view(u1 - u0, L), dN[u0:u1, :L].cpu()))
        if not same:
            raise RuntimeError(f"end-to-end leg: caches {u0}..{u1 - 1} differ from one call over the whole cache")
    link = host_link()
    # attention decode steps from host buffers: H2D of q, k, v; append; attend; D2H of o
    nsteps = min(50, w.steps)
    hq = d["q"][:nsteps].cpu().pin_memory()
    hk = d["k_dec"][:nsteps].cpu().pin_memory()
    hv = d["v_dec"][:nsteps].cpu().pin_memory()
    ho = torch.empty_like(p.out[:nsteps], device="cpu").pin_memory()
    dq, dk, dv = torch.empty_like(d["q"][:nsteps]), torch.empty_like(d["k_dec"][:nsteps]), torch.empty_like(
        d["v_dec"][:nsteps])
    dout = torch.empty_like(p.out[:nsteps])
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dq.copy_(hq, non_blocking=True)
    dk.copy_(hk, non_blocking=True)
    dv.copy_(hv, non_blocking=True)
    B.csm_decode_run(d["K"], d["V"], d["N"], d["len"], dq, dk, dv, dout, w.n1, w.n2, w.c, rounds=(),
                     head_mask=p.head_mask, ws_csm=p.ws_csm, ws_append=p.ws_app, ws_attn=p.ws_att, steps=nsteps,
                     fused_append=True)
    ho.copy_(dout, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    lens = d["len"].cpu().numpy()
    step_bytes = attn_bytes(w, lens - nsteps // 2)
    att_s = e0.elapsed_time(e1) / 1e3
    # the host link's own rates bound this leg: the upload alone takes h2d / link h2d
    bound = max(h2d / link["h2d_gbs"], (h2d + d2h) / link["both_gbs"]) / 1e9
    return {"value": tokens / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "what": "prefill CSM round from pinned host buffers: H2D cache, "
            f"compress, D2H compacted rows, pipelined over {G} groups of caches"
            + (", one CUDA graph replayed per iteration" if graph is not None else ", issued eagerly"),
            "ms": t_e2e * 1e3, "h2d_gbs": h2d / t_e2e / 1e9, "host_link_gbs": (h2d + d2h) / t_e2e / 1e9,
            "link": link, "link_bound_ms": bound * 1e3, "link_frac": bound / t_e2e,
            "decode_attn_gbs_at_prefill_round_length": step_bytes * nsteps / att_s / 1e9,
            "decode_step_h2d_bytes": int((dq.numel() * dq.element_size() + 2 * dk.numel() * dk.element_size()) // nsteps),
            "decode_step_d2h_bytes": int(ho[0].numel() * ho[0].element_size())}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="llama_64k_32l")
    ap.add_argument("--ref-units", type=int, default=16)
    ap.add_argument("--cpu-units", type=int, default=256,
                    help="(layer, KV head) units in the oracle's timed sample (about 10 s on 16 cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2-flush", default="auto", choices=["auto", "on", "off"],
                    help="zero a 2xL2 buffer before every attention call (auto: when a call reads < 2xL2)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run the workload with this many layers (e.g. a small stack for profiling captures)")
    ap.add_argument("--budget-exact", action="store_true",
                    help="each round merges only the oldest chunks needed to bring s under the budget")
    ap.add_argument("--paged", action="store_true",
                    help="run on a paged (block-table) copy of the cache: pages of --page-rows rows at scattered "
                         "pool pages")
    ap.add_argument("--page-rows", type=int, default=256)
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the fused prefill attention + first round leg")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="issue the end-to-end leg's copies and calls from the host every iteration (no CUDA graph)")
    ap.add_argument("--e2e-groups", type=int, default=32,
                    help="the end-to-end leg pipelines uploads, compression and downloads over this many "
                         "groups of cache rows")
    ap.add_argument("--shard", default="weak", choices=["weak", "strong"],
                    help="with N ranks: weak = N copies of the workload's shape, one per rank (per-GPU work "
                         "fixed); strong = the workload's own units split over the ranks")
    ap.add_argument("--csm-kernel", default="auto", choices=sorted(CSM_KERNELS),
                    help="compression kernel: auto, simt (CUDA cores) or split (tensor cores)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
