"""Sharding a workload over ranks (one GPU each), on the CPU.

The path has no exchange between (layer, sequence, KV head) units [Chelsea §三
算法流程: per layer and head the cache state, its compression schedule and its
attention are independent], so N ranks run disjoint sets of units and need no
collective. Checked here:
* world size 2 over gloo: the ranks' unit sets are disjoint and together cover
  the whole workload exactly once; every rank's host plan (rounds, lengths) and
  final lengths equal the single-rank plan's entries for its units;
* a shard's inputs are exactly the whole workload's inputs at its units;
* the weak mode's whole job is world copies of the per-rank shape.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from online_kv_cache_chunked_gb300 import synth
from online_kv_cache_chunked_gb300.pipeline import final_lengths, plan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [("llama_64k_32l", "strong"), ("llama_32k_b4", "strong"), ("qwen2_ragged", "strong"),
         ("llama_16k", "strong"), ("llama_32k_b4", "weak"), ("llama_64k_32l", "weak")]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_view(name, mode, rank, world):
    """What a rank knows about its shard: global unit ids, and per global sequence its
    rounds (step, r, s_before, s_after) and per unit its final length."""
    w = synth.shard(synth.WORKLOADS[name], rank, world, mode)
    rounds = {}
    for rd in plan(w):
        for i, sb, sa in zip(rd.seqs, rd.s_before, rd.s_after):
            rounds.setdefault(w.seq0 + i, []).append((rd.step, rd.r, sb, sa))
    fl = final_lengths(w).reshape(-1)
    u = synth.units(w)
    return dict(units=u, rounds=rounds, final={k: int(x) for k, x in zip(u, fl)}, axis=synth.shard_axis(w))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    views = {f"{n}/{m}": _rank_view(n, m, rank, world) for n, m in CASES}
    got = [None] * world
    dist.all_gather_object(got, views)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_two_ranks_cover_every_unit_once_with_the_single_rank_plan():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get() for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res[0] == res[1]  # every rank gathered the same views
    views = res[0]
    for name, mode in CASES:
        w = synth.WORKLOADS[name]
        key = f"{name}/{mode}"
        r0, r1 = views[0][key], views[1][key]
        u0, u1 = set(r0["units"]), set(r1["units"])
        assert not (u0 & u1)
        whole = w if mode == "strong" else synth.scaled(w, seqs=2 * w.seqs, n=tuple(w.n) * 2)
        assert u0 | u1 == set(synth.units(whole)) and len(u0) + len(u1) == whole.batch * whole.h_kv
        ref = _rank_view(whole.name, "strong", 0, 1) if mode == "strong" else None
        if ref is None:  # the weak job is two copies: sequence i + seqs follows sequence i's plan
            base = _rank_view(name, "strong", 0, 1)
            ref = dict(rounds={**base["rounds"], **{i + w.seqs: v for i, v in base["rounds"].items()}},
                       final={**base["final"], **{(l, s + w.seqs, h): v for (l, s, h), v in base["final"].items()}})
        for rv in (r0, r1):
            for sq, rds in rv["rounds"].items():
                assert rds == ref["rounds"][sq], (key, sq)
            for unit, length in rv["final"].items():
                assert length == ref["final"][unit], (key, unit)
        if mode == "strong":
            assert r0["axis"] == {"llama_64k_32l": "layers", "llama_16k": "kv heads"}.get(name, "sequences")
        else:
            assert r0["axis"] == "sequences"


@pytest.mark.parametrize("mode,world", [("strong", 2), ("strong", 4), ("weak", 2)])
def test_shard_inputs_are_the_whole_workloads_inputs(mode, world):
    w = synth.scaled(synth.WORKLOADS["llama_32k_b4"], n=(700, 650, 700, 333), steps=3, layers=2)
    whole = w if mode == "strong" else synth.scaled(w, seqs=world * w.seqs, n=tuple(w.n) * world)
    d = synth.make_device(whole, "cpu")
    for rank in range(world):
        ws = synth.shard(w, rank, world, mode)
        ds = synth.make_device(ws, "cpu")
        idx = [whole.seqs * l + s for (l, s, h) in synth.units(ws)[::ws.h_kv]]
        heads = slice(ws.head0, ws.head0 + ws.h_kv)
        G = w.h_q // w.h_kv
        for k in ("K", "V", "N"):  # rows past the shard's capacity are empty in the whole too
            assert torch.equal(ds[k], d[k][idx][:, heads][:, :, :ws.cap]), (rank, k)
            assert not d[k][idx][:, heads][:, :, ws.cap:].any()
        assert torch.equal(ds["len"], d["len"][idx][:, heads])
        for k in ("k_dec", "v_dec"):
            assert torch.equal(ds[k], d[k][:, idx][:, :, heads]), (rank, k)
        assert torch.equal(ds["q"], d["q"][:, idx][:, :, ws.head0 * G:(ws.head0 + ws.h_kv) * G])
        assert np.array_equal(ds["head_mask"].numpy(), d["head_mask"].numpy()[heads])


def test_head_shards_split_the_query_heads_with_their_kv_heads():
    w = synth.scaled(synth.WORKLOADS["llama_16k"], n=(400,), steps=2)
    d = synth.make_device(w, "cpu")
    for rank in range(4):
        ws = synth.shard(w, rank, 4, "strong")
        assert (ws.h_kv, ws.h_q, ws.head0) == (2, 8, 2 * rank)
        ds = synth.make_device(ws, "cpu")
        assert torch.equal(ds["K"], d["K"][:, 2 * rank:2 * rank + 2])
        assert torch.equal(ds["q"], d["q"][:, :, 8 * rank:8 * rank + 8])


def test_shards_that_do_not_divide_are_refused():
    with pytest.raises(ValueError):
        synth.shard(synth.WORKLOADS["tiny_f32"], 0, 3, "strong")
    with pytest.raises(ValueError):
        synth.shard(synth.shard(synth.WORKLOADS["llama_32k_b4"], 0, 2), 0, 2)
