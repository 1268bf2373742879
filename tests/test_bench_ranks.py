"""The multi-process side of bench.py on CPU: world size 2 over gloo.

The path shards by (layer, sequence, KV head) with no data-path exchange, so a
run on N GPUs is N independent replicas; the only collective is the final
aggregation (units summed over ranks, times maxed). Here two gloo ranks check
that aggregation and that the reference arm runs on rank 0 alone."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = dict(tokens=100.0 * (rank + 1), attn_bytes=1e9 * (rank + 1), steps_done=3, elapsed_s=1.0 + rank,
                 csm_s=0.25 * (rank + 1), attn_s=0.5 + 0.125 * rank)
    agg = bench.aggregate(local, world)

    class A:
        gpus, steps, warmup, workload, ref_units = world, 1, 0, "tiny_f32", 2

    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(A)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, agg, rc, buf.getvalue()))


def test_two_rank_aggregation_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(2):
        rank, agg, rc, text = q.get()
        out[rank] = (agg, rc, text)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank in (0, 1):
        agg, rc, _ = out[rank]
        assert rc == 0
        assert agg["tokens"] == 300.0 and agg["attn_bytes"] == 3e9 and agg["steps_done"] == 6
        assert agg["elapsed_s"] == 2.0 and agg["csm_s"] == 0.5 and agg["attn_s"] == 0.625
    line = json.loads(out[0][2].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert out[1][2].strip() == ""  # rank 1 prints nothing and does no work
