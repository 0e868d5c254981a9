"""The N > 1 bench plumbing on CPU: world-size-2 gloo ranks (no GPU).

Each rank of a multi-GPU run processes its own replica of the workload (independent problems,
no data-path collective); the only cross-rank steps are the barrier and the max-reduction of
the step time, and the reference arm runs on rank 0 alone.
"""
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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank             # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        dist.barrier()
        value = bench.aggregate_value(1e12, world, ms)
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), rank, world)
        q.put((rank, ms, value, buf.getvalue()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(600)
def test_two_rank_gloo_time_reduction_and_rank0_reference():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        r, ms, value, out = q.get(timeout=540)
        res[r] = (ms, value, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank reports the slowest rank's time and the whole-job aggregate
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(1e12 * 2 / 15e-3 / 1e12)
    # the reference (oracle) arm prints one JSON line on rank 0 only
    assert res[1][2] == ""
    line = json.loads(res[0][2])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
