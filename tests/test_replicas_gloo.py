"""The multi-replica path of the benchmark on CPU: two gloo ranks (spawned
processes, rendezvous on 127.0.0.1) each report a different step time; the
job time is the slowest rank's and the value counts both ranks' work."""
import json
import os
import socket
import sys
import tempfile

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def max_over_ranks(v):
        t = torch.tensor([v], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    dist.barrier()
    my_ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    tot_ms, value = bench.aggregate_replicas(my_ms, world, 3, 1e9, max_over_ranks)
    with open(f"{out}.{rank}", "w") as f:
        json.dump({"tot_ms": tot_ms, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "r")
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = [json.load(open(f"{out}.{r}")) for r in range(world)]
    for r in res:
        assert r["tot_ms"] == 20.0
        # 2 ranks x 3 steps x 1 GFLOP in 20 ms = 300 GFLOP/s
        assert abs(r["value"] - 300.0) < 1e-9


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    tot, val = bench.aggregate_replicas(4.0, 1, 2, 2e9, None)
    assert tot == 4.0 and abs(val - 1000.0) < 1e-9
