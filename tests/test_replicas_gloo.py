"""The multi-process path of bench.py (independent replicas, one process per
GPU): its barrier and its max over ranks of the step time, run as two gloo
processes on the host (no GPU)."""
import json
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    ms = bench.max_over_ranks(1.5 + 2.0 * r, w)   # rank r timed 1.5 + 2r ms
    with open(os.path.join(outdir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "backend": dist.get_backend(), "max_ms": ms}, f)
    dist.destroy_process_group()


def test_two_replicas_take_the_max_step_time(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r
        assert d["backend"] == "gloo"
        assert d["max_ms"] == 1.5 + 2.0 * (world - 1)   # every rank sees the slowest
