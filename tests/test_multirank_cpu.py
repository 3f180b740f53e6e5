"""The bench's multi-rank host logic on CPU with two gloo ranks (127.0.0.1):
rendezvous from the torchrun environment variables, the barrier, and the
max-over-ranks reduction the timed region uses.  Each rank runs the whole
step on its own GPU (replicas: no collective on the data path); this covers
the process plumbing around them."""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_path: str):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    import torch.distributed as dist
    args = argparse.Namespace(impl="ours", gpus=world)
    w, r, _ = bench.dist_setup(args)
    bench.barrier(w)
    got = bench.reduce_max(10.0 * (r + 1), w)          # rank r times 10 (r + 1) ms
    backend = dist.get_backend()
    bench.barrier(w)
    dist.destroy_process_group()
    with open(f"{out_path}.{r}", "w") as f:
        json.dump({"world": w, "rank": r, "max": got, "backend": backend}, f)


@pytest.mark.timeout(120)
def test_two_gloo_ranks_reduce_the_max_time(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    out = str(tmp_path / "rank")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    for r, d in enumerate(res):
        assert d == {"world": 2, "rank": r, "max": 20.0, "backend": "gloo"}
