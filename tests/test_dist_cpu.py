"""The multi-rank path of bench.py (one independent replica per GPU, launched by
torchrun; no collective on the data path) on CPU with the gloo backend at
world size 2: the step time is the slowest rank's (max-reduction), the value
is the whole job's (world x per-rank FLOPs over that time), every rank draws
its own inputs, and the reference arm does its work on rank 0 only."""
import argparse
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out) -> None:
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.allreduce_max(ms, torch.device("cpu"), world)
        value = bench.job_tflops(1e12, slowest, world)
        ref = None
        if rank != 0:  # rank 0 would run the oracle; the others must return at once
            args = argparse.Namespace(config="C1", seed=0, warmup=3, steps=1)
            ref = bench.run_reference(args, rank, world)
        torch.distributed.barrier()
        out.put((rank, slowest, value, bench.rank_seed(7, rank), ref))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_on_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for _, slowest, value, _, _ in results:
        assert slowest == 15.0
        assert abs(value - 2 * 1e12 / 15e-3 / 1e12) < 1e-9
    assert [r[3] for r in results] == [7, 8]  # independent inputs per rank
    assert results[1][4] is None
