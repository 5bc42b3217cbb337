"""The N > 1 path of bench.py on CPU: world-size-2 gloo process groups stand
in for the NCCL ranks.  The layer runs as independent replicas (no data-path
collective); what the ranks share is the barrier around the timed region and
the max over ranks of the step time, and only rank 0 reports."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = synth.CONFIGS["tiny"]
    rcfg = bench.replica_config(cfg, rank)
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist)  # rank 1 is the slower one
    dist.barrier()

    class Args:
        steps, warmup, ref_budget_s = 1, 0, 2.0
    line = bench.run_reference(Args, cfg, rank, world)
    out.put((rank, rcfg.seed, ms, None if line is None else line["n_gpus"]))
    dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_time_and_only_rank0_reports():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, ms0, n0), (r1, seed1, ms1, n1) = res
    assert (r0, r1) == (0, 1)
    assert ms0 == ms1 == 15.0               # both ranks see the slowest rank's time
    assert seed0 != seed1                   # each replica routes its own tokens
    assert n0 == world and n1 is None       # rank 0 alone runs the reference arm and reports
