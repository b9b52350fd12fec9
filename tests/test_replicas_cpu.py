"""The bench's multi-process path on the CPU: two ranks over gloo
(rendezvous on 127.0.0.1). Each rank runs an independent replica; the only
collectives are the timing barrier and the maximum over ranks of the step
time, from which the whole-job value is world x B x K / max time (weak
scaling). The reference arm runs on rank 0 alone."""
import argparse
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r = bench.dist_setup()
    bench.barrier(w)
    step_s = 0.010 + 0.001 * r  # this rank's time for K steps
    worst = bench.max_over_ranks(step_s, w)
    B, K = 32, 5
    q.put((r, w, worst, w * B * K / worst))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_replicas_share_only_the_barrier_and_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for r, w, worst, value in got:
        assert w == 2
        assert abs(worst - 0.011) < 1e-12                      # the slower rank's time on both ranks
        assert abs(value - 2 * 32 * 5 / 0.011) < 1e-6          # units of both ranks / the max time


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(workload="qwen", splits=None, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, 2, 1) is None                  # rank 1: no work, no line
    assert capsys.readouterr().out == ""
