"""The multi-rank plumbing of bench.py on CPU (gloo, world size 2).

Each GPU runs an independent replica of the workload; the only cross-rank
steps are the timing barrier and the max of the elapsed times, and the CPU
reference arm runs on rank 0 alone.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # the slowest rank's time is the job's time
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    ref = bench.run_reference(bench.parse_args(["--steps", "1", "--warmup", "0", "--cpu-sample-layers", "1",
                                                "--cpu-sample-tokens", "4"]), r, w) if rank == 1 else None
    out[rank] = (t, ref is None)
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_barrier_and_max_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(240)
        assert p.exitcode == 0
    assert out[0][0] == 15.0 and out[1][0] == 15.0
    assert out[1][1] is True          # a non-zero rank does no reference work
