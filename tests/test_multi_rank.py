"""The multi-rank path of bench.py on the CPU (gloo, two ranks).

Under torchrun every rank runs its own canvases (replicas, no collective on
the data path); the ranks only agree on the slowest rank's time and report
the whole job's rate from rank 0, and the reference arm runs on rank 0
alone.  These tests run that host logic in two spawned processes.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    import bench
    import dg_synth

    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        # each rank timed its own replica; every rank gets the slowest time
        slowest = bench._reduce_max(1.5 + rank, "cpu")
        value = bench._replica_value(ws, slowest)
        ref_rc = None
        if rank != 0:
            # the reference arm is rank 0's alone: the others return at once
            class A:
                steps, warmup, gpus = 1, 1, world
            ref_rc = bench.run_reference(A, dg_synth.CONFIGS["step_small"])
        tdist.barrier()
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%d %d %d %r %r %r\n" % (ws, r, local, slowest, value, ref_rc))
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    rows = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for r, (ws, rank, local, slowest, value, ref_rc) in enumerate(rows):
        assert (int(ws), int(rank), int(local)) == (world, r, r)
        # the slowest replica (rank 1: 2.5 ms) sets the job time on every rank
        assert float(slowest) == pytest.approx(2.5)
        # two replicas at 2.5 ms each: 800 units/s for the whole job
        assert float(value) == pytest.approx(2 * 1e3 / 2.5)
    assert rows[1][5] == "0"          # rank 1 left the reference arm with status 0


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._reduce_max(3.25, "cpu") == 3.25
    assert bench._replica_value(1, 4.0) == pytest.approx(250.0)
