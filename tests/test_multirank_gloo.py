"""The multi-process harness of bench.py on CPU with gloo (world size 2):
max-over-ranks timing, independent replicas per rank, whole-job throughput.
(The data path has no collective: each rank runs its own layer.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from synth import WORKLOADS, make_logit_offset
        # each rank's "step time": rank 1 is the slow one
        t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        wl = bench.replica_workload(WORKLOADS["small"].with_(T=64), rank)
        logits = make_logit_offset(wl)
        gathered = [torch.zeros(64, 16) for _ in range(world)]
        dist.all_gather(gathered, torch.from_numpy(logits))
        same_seed = bool(torch.equal(gathered[0], gathered[1]))
        out[rank] = (t, wl.seed, same_seed,
                     bench.whole_job_tokens_per_s(world, wl.T, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_harness():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0          # the max over ranks
    assert out[0][1] != out[1][1]                  # own seed per replica
    assert out[0][2] is False                      # so their inputs differ
    # whole-job throughput counts every rank's tokens over the max time
    assert out[0][3] == pytest.approx(2 * 64 / 0.015)


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
