"""The multi-process side of bench.py on the CPU: two gloo ranks, as torchrun would start them (one process per
rank, rendezvous on 127.0.0.1). The (sequence, KV head) units are independent, so ranks share no data; the only
cross-rank steps are the barrier around the timed region and the maximum of the ranks' times."""
import math
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from transform_coded_kv_02_b300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own time; the job's time is the slowest rank's
        own = [0.5, 0.75][rank]
        dist.barrier()
        t = bench.max_over_ranks(own, world, "cpu")
        # each rank takes its own layer of the model: same shapes, different data
        w = synth.WORKLOADS["llama_decode_32k"]
        L = synth.make_layer(w, layer=rank, T=32, steps=1)
        fp = torch.tensor([float(np.sum(synth.as_float(L.k)[0, 0, :4, :4]))], dtype=torch.float64)
        fps = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(fps, fp)
        # the reference arm: ranks other than 0 leave at once, without work or output
        ref = bench.run_reference(None, rank, world) if rank != 0 else None
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([t, fps[0].item(), fps[1].item(), L.k.shape[2], 0.0 if ref is None else 1.0]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_layers(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == 0.75                 # both ranks see the slowest rank's time
    assert r0[1] == r1[1] and r0[2] == r1[2]      # the same gathered fingerprints on both ranks
    assert r0[1] != r0[2]                         # rank 0 and rank 1 drew different layers
    assert r0[3] == r1[3] == 32                   # of the same shape
    assert r1[4] == 0.0                           # rank 1 of the reference arm did nothing


def test_job_throughput_counts_every_rank_at_the_slowest_time():
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    # two ranks, 3 GB each, slowest rank 2 s -> 3 GB/s for the job
    assert math.isclose(bench.job_gbs(3e9, 2.0, 2), 3.0)
    assert math.isclose(bench.job_gbs(3e9, 2.0, 1), 1.5)
