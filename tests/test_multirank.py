"""The N > 1 benchmark path on CPU with gloo (world size 2): each rank gets
its own micro-batches (disjoint seeds, shared weights), the step time is the
maximum over ranks, and the whole-job value counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from bitwise_reproducible_int8_gb300 import inputs
        wl = bench.replica_workload(inputs.WORKLOADS["down_accum"], rank)
        seeds = torch.tensor([wl.x_seed_base + j for j in range(wl.microbatches)])
        gathered = [torch.zeros_like(seeds) for _ in range(world)]
        dist.all_gather(gathered, seeds)
        x0 = inputs.activation(wl, 0, 0, rows=2)            # first rows of this rank's data
        w0 = inputs.weight(wl, 0)[:2]                        # weights are shared
        xs = [torch.zeros(x0.size) for _ in range(world)]
        ws = [torch.zeros(w0.size) for _ in range(world)]
        dist.all_gather(xs, torch.from_numpy(x0.ravel().copy()))
        dist.all_gather(ws, torch.from_numpy(w0.ravel().copy()))
        ms = 100.0 + 50.0 * rank
        ms_max = bench.max_over_ranks(ms, world, "cpu")
        value = bench.whole_job_tokens_per_s(65536, 10, world, ms_max)
        out[rank] = (sorted(int(x) for g in gathered for x in g.tolist()),
                     not torch.equal(xs[0], xs[1]), torch.equal(ws[0], ws[1]), ms_max, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_only():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        seeds, data_differs, weights_same, ms_max, value = res[rank]
        assert seeds == list(range(8))                 # 4 micro-batches each, disjoint
        assert data_differs and weights_same
        assert ms_max == 150.0                         # slowest rank
        assert np.isclose(value, 65536 * 10 * 2 / 0.150)
