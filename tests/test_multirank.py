"""The replica (N > 1) logic of bench.py on CPU with two gloo ranks.

Tokens are independent, so N GPUs run N replicas with no collective on the
data path: each rank draws its own batch with shared weights, the job time is
the slowest rank's, and the job throughput counts every rank's tokens.
"""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from token_routing_expert_gb300.workloads import WORKLOADS

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = WORKLOADS["tiny"]
    inp = bench.rank_inputs(spec, rank)
    digest = torch.tensor([float(inp["x"].float().sum()), float(inp["w_up_gate"].float().sum())], dtype=torch.float64)
    gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, digest)
    slowest = bench.max_over_ranks(1.0 + rank, dist, "cpu")   # rank r "took" 1 + r ms
    out[rank] = (gathered[0][0] != gathered[1][0]).item(), (gathered[0][1] == gathered[1][1]).item(), slowest, \
        bench.job_tokens_per_s(world, spec.T, slowest), bench.bench_config(spec, world)["global_tokens"]
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        x_differs, weights_equal, slowest, tps, global_tokens = res[rank]
        assert x_differs and weights_equal          # own batch, shared weights
        assert slowest == 2.0                       # the max over ranks
        assert tps == 2 * 256 / 2e-3                 # every rank's tokens over the slowest time
        assert global_tokens == 512
