"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2):
heads are independent, so ranks run replicas with distinct seeded inputs and
no data-path collective; the only cross-rank step is the max over ranks of
the measured time."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from exact_io_aware_tma_gb300.workloads import make_inputs
    # per-rank replicas: same shape, different seeded inputs
    inp = make_inputs(B=1, H=2, N=64, d=64, mask="causal", seed=bench.rank_seed(3, rank))
    gathered = [torch.zeros_like(inp["q"].float()) for _ in range(world)]
    dist.all_gather(gathered, inp["q"].float())
    # time reduction: max over ranks
    m = bench.max_over_ranks(10.0 + rank)
    out[rank] = (m, bool(torch.equal(gathered[0], gathered[1])), tuple(inp["q"].shape))
    dist.destroy_process_group()


def test_two_rank_replicas_and_time_max():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as man:
        out = man.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 11.0          # max over ranks
    assert res[0][1] is False                       # replicas see different inputs
    assert res[0][2] == res[1][2] == (1, 2, 64, 64)


def test_rank_seed_single_rank_is_identity():
    import bench
    assert bench.rank_seed(3, 0) == 3
    assert len({bench.rank_seed(3, r) for r in range(8)}) == 8
    assert bench.max_over_ranks(2.5) == 2.5
