"""The bench's multi-process path on CPU: two gloo ranks agree on the slowest rank's time.

The layer is single-GPU; with N > 1 the bench runs N independent replicas and reports the step
time of the slowest one.  This exercises that reduction without a GPU (world_size 2, gloo)."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == 15.0 and out[1] == 15.0


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
