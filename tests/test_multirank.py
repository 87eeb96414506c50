"""The N > 1 path of bench.py on CPU: ranks are independent replicas (each its own batch,
no collective on the data path); only the timing reduction (max step time, summed work)
crosses ranks. Run as two gloo processes."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sec, units = bench.reduce_over_ranks(0.5 + rank, 10.0 * (rank + 1))
    recipe = bench._rank_recipe(2, rank) if rank > 0 else None
    q.put((rank, sec, units, None if recipe is None else int(np.asarray(recipe["past"]).sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, sec, units, _ in res:
        assert sec == 1.5          # max over ranks
        assert units == 30.0       # sum over ranks
    import workloads as w
    assert res[1][3] != int(w.config(2).past_seqlens.sum())  # rank 1 has its own batch


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_over_ranks(0.25, 7.0) == (0.25, 7.0)
