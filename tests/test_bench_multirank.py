"""The benchmark's multi-rank host logic on CPU with the gloo backend, world size 2:
each rank gets its own batch seed and the reported time is the slowest rank's."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from latent_moe_layer_rmsnorm_gb300 import synth
    t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    seed = bench.rank_seed(0, rank)
    shape = synth.TINY_F32.replace(T=4)
    x = synth.make_dense(shape, seed=seed)["x"]
    q.put((rank, t, seed, x.sum().item()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]          # max over ranks
    assert res[0][2] != res[1][2]                        # distinct batch seeds
    assert res[0][3] != res[1][3]                        # so distinct batches
    assert bench_single_rank() == 7.0


def bench_single_rank():
    import bench
    return bench.max_over_ranks(7.0, "cpu")
