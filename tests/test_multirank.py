"""Multi-rank logic of bench.py on CPU (gloo, world size 2): every rank codes its
own cache (weak scaling, no data-path collective); the step time is the maximum
over ranks and the value sums all ranks' bytes."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, world)
        bench.barrier(world)
        # each rank draws its own cache: the seeds differ, the shapes agree
        import synth
        spec = synth.WORKLOADS["tiny-bf16"].scaled(T=16)
        w = synth.make(spec, seed=bench.rank_seed(rank))
        digest = float(w.kv.view(torch.int16).double().sum().item())
        dig = [0.0] * world
        dist.all_gather_object(dig, digest)
        q.put((rank, t, dig))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_independent_caches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, dig in out:
        assert t == 2.0
        assert dig[0] != dig[1]


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_seed(0) == 0
