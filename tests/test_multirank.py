"""Multi-rank logic on CPU (gloo, world size 2): one cache split across ranks by
contiguous layer ranges.  Each rank draws only its layers, encodes its part
(the oracle stands in for the rank's GPU), and one all-gather of the parts'
u64 payload sizes, scanned exclusively, gives every rank the place of its
part in the single container.  Rank 0 merges the parts with the library's
skv_merge_parts and the result must be the oracle's container of the whole
cache byte for byte.  The bench's own rank helpers (the layer split, the
exclusive scan, the max over ranks) run in the same processes."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


SPECS = {
    "bf16": ("tiny-bf16", dict(L=5)),
    "e4m3": ("qwen3-8b-e4m3", dict(L=3, H=2, T=300, D=64, Tb=128, G=4)),
}


def _worker(rank, world, port, kind, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import oracle as O
    import synth
    import lossless_kv_cache_fixed_gb300 as P
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        name, kw = SPECS[kind]
        spec = synth.WORKLOADS[name].scaled(**kw)
        l0, l1 = bench.layer_range(rank, world, spec.L)
        w = synth.make(spec, layers=(l0, l1))
        kv, mu, sig, cnt = synth.to_numpy(w)
        s = w.spec
        m = O.Model(s.dtype, s.L, s.H, s.T, s.D, s.Tb, s.G, sig, counts=cnt)
        rc, part = O.encode(m, kv, mu)
        assert rc == 0
        nc = m.num_chunks()
        total = int(part[64 + 8 * nc: 64 + 8 * (nc + 1)].view(np.uint64)[0])
        # the one collective of the data path: every rank's payload size
        bases, whole_payload = bench.payload_bases(total, world)
        parts = [None] * world
        dist.all_gather_object(parts, part)     # test plumbing: bring the parts to rank 0
        t = bench.max_over_ranks(1.0 + rank, world)
        res = None
        if rank == 0:
            full = synth.make(spec)
            kvf, muf, sigf, cntf = synth.to_numpy(full)
            mf = O.Model(spec.dtype, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sigf,
                         counts=cntf)
            rc, want = O.encode(mf, kvf, muf)
            assert rc == 0
            params = P.SkvParams(spec.dtype, spec.Tb, spec.G, 0, None, None, None)
            shape = P.SkvShape(spec.L, 2, spec.H, spec.T, spec.D)
            out = np.zeros(want.size, dtype=np.uint8)
            rc, nb = P.skv_merge_parts(params, shape, O.model_hash(mf), parts, out)
            res = (rc, bool(nb == want.size and np.array_equal(out[:nb], want)), want)
        q.put((rank, (l0, l1), bases, whole_payload, total, t, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_two_ranks_one_container(kind):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, kind, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted([q.get(timeout=300) for _ in procs])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rng0, b0, tot0, own0, t0, res), (r1, rng1, b1, tot1, own1, t1, _) = out
    assert rng0[0] == 0 and rng0[1] == rng1[0] and rng1[1] == SPECS[kind][1]["L"]
    assert b0 == b1 == [0, own0] and tot0 == tot1 == own0 + own1
    assert t0 == t1 == 2.0
    rc, equal, want = res
    assert rc == 0 and equal
    # rank 1's part starts where the exclusive scan put it
    nc = int(want[40:48].view(np.uint64)[0])
    offs = want[64: 64 + 8 * (nc + 1)].view(np.uint64)
    first_of_rank1 = nc * (rng1[0] - rng0[0]) // SPECS[kind][1]["L"]
    assert int(offs[first_of_rank1]) == b1[1]


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.layer_range(0, 1, 64) == (0, 64)
    # contiguous, covering, balanced to within one layer
    for world in (2, 3, 8):
        rs = [bench.layer_range(r, world, 64) for r in range(world)]
        assert rs[0][0] == 0 and rs[-1][1] == 64
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
        assert max(b - a for a, b in rs) - min(b - a for a, b in rs) <= 1
    assert bench.payload_bases(7, 1) == ([0], 7)
