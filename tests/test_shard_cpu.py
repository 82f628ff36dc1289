"""Multi-rank split of the (batch, kv-head) groups, checked on CPU with gloo.

Two ranks each run the fp64 oracle on their own groups; the gathered shards
must equal the unsharded result bit for bit (the groups share nothing)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_io_aware_20_gb300.inputs import Workload, make_inputs
from exact_io_aware_20_gb300.shard import shard_views, unit_range


def test_unit_ranges_cover_all_units():
    for B, Hkv, world in ((2, 8, 2), (3, 5, 4), (1, 1, 1), (1, 3, 8)):
        got = [unit_range(B, Hkv, r, world) for r in range(world)]
        assert got[0][0] == 0 and got[-1][1] == B * Hkv
        for (a, b), (c, _) in zip(got, got[1:]):
            assert b == c
        sizes = [b - a for a, b in got]
        assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        unit_range(2, 2, 2, 2)


def test_shard_views_are_the_groups():
    w = Workload("s", 2, 6, 3, 5, 64, "bf16", True, 1)
    q, k, v, do = make_inputs(w)
    lse = torch.randn(2, 6, 5)
    qs, ks, vs, dos, ls = shard_views(q, k, v, 2, 5, do, lse)
    G = 2
    for j, u in enumerate(range(2, 5)):
        b, kh = divmod(u, 3)
        assert torch.equal(ks[0, j], k[b, kh]) and torch.equal(vs[0, j], v[b, kh])
        assert torch.equal(qs[0, j * G:(j + 1) * G], q[b, kh * G:(kh + 1) * G])
        assert torch.equal(dos[0, j * G:(j + 1) * G], do[b, kh * G:(kh + 1) * G])
        assert torch.equal(ls[0, j * G:(j + 1) * G], lse[b, kh * G:(kh + 1) * G])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, w, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    q, k, v, do = make_inputs(w)
    u0, u1 = unit_range(w.B, w.Hkv, rank, world)
    qs, ks, vs, dos = shard_views(q, k, v, u0, u1, do)
    o, lse = oracle.forward(qs, ks, vs, w.causal, w.scale)
    dq, dk, dv = oracle.backward(qs, ks, vs, dos, w.causal, w.scale)
    parts = [torch.from_numpy(x).reshape(-1) for x in (o, lse, dq, dk, dv)]
    flat = torch.cat(parts)
    sizes = torch.tensor([flat.numel()])
    all_sizes = [torch.zeros(1, dtype=torch.long) for _ in range(world)]
    dist.all_gather(all_sizes, sizes)
    maxn = int(max(s.item() for s in all_sizes))
    padded = torch.zeros(maxn, dtype=torch.float64)
    padded[:flat.numel()] = flat
    gathered = [torch.zeros(maxn, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, padded)
    if rank == 0:
        torch.save({"gathered": [g[:int(n.item())] for g, n in zip(gathered, all_sizes)]},
                   os.path.join(out_dir, "gathered.pt"))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("causal", [False, True])
def test_two_rank_split_equals_unsharded(tmp_path, causal):
    w = Workload("shard", 2, 4, 2, 40, 8, "bf16", causal, 31)
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), w, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    import oracle
    q, k, v, do = make_inputs(w)
    o, lse = oracle.forward(q, k, v, w.causal, w.scale)
    dq, dk, dv = oracle.backward(q, k, v, do, w.causal, w.scale)
    got = torch.load(os.path.join(tmp_path, "gathered.pt"))["gathered"]
    G = w.H // w.Hkv
    for rank, flat in enumerate(got):
        u0, u1 = unit_range(w.B, w.Hkv, rank, world)
        qs, ks, vs, dos = shard_views(*(torch.from_numpy(x) for x in (o, dk, dv)),
                                      u0, u1, torch.from_numpy(dq))
        ls = shard_views(torch.from_numpy(o), torch.from_numpy(dk), torch.from_numpy(dv), u0, u1,
                         torch.from_numpy(lse))[3]
        want = torch.cat([t.reshape(-1) for t in (qs, ls, dos, ks, vs)])
        assert torch.equal(flat, want), f"rank {rank} shard differs from the unsharded result"
