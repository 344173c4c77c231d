"""The N > 1 path on CPU: two gloo ranks, each with its own shard of the batch.

The benchmark's multi-GPU mode gives rank r the global batch rows
r*B .. r*B+B-1 (weak scaling) and uses no collective on the data path.  Here
two processes draw their shards with the same generator, run the oracle on
them, and all-gather the results; rank 0 checks that the shards are disjoint,
cover the global batch, and reproduce a single-process run bit for bit.  The
max-over-ranks reduction the benchmark uses for its timing is checked too.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CFG = dict(B=2, H=3, T=40, dk=16, dv=24, dtype="bf16", phi=True, normalize=True, causal=True,
           gamma=("list", [0.9, 0.95, 1.0]), scale_q=0.25, scale_k=0.25, scale_v=1.0, seed=7)


def _rank_main(rank, world, port, out_path):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H = CFG["B"], CFG["H"]
        pairs = workloads.shard_pairs(rank, world, B, H)
        glob = dict(CFG, B=B * world)
        x = workloads.make_inputs(glob, pairs=pairs)
        O, S, z = oracle.recurrent(x["q"][None], x["k"][None], x["v"][None], x["gamma_pairs"],
                                   phi=True, normalize=True)
        mine = torch.from_numpy(np.ascontiguousarray(O[0]))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        idx = torch.tensor(pairs, dtype=torch.int64)
        idxs = [torch.empty_like(idx) for _ in range(world)]
        dist.all_gather(idxs, idx)
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            torch.save({"parts": parts, "idxs": idxs, "max": float(t.item())}, out_path)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_sharding_matches_single_process(tmp_path):
    import oracle
    import workloads
    world = 2
    out = str(tmp_path / "gathered.pt")
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    got = torch.load(out)
    assert got["max"] == float(world)
    B, H = CFG["B"], CFG["H"]
    all_pairs = [tuple(p) for t in got["idxs"] for p in t.tolist()]
    assert len(all_pairs) == len(set(all_pairs)) == B * world * H
    assert set(all_pairs) == {(b, h) for b in range(B * world) for h in range(H)}
    # single process over the whole global batch
    glob = dict(CFG, B=B * world)
    x = workloads.make_inputs(glob)
    O, _, _ = oracle.recurrent(x["q"], x["k"], x["v"], x["gamma"], phi=True, normalize=True)
    k = 0
    for r in range(world):
        for i, (b, h) in enumerate(got["idxs"][r].tolist()):
            assert np.array_equal(got["parts"][r][i].numpy(), O[b, h])
            k += 1
    assert k == B * world * H
