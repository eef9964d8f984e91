"""Two ranks (gloo, CPU) each update their contiguous shard of a flattened
parameter set with the oracle; the gathered result is bitwise the whole
update.  Covers the shard planning used for multi-rank runs."""
import os
import socket

import numpy as np
import pytest

from stochastic_rounding_gb300 import sharding

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
SIZES = [4096, 1, 7, 10007, 3, 2048, 4097, 513]


def _data(seed=0):
    from stochastic_rounding_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    total = sum(SIZES)
    p = W.to_bf16_bits(W.normal_f32(rng, total, 0.02))
    g = W.to_bf16_bits(W.normal_f32(rng, total, 1e-3))
    m = W.normal_f32(rng, total, 1e-4)
    v = np.abs(W.normal_f32(rng, total, 1e-6))
    return p, g, m, v


def _rank_main(rank, world, port, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    o = oracle.get()
    p, g, m, v = _data()
    start, end = sharding.shard_bounds(len(p), world, rank)
    pieces = sharding.shard_pieces(SIZES, start, end)
    # the rank's buffers are its range only; each piece carries its base index
    P, G, M, V = (a[start:end].copy() for a in (p, g, m, v))
    for t, off, n, base in pieces:
        a = base - start
        sl = slice(a, a + n)
        pp, mm, vv = P[sl].copy(), M[sl].copy(), V[sl].copy()
        o.adamw_step(pp, G[sl].copy(), mm, vv, step=3, seed=99, base_index=base, **HP)
        P[sl], M[sl], V[sl] = pp, mm, vv
    gathered = [None] * world
    dist.all_gather_object(gathered, (start, end, P, M, V))
    if rank == 0:
        np.savez(os.path.join(out_dir, "gathered.npz"),
                 **{f"{k}{r}": x for r, tup in enumerate(gathered) for k, x in zip("sePMV", tup)})
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_two_gloo_ranks_equal_whole(tmp_path):
    import torch.multiprocessing as mp

    import oracle
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    d = np.load(tmp_path / "gathered.npz")
    p, g, m, v = _data()
    o = oracle.get()
    o.adamw_step(p, g, m, v, step=3, seed=99, base_index=0, **HP)
    covered = 0
    for r in range(world):
        s, e = int(d[f"s{r}"]), int(d[f"e{r}"])
        assert s == covered, "shards must be contiguous"
        covered = e
        assert np.array_equal(d[f"P{r}"], p[s:e])
        assert np.array_equal(d[f"M{r}"].view(np.uint32), m[s:e].view(np.uint32))
        assert np.array_equal(d[f"V{r}"].view(np.uint32), v[s:e].view(np.uint32))
    assert covered == len(p)


@pytest.mark.parametrize("total,world", [(0, 1), (1, 3), (10, 4), (8_030_261_248, 8), (1001, 7)])
def test_shard_bounds_partition(total, world):
    prev = 0
    for r in range(world):
        s, e = sharding.shard_bounds(total, world, r)
        assert s == prev and s <= e
        assert s % 4 == 0 or s == total
        prev = e
    assert prev == total


def test_shard_pieces_cover_range():
    total = sum(SIZES)
    for start, end in ((0, total), (3, 4100), (4096, 4097), (total - 5, total), (10, 10)):
        pieces = sharding.shard_pieces(SIZES, start, end)
        assert sum(n for _, _, n, _ in pieces) == end - start
        pos = start
        for t, off, n, base in pieces:
            assert base == pos and 0 <= off and off + n <= SIZES[t]
            pos += n


def _optim_rank_main(rank, world, port, out_dir):
    """One rank: an AdamWSR over the pieces of its share of the flat vector
    (cut on any element, align=1), numbered from the share's start."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch
    import torch.distributed as dist

    from stochastic_rounding_gb300.optim import AdamWSR
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    start, end = sharding.shard_bounds(sum(SIZES), world, rank, align=1)
    pieces = sharding.shard_pieces(SIZES, start, end)
    params = [torch.nn.Parameter(torch.zeros(n, dtype=torch.bfloat16)) for _, _, n, _ in pieces]
    opt = AdamWSR(params, base_offset=start)
    mine = [(t, off, n, opt.base_index(p)) for (t, off, n, _), p in zip(pieces, params)]
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        import json
        with open(os.path.join(out_dir, "positions.json"), "w") as f:
            json.dump(gathered, f)
    dist.barrier()
    dist.destroy_process_group()


def test_rank_local_optimizers_number_like_the_whole(tmp_path):
    """Three gloo ranks, each holding an AdamWSR over its share of the flat
    parameter vector cut at arbitrary elements and given the share's start
    as base_offset: every piece's global position equals the position of the
    same elements in one optimizer over the whole model, and the pieces tile
    the vector exactly once."""
    import json

    import torch
    import torch.multiprocessing as mp

    from stochastic_rounding_gb300.optim import AdamWSR
    world = 3
    mp.start_processes(_optim_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    with open(tmp_path / "positions.json") as f:
        gathered = json.load(f)
    whole = AdamWSR([torch.nn.Parameter(torch.zeros(n, dtype=torch.bfloat16)) for n in SIZES])
    starts = [whole.base_index(p) for p in whole.param_groups[0]["params"]]
    seen = []
    for rank_pieces in gathered:
        for t, off, n, pos in rank_pieces:
            assert pos == starts[t] + off
            seen.append((pos, n))
    seen.sort()
    covered = 0
    for pos, n in seen:
        assert pos == covered
        covered += n
    assert covered == sum(SIZES)
    assert any(pos % 4 for pos, _ in seen), "expected cuts off a multiple of 4"
