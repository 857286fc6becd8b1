"""The multi-rank layout of the benchmark, on CPU with gloo (world size 2).

BRA routes each image on its own, so ranks shard the batch by image with no
collective on the data path; the only collective is the max over ranks of
the timed region. These tests run two gloo ranks and check that the shards
tile the batch and that the per-rank results, gathered, are exactly the
single-process result (computed with the oracle on each side).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bra_synth
import oracle

WORLD = 2
WL = bra_synth.Workload("shard", 2, 8, 8, 16, 2, 2, 2, 3, "f32")  # per-rank batch 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl_global = WL.replace(B=WL.B * world)
        x = bra_synth.make_inputs(wl_global, seed=9, batch=bra_synth.rank_slice(WL.B, rank))
        out, idx = oracle.forward(x.q, x.k, x.v, WL.heads, WL.S, WL.topk, x.lepe_w, x.lepe_b)
        # the timing reduction the benchmark uses: max over ranks
        t = torch.tensor([10.0 * (rank + 1)])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        outs = [None] * world if rank == 0 else None
        dist.gather_object((out, idx, float(t.item())), outs, dst=0)
        if rank == 0:
            np.save(result_path, np.array(outs, dtype=object), allow_pickle=True)
    finally:
        dist.destroy_process_group()


def test_rank_slices_tile_the_batch():
    cover = []
    for r in range(3):
        sl = bra_synth.rank_slice(4, r)
        cover.extend(range(sl.start, sl.stop))
    assert cover == list(range(12))


def test_sharded_forward_equals_single_process(tmp_path):
    path = str(tmp_path / "gathered.npy")
    mp.spawn(_worker, args=(WORLD, _free_port(), path), nprocs=WORLD, join=True)
    gathered = np.load(path, allow_pickle=True)
    wl_global = WL.replace(B=WL.B * WORLD)
    x = bra_synth.make_inputs(wl_global, seed=9)
    ref_out, ref_idx = oracle.forward(x.q, x.k, x.v, WL.heads, WL.S, WL.topk, x.lepe_w,
                                      x.lepe_b)
    out = np.concatenate([g[0] for g in gathered])
    idx = np.concatenate([g[1] for g in gathered])
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_array_equal(out, ref_out)  # same images, same arithmetic
    assert all(g[2] == 10.0 * WORLD for g in gathered)
