"""Two-rank (gloo, CPU) tests of the multi-GPU host logic: head sharding,
the max-over-ranks timing reduction and the whole-job aggregate, with each
rank computing its shard of a problem on the oracle."""
import os
import socket

import numpy as np
import pytest

from attention_forward_12_gb300 import multirank, synth

torch = pytest.importorskip("torch")


def test_shard_heads_cover_exactly():
    for BH in (0, 1, 5, 64, 129):
        for world in (1, 2, 3, 8):
            ranges = [multirank.shard_heads(BH, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == BH
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        multirank.shard_heads(4, 2, 2)


def test_aggregate_and_seeds():
    assert multirank.aggregate_tflops(1e12, 4, 1000.0) == pytest.approx(4.0)
    assert multirank.rank_seed(5, 0) == 5 and multirank.rank_seed(5, 1) != 5
    assert multirank.max_over_ranks(3.5) == 3.5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    B, H, N, D = 1, 5, 40, 16
    q, k, v = synth.make_qkv(B, H, N, N, D, seed=3)
    lo, hi = multirank.shard_heads(B * H, rank, world)
    qs, ks, vs = (x.reshape(B * H, 1, -1, D)[lo:hi].copy() for x in (q, k, v))
    O, L = oracle.attn_full(qs, ks, vs, 0.25, True, nthreads=1)
    np.save(os.path.join(out_dir, f"o{rank}.npy"), O.reshape(hi - lo, N, D))
    np.save(os.path.join(out_dir, f"l{rank}.npy"), L.reshape(hi - lo, N))
    slow = multirank.max_over_ranks(10.0 + rank, dist)
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([slow]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_shard_and_reduce(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    import oracle
    B, H, N, D = 1, 5, 40, 16
    q, k, v = synth.make_qkv(B, H, N, N, D, seed=3)
    O, L = oracle.attn_full(q, k, v, 0.25, True, nthreads=1)
    Og = np.concatenate([np.load(tmp_path / f"o{r}.npy") for r in range(world)])
    Lg = np.concatenate([np.load(tmp_path / f"l{r}.npy") for r in range(world)])
    assert np.array_equal(Og, O.reshape(B * H, N, D))
    assert np.array_equal(Lg, L.reshape(B * H, N))
    for r in range(world):
        assert float(np.load(tmp_path / f"t{r}.npy")[0]) == 11.0
