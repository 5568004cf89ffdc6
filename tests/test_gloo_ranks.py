"""The multi-rank path of bench.py on CPU (gloo, world size 2).

Requests are independent, so the verification shards by request with no
data exchange: each rank verifies its own batch (weak scaling) and only the
timing crosses ranks, as a max. This test runs those pieces on two gloo ranks
with the CPU oracle standing in for the GPU work (test infrastructure only):
the max-over-ranks reduction, the per-rank seeds, and the independence of
requests (a batch split across ranks gives, concatenated, the result of one
process on the whole batch).
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    import oracle
    from workloads import synthetic
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synthetic.WORKLOADS[4].variant(B=12, V=512)
    # weak scaling: this rank's own batch
    mine = synthetic.generate(w, k=bench.rank_seed_k(rank))
    o_mine, n_mine, _ = oracle.verify(*mine.arrays())
    # timing: every rank learns the slowest rank's time
    slowest = bench.max_over_ranks(10.0 * (rank + 1), dist)
    # request independence: rank r verifies half of one shared batch
    shared = synthetic.generate(w, k=7)
    lo, hi = rank * w.B // world, (rank + 1) * w.B // world
    o_half, n_half, _ = oracle.verify(*shared.slice(lo, hi).arrays())
    gathered = [None] * world
    dist.all_gather_object(gathered, (o_half, n_half))
    if rank == 0:
        np.savez(os.path.join(out_dir, "rank0.npz"), slowest=slowest,
                 o_cat=np.concatenate([g[0] for g in gathered]),
                 n_cat=np.concatenate([g[1] for g in gathered]), o_mine=o_mine, n_mine=n_mine)
    else:
        np.savez(os.path.join(out_dir, "rank1.npz"), slowest=slowest, o_mine=o_mine, n_mine=n_mine)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path, oracle_lib):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    import oracle
    from workloads import synthetic
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    assert float(r0["slowest"]) == 20.0 and float(r1["slowest"]) == 20.0
    w = synthetic.WORKLOADS[4].variant(B=12, V=512)
    o_all, n_all, _ = oracle.verify(*synthetic.generate(w, k=7).arrays())
    assert np.array_equal(r0["o_cat"], o_all) and np.array_equal(r0["n_cat"], n_all)
    for k, r in ((0, r0), (1, r1)):
        o, n, _ = oracle.verify(*synthetic.generate(w, k=k).arrays())
        assert np.array_equal(r["o_mine"], o) and np.array_equal(r["n_mine"], n)
    # the two ranks verified different batches
    assert not np.array_equal(r0["o_mine"], r1["o_mine"])
