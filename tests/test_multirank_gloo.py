"""The benchmark's multi-rank path on CPU: two gloo ranks, no GPU.

Ranks are independent replicas (each compresses its own sequence; weak scaling): the only
collectives are the barrier and the max over ranks of the timed region. This checks that host
logic with world_size 2: each rank gets the slowest rank's time, the whole-job value counts every
rank's units, the ranks' sequences (and so their inputs and results) are distinct, and the
reference arm prints only on rank 0.
"""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        from oracle import snapkv_oracle as orc

        # max over ranks: every rank sees the slowest rank's timed region
        mine = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(mine, world, torch.device("cpu"))
        assert slowest == 5.0
        assert bench.max_over_ranks(mine, 1, torch.device("cpu")) == mine
        # whole-job value: all ranks' units over the slowest rank's step time
        assert bench.whole_job_rate(1000.0, world, 5.0) == pytest.approx(2 * 1000.0 / 5e-3)

        # each rank compresses its own sequence: distinct inputs, independent results
        seq = bench.replica_sequence(rank)
        seqs = [None] * world
        dist.all_gather_object(seqs, seq)
        assert sorted(seqs) == list(range(world))
        # a batch workload: rank r takes sequences r*B .. r*B + B - 1, disjoint across ranks
        first = bench.replica_batch(rank, 8)
        firsts = [None] * world
        dist.all_gather_object(firsts, first)
        spans = [set(range(f, f + 8)) for f in firsts]
        assert not (spans[0] & spans[1]) and firsts[0] == 0
        wl = synth.WORKLOADS[0]
        hi = synth.host_head(wl, 0, seq, 0, l_prompt=wl.l_prompt, threads=1)
        ref = orc.compress_head(hi.q_obs, hi.k, hi.v, pool_kernel=wl.pool_kernel, ratio_p=wl.ratio_p)
        keys = [None] * world
        dist.all_gather_object(keys, (hi.k[:4].tobytes(), ref.idx.tolist()))
        assert keys[0][0] != keys[1][0]           # the replicas' inputs differ
        assert keys[0][1] != keys[1][1]           # and so do their selections
        assert len(keys[0][1]) == len(keys[1][1]) == orc.kept_slots(wl.l_prompt - wl.l_obs, wl.ratio_p)

        # the reference arm runs and prints on rank 0 only; other ranks exit without work
        if rank != 0:
            out = io.StringIO()
            with contextlib.redirect_stdout(out):
                bench.run_reference(None, rank, world)   # returns before reading any argument
            assert out.getvalue() == ""
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_as_independent_replicas():
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port), nprocs=2, join=True, start_method="spawn")
