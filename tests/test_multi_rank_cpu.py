"""The N > 1 path of bench.py on CPU, over gloo with world size 2.

Every rank runs its own batch (weak scaling: the sequences shard across GPUs
with no data-path collective), seeded by its rank; the step time is the max
over ranks and the throughput counts the tokens of all ranks. These tests run
those host-side pieces in two processes on CPU (no GPU, no NCCL).
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from block_diffusion_decoding_attn_b300 import workload as wl
    w = wl.WORKLOADS["tiny_c256_l32"]
    inps = bench.attn_calls(w, seed=rank)
    cinp = wl.commit_inputs(w, seed=rank)
    # a per-rank step time; the reported one is the max over ranks
    ms = bench.max_over_ranks(1.0 + rank, dist)
    q.put((rank, ms, inps[0].q.tobytes()[:64], cinp.logits[0, :8].tobytes(),
           bench.tokens_per_step(w, len(inps), world)))
    dist.destroy_process_group()


def test_two_ranks_shard_batches_and_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, q0, l0, t0), (r1, ms1, q1, l1, t1) = res
    assert ms0 == ms1 == 2.0                 # max over ranks, the same on every rank
    assert q0 != q1 and l0 != l1             # each rank draws its own batch
    from block_diffusion_decoding_attn_b300 import workload as wl
    w = wl.WORKLOADS["tiny_c256_l32"]
    assert t0 == t1 == 2 * w.B * w.L         # whole-job tokens: both ranks' batches
