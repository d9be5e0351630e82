"""The multi-GPU path of the bench on the CPU: two gloo ranks, no GPU.

The hot path shards with no exchange (every sequence and kv head is independent), so N GPUs run N
replica batches (weak scaling) and only host scalars cross ranks: the max of the timed region and the
sum of the work.  This checks those reductions and that each rank gets its own batch."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        b = bench.rank_decode_batch(rank, num_seqs=8)
        kv = bench.decode_kv_bytes(b)
        total = bench.reduce_over_ranks(float(kv), "sum", world)
        slowest = bench.reduce_over_ranks(float(10 + rank), "max", world)
        out.put((rank, kv, total, slowest, [int(x) for x in b.seq_lens]))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, kv0, tot0, max0, lens0), (r1, kv1, tot1, max1, lens1) = res
    assert tot0 == tot1 == float(kv0 + kv1)          # whole-job work is the sum over ranks
    assert max0 == max1 == 11.0                      # the job time is the slowest rank's
    assert lens0 != lens1                            # each rank draws its own batch


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, "max", 1) == 3.5
    assert bench.reduce_over_ranks(3.5, "sum", 1) == 3.5
