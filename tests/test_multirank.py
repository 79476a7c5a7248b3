"""The benchmark's N-process path on CPU (gloo, world size 2): requests are
sharded by rank (independent workloads, no collective on the data path), the
timing is the max over ranks, the row count is the sum, and the reference arm
returns at once, printing nothing, on every rank but 0."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from compressed_kv_attention_compressplan_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.5 + rank, world)
        rows = bench.sum_over_ranks(10.0 * (rank + 1), world)
        bench.barrier(world)
        # each rank draws its own independent requests (seed + rank)
        w = wl.c4_prefill(seed=rank, batch=4, head_dim=128, max_prefix=64, max_extend=64)
        # the reference arm: every rank but 0 returns at once, without work or output
        ref_out = None
        if rank != 0:
            import contextlib
            import io

            buf = io.StringIO()
            with contextlib.redirect_stdout(buf):
                assert bench.bench_reference(None, world, rank) is None
            ref_out = buf.getvalue()
        q.put((rank, t, rows, w.seq_lens.tolist(), ref_out))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_reduction_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, rows0, sl0, _), (r1, t1, rows1, sl1, ref1) = res
    assert t0 == t1 == 2.5            # max over ranks
    assert rows0 == rows1 == 30.0     # whole-job count
    assert sl0 != sl1                 # independent shards
    assert ref1 == ""                 # the reference arm printed nothing on rank 1


def test_reference_arm_other_ranks_do_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        seed = 0
        warmup = 0
        steps = 1
        ref_fraction = 0.1

    bench.bench_reference(A(), 2, 1)  # rank 1 of 2: returns at once, prints nothing
    assert capsys.readouterr().out == ""
