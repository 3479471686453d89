"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The decode step shards by sequence with no data-path collective: each rank owns
its own sequences, KV pool and block tables.  The only cross-rank operations are
the benchmark's barrier, the max of the per-rank step times and the sum of the
per-rank byte counts; this test runs them as two gloo ranks.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), PKV_DIST_BACKEND="gloo")
    import bench
    n, r, local = bench._dist()
    assert (n, r, local) == (world, rank, rank)
    bench._barrier(n)
    mx = bench._max_over_ranks(1.5 + rank, n, "cpu")
    sm = bench._sum_over_ranks(10.0 * (rank + 1), n, "cpu")
    # every rank builds its own shard of the workload: identical shape, own tables
    from paged_kv_decode_table_gb300 import workloads as W
    w = W.workload(2, batch=3, len_lo=20, len_hi=60)
    inp = W.make_decode_inputs(w, "cpu", with_logits=False)
    q.put((rank, mx, sm, int(inp["seq_lens"].sum())))
    torch.distributed.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_reduction():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, mx, sm, toks in res:
        assert mx == 2.5          # max over ranks of 1.5, 2.5
        assert sm == 30.0         # 10 + 20
    assert res[0][3] == res[1][3]  # same per-rank workload (weak scaling)
