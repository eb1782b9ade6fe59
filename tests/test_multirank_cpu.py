"""The bench's multi-rank plumbing on CPU: world size 2 over gloo, no GPU.

`bench.py --gpus N` runs N independent replicas of the single-GPU path (the tensor-parallel
shards are logical, on one device each): a barrier brackets the timed region, each rank's
time is reduced with MAX, and only rank 0 prints.  The replicas have no data-path
collective, so the host logic is all there is to check across ranks."""
import io
import os
import socket
import sys
import contextlib

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "BENCH_BACKEND": "gloo"})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each rank's "time" differs; every rank must see the maximum
    m = bench.max_over_ranks(1.5 + rank, w, "cpu")
    # the reference arm prints on rank 0 only; the other ranks return without work
    out = io.StringIO()

    class A:
        steps, warmup = 1, 3
    if rank != 0:
        with contextlib.redirect_stdout(out):
            bench.run_reference(A, rank, w)
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((rank, m, out.getvalue()))


def test_two_ranks_barrier_max_and_rank0_output():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(m == pytest.approx(2.5) for _, m, _ in res)     # the max over ranks
    assert res[1][2] == ""                                       # rank 1 printed nothing
