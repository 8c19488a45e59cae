"""bench.py's multi-rank logic on CPU: two gloo ranks, max-over-ranks timing
and the weak-scaling value (no GPU; the data path has no collective)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]   # rank 1 slower in the first, faster in the second
    mx = bench.max_over_ranks(local_ms, torch.device("cpu"))
    value = bench.weak_scaling_value(64, 30, world, mx[0])
    out_q.put((rank, mx, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_sum_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, mx, value in res:
        assert mx == [15.0, 20.0]
        assert value == pytest.approx(64 * 30 * 2 / 0.015)
