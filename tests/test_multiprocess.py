"""The N > 1 host path of bench.py on CPU: two gloo ranks, rendezvous on
127.0.0.1.  Each rank reads its place from the torchrun environment variables,
meets the other at the barriers that bracket the timed region, and takes the
maximum of the per-rank step times, as the benchmark does before rank 0
prints.  Attention itself needs no exchange between ranks (replicas only), so
no collective appears on the data path."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        bench.barrier(w)
        step_ms = 1.0 + 0.25 * r          # rank r's own timing
        results[r] = (w, r, local, bench.max_over_ranks(step_ms, w))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    assert sorted(got) == [0, 1]
    for r in range(world):
        w, rr, local, mx = got[r]
        assert (w, rr, local) == (world, r, r)
        assert mx == pytest.approx(1.25)
