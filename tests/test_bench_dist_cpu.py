"""bench.py's multi-process plumbing on CPU: two ranks over gloo, as torchrun
would launch them (RANK / WORLD_SIZE / MASTER_* from the environment). The
decode step is "replicas only" (no collective on the data path); the ranks
share only the barrier around the timed region and the max-over-ranks time."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _Args:
    impl = "reference"  # gloo backend


def _worker(rank: int, world: int, port: int, q) -> None:
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    w, r, local, pg = bench.dist_setup(_Args)
    bench.barrier(pg)
    m = bench.max_over_ranks(pg, float(r) + 1.5)
    bench.barrier(pg)
    q.put((r, w, local, m))
    pg.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == g[0] for g in got)
    # every rank sees the maximum over ranks (rank 1's 2.5)
    assert all(g[3] == pytest.approx(2.5) for g in got)


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    w, r, local, pg = bench.dist_setup(_Args)
    assert (w, r, local, pg) == (1, 0, 0, None)
    assert bench.max_over_ranks(pg, 3.25) == 3.25
