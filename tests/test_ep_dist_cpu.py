"""The expert-parallel exchange step on CPU: two ranks over gloo.

Each rank takes its expert range from shard_bounds, computes its partial with
the oracle on planes whose non-owned experts are zeroed (their outputs are
then exactly 0, routing unchanged), and the ranks sum the partials with the
library's all-reduce helper. Every rank must then hold the whole step's output
(the oracle on the full planes) to f32 rounding. No GPU is involved."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SHAPE = dict(E=16, top_k=4, D=256, F=128, act_dtype="f32", router_std=0.08)


def _worker(rank: int, world: int, port: int, q) -> None:
    import torch
    import torch.distributed as dist

    import moe_synth as ms
    import oracle
    from quantized_moe_decode_softmax_gb300.ep import allreduce_partials, shard_bounds
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    shape = ms.LayerShape(**SHAPE)
    lay = ms.make_layer(shape, 41, 0)
    x = ms.draw_tokens(shape, lay.router_w, None, 41, 0, 5)
    lo, hi = shard_bounds(shape.E, world, rank)
    arrs = []
    for name, a in zip(ms.ExpertPlanes.FIELDS, lay.planes.arrays()):
        a = a.copy()
        if not name.endswith("_q"):
            a[:lo] = 0
            a[hi:] = 0
        arrs.append(a)
    part = oracle.moe_forward(x, lay.router_w, None, ms.ExpertPlanes(*arrs), shape.top_k)
    full = oracle.moe_forward(x, lay.router_w, None, lay.planes, shape.top_k)
    t = torch.from_numpy(part["out"].copy())
    allreduce_partials(t)
    err = float(np.abs(t.numpy().astype(np.float64) - full["out"]).max())
    rms = float(np.sqrt(np.mean(np.square(full["out"].astype(np.float64)))))
    same_routing = bool(np.array_equal(part["topk_idx"], full["topk_idx"]))
    q.put((rank, (lo, hi), err / rms, same_routing))
    dist.destroy_process_group()


def test_two_ranks_sum_their_expert_partials():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [g[1] for g in got] == [(0, 8), (8, 16)]
    for rank, _, rel, same in got:
        assert same, rank
        assert rel <= 1e-6, (rank, rel)


@pytest.mark.parametrize("E,world", [(128, 1), (128, 2), (128, 3), (256, 8), (7, 7)])
def test_shard_bounds_partition_the_experts(E, world):
    from quantized_moe_decode_softmax_gb300.ep import shard_bounds
    bounds = [shard_bounds(E, world, r) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == E
    assert all(a[1] == b[0] for a, b in zip(bounds, bounds[1:]))
    sizes = [b - a for a, b in bounds]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1


def test_shard_bounds_rejects_impossible_splits():
    from quantized_moe_decode_softmax_gb300.ep import shard_bounds
    for E, world, rank in ((4, 5, 0), (8, 2, 2), (8, 0, 0)):
        with pytest.raises(ValueError):
            shard_bounds(E, world, rank)
