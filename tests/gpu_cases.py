"""Shared helpers for the GPU parity tests: seeded cases, the device run
through the C ABI, the oracle run, and the comparisons."""
from __future__ import annotations

import functools
import os

import numpy as np

import moe_synth as ms
import oracle

# tolerance on bf16 outputs and on the tensor-core path: 2e-2 * RMS(out)
TOL_BF16 = 2e-2
# tolerance of the f32 check path (MOE_FLAG_F32_DEBUG): 1e-4 * RMS(out)
TOL_F32 = 1e-4
# routing weights: absolute
TOL_W = 1e-6

WORKERS = max(1, min(16, (os.cpu_count() or 2)))


def rms(a) -> float:
    return float(np.sqrt(np.mean(np.square(np.asarray(a, np.float64)))))


@functools.lru_cache(maxsize=None)
def full_layer(shape_name: str, seed: int, layer: int = 0):
    """All experts drawn (cached per process)."""
    return ms.make_layer(ms.SHAPES[shape_name], seed, layer, workers=WORKERS)


def case(shape_name: str, seed: int, n: int, kind: str = "independent", cohort: int = 0,
         full: bool = False):
    """(layer, x). full=False draws only the routed experts' planes."""
    shape = ms.SHAPES[shape_name]
    if full:
        lay = full_layer(shape_name, seed)
        x = ms.draw_tokens(shape, lay.router_w, lay.router_bias, seed, 0, n, kind, cohort)
        return lay, x
    return ms.make_case(shape_name, seed, n, kind, cohort=cohort, lazy=True,
                        workers=WORKERS if n * ms.SHAPES[shape_name].top_k > 16 else 1)


def device_layer(lay):
    from quantized_moe_decode_softmax_gb300 import DeviceLayer
    return DeviceLayer.from_host(ms.router_storage(lay.shape, lay.router_w), lay.router_bias,
                                 lay.planes, lay.shape.top_k)


def x_tensor(shape, x):
    import torch
    st = ms.x_storage(shape, x)
    if st.dtype == np.uint16:
        return torch.from_numpy(st.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(st).cuda()


def make_plan(shape, flags=0, out_dtype=None, max_tokens=64, mma_min_tokens=0, activation=0,
              act_limit=0.0, experts=None):
    from quantized_moe_decode_softmax_gb300 import MoeDecodeLayer
    return MoeDecodeLayer(shape.E, shape.top_k, shape.D, shape.F, max_tokens=max_tokens,
                          act_dtype=shape.act_dtype, out_dtype=out_dtype, flags=flags,
                          mma_min_tokens=mma_min_tokens, activation=activation,
                          act_limit=act_limit, down_bits=shape.down_bits, experts=experts)


# measured parity margins of this session: one dict per compared output
MARGINS: list = []


def path_name(n, launches, flags=0):
    """Which path a forward call took, from the kernels it launched."""
    if flags & 1:
        return "grouped, f32 check path"
    if launches == 1:
        return "single launch"
    if 9 <= n <= 16 and launches == (n + 7) // 8 + 1:
        return f"chunks of the single launch ({(n + 7) // 8})"
    return "grouped multi-kernel"


def record_margin(test, shape_name, n, kind, path, out_dtype, tol, err_rel):
    MARGINS.append(dict(test=test, shape=shape_name, n=int(n), kind=kind, path=path,
                        out=out_dtype or "act", tol=tol, err_rel=err_rel,
                        used=err_rel / tol if tol else None))


def run_gpu(plan, dl, shape, x, launches=None):
    """Forward through the C ABI; `launches` (a list) receives the kernel count."""
    import torch
    from quantized_moe_decode_softmax_gb300 import moe_plan_launch_count
    xt = x_tensor(shape, x)
    c0 = moe_plan_launch_count(plan.plan)
    out = plan.forward(xt, dl)
    torch.cuda.synchronize()
    plan.check()
    if launches is not None:
        launches.append(moe_plan_launch_count(plan.plan) - c0)
    return out.float().cpu().numpy(), plan.routing(x.shape[0])


def run_oracle(lay, x, activation=0, limit=0.0, planes=None):
    return oracle.moe_forward(x, lay.router_w, lay.router_bias, lay.planes if planes is None else planes,
                              lay.shape.top_k, want_bf16=True, activation=activation, limit=limit,
                              down_bits=lay.shape.down_bits)


def planes_owned(lay, lo, hi):
    """The layer's planes with the scales and biases of every expert outside
    [lo, hi) zeroed: those experts' weights are all 0, so their outputs are
    exactly 0 and the oracle step is the shard's partial (routing unchanged)."""
    arrs = []
    for name, a in zip(ms.ExpertPlanes.FIELDS, lay.planes.arrays()):
        a = a.copy()
        if not name.endswith("_q"):
            a[:lo] = 0
            a[hi:] = 0
        arrs.append(a)
    return ms.ExpertPlanes(*arrs)


def assert_routing_equal(r, ref):
    assert np.array_equal(r["topk_idx"], ref["topk_idx"]), "top-k indices differ"
    assert np.abs(r["topk_w"] - ref["topk_w"]).max() <= TOL_W, "routing weights differ"
    for key in ("counts", "offsets", "slot_token", "slot_k", "unique"):
        assert np.array_equal(r[key], ref[key]), f"{key} differs"
    assert r["U"] == ref["U"]


def assert_out_close(out, ref_out, tol):
    err = float(np.abs(out.astype(np.float64) - ref_out.astype(np.float64)).max())
    bound = tol * rms(ref_out)
    assert err <= bound, f"max|err| {err:.3e} > {tol} * RMS = {bound:.3e}"
    return err / max(rms(ref_out), 1e-30)
