"""Layer variants and the expert-parallel split on the GPU, against the oracle.

- Activations (GeGLU, GeGLU in its tanh form, clamped SwiGLU) on the single
  launch, its chunks, the grouped path's GEMV and tcgen05 variants and the
  f32 check path.
- 6-bit down planes (4-bit gate/up) on the grouped path, GEMV and tcgen05
  variants and the f32 check path (the single launch declines them).
- Expert-parallel shards: G plans over a partition of the experts, each
  writing an f32 partial; each partial matches the oracle on planes whose
  non-owned experts are zeroed, and the partials summed on the device match
  the whole step. Routing is the same in every shard; the grouping arrays
  cover the owned experts.
"""
import numpy as np
import pytest

import quantized_moe_decode_softmax_gb300 as q
from gpu_cases import (TOL_BF16, TOL_F32, assert_out_close, assert_routing_equal, case,
                       device_layer, make_plan, path_name, planes_owned, record_margin, rms,
                       run_gpu, run_oracle, x_tensor)

pytestmark = pytest.mark.gpu

F32_DEBUG = q.MOE_FLAG_F32_DEBUG
GROUPED = q.MOE_FLAG_GROUPED_COHORTS
ACTS = {"geglu": q.MOE_ACT_GEGLU, "geglu_tanh": q.MOE_ACT_GEGLU_TANH,
        "swiglu_clamped": q.MOE_ACT_SWIGLU_CLAMPED}
# clamp bounds near the pre-activations' standard deviation, so that the clamp
# acts on about a third of the gate and up values
LIMIT = {"qwen3": 0.75, "e256": 0.75, "tiny": 0.25, "dots": 0.35}


def _check(shape_name, seed, n, kind="independent", full=False, flags=0, out_dtype=None,
           mma_min_tokens=0, act="swiglu", tol=None):
    import os
    lay, x = case(shape_name, seed, n, kind, full=full)
    shape = lay.shape
    a = ACTS.get(act, q.MOE_ACT_SWIGLU)
    limit = LIMIT[shape_name] if act == "swiglu_clamped" else 0.0
    ref = run_oracle(lay, x, activation=a, limit=limit)
    plan = make_plan(shape, flags=flags, out_dtype=out_dtype, mma_min_tokens=mma_min_tokens,
                     activation=a, act_limit=limit)
    launches = []
    out, routing = run_gpu(plan, device_layer(lay), shape, x, launches)
    assert_routing_equal(routing, ref)
    tol = tol or (TOL_F32 if flags & F32_DEBUG else TOL_BF16)
    err_rel = float(np.abs(out.astype(np.float64) - ref["out"]).max()) / max(rms(ref["out"]), 1e-30)
    path = path_name(n, launches[0], flags) + (f", tensor-core threshold {mma_min_tokens}" if mma_min_tokens else "")
    record_margin(os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], shape_name, n, kind,
                  path + f", {act}", out_dtype, tol, err_rel)
    assert_out_close(out, ref["out"], tol)


@pytest.mark.parametrize("act", sorted(ACTS))
@pytest.mark.parametrize("n,kind,flags,mma", [
    (1, "independent", 0, 0),          # single launch
    (8, "shared", 0, 0),               # single launch, 8 tokens on 8 experts
    (12, "independent", 0, 0),         # chunks of the single launch
    (24, "independent", 0, 0),         # grouped, GEMV variant
    (24, "shared", GROUPED, 0),        # grouped, tcgen05 GEMMs (24 tokens per expert)
    (4, "independent", F32_DEBUG, 0),  # f32 check path
])
def test_activation_variants_qwen3(act, n, kind, flags, mma):
    _check("qwen3", 2, n, kind, flags=flags, mma_min_tokens=mma, act=act,
           out_dtype="f32" if flags & F32_DEBUG else None)


@pytest.mark.parametrize("act", sorted(ACTS))
def test_activation_variants_other_shapes(act):
    _check("tiny", 0, 3, full=True, act=act)                            # grouped, f32 x
    _check("tiny", 0, 12, full=True, act=act, flags=GROUPED, mma_min_tokens=1)  # tcgen05 GEMMs
    _check("e256", 3, 4, act=act)                                       # single launch, D = 4096


@pytest.mark.parametrize("n,flags,mma,out_dtype", [
    (1, 0, 0, None),             # grouped (the single launch declines 6-bit down)
    (3, 0, 0, None),
    (12, GROUPED, 1, None),      # tcgen05 GEMMs for every expert
    (5, F32_DEBUG, 0, "f32"),    # f32 check path
])
def test_six_bit_down_planes(n, flags, mma, out_dtype):
    _check("dots", 5, n, full=True, flags=flags, mma_min_tokens=mma, out_dtype=out_dtype)


def test_six_bit_down_planes_qwen3_shape():
    _check("qwen3_d6", 2, 1)
    _check("qwen3_d6", 2, 16, "shared", mma_min_tokens=8)
    _check("qwen3_d6", 2, 4, act="geglu")


def test_six_bit_down_planes_take_the_grouped_path():
    import torch
    lay, x = case("dots", 5, 2, full=True)
    plan = make_plan(lay.shape)
    c0 = q.moe_plan_launch_count(plan.plan)
    plan.forward(x_tensor(lay.shape, x), device_layer(lay))
    torch.cuda.synchronize()
    assert q.moe_plan_launch_count(plan.plan) - c0 > 1


def _expected_shard_grouping(ref, lo, hi, E):
    counts = np.array(ref["counts"], np.int64)
    counts[:lo] = 0
    counts[hi:] = 0
    offsets = np.concatenate([[0], np.cumsum(counts)])
    a, b = int(ref["offsets"][lo]), int(ref["offsets"][hi])
    unique = np.array([e for e in ref["unique"] if lo <= e < hi], np.int32)
    return dict(counts=counts, offsets=offsets, slot_token=ref["slot_token"][a:b],
                slot_k=ref["slot_k"][a:b], unique=unique, U=len(unique))


@pytest.mark.parametrize("G", [2, 3])
@pytest.mark.parametrize("shape_name,n,kind,flags,mma", [
    ("qwen3", 4, "independent", 0, 0),        # single launch
    ("qwen3", 12, "independent", 0, 0),       # chunks of the single launch
    ("qwen3", 24, "independent", 0, 0),       # grouped, GEMV variant
    ("qwen3", 24, "shared", GROUPED, 0),      # grouped, tcgen05 GEMMs
    ("qwen3", 4, "independent", F32_DEBUG, 0),  # f32 check path
    ("dots", 6, "independent", 0, 0),         # 6-bit down planes
])
def test_expert_shards_sum_to_the_step(G, shape_name, n, kind, flags, mma):
    import torch
    lay, x = case(shape_name, 2 if shape_name == "qwen3" else 5, n, kind, full=shape_name == "dots")
    shape = lay.shape
    E = shape.E
    dl = device_layer(lay)
    xt = x_tensor(shape, x)
    full = run_oracle(lay, x)
    scale = rms(full["out"])
    tol = TOL_F32 if flags & F32_DEBUG else TOL_BF16
    total = torch.zeros((n, shape.D), dtype=torch.float32, device="cuda")
    for g in range(G):
        lo, hi = g * E // G, (g + 1) * E // G
        plan = make_plan(shape, flags=flags, out_dtype="f32", mma_min_tokens=mma, experts=(lo, hi))
        part = plan.forward(xt, dl)
        torch.cuda.synchronize()
        plan.check()
        total += part
        r = plan.routing(n)
        assert np.array_equal(r["topk_idx"], full["topk_idx"])
        assert np.abs(r["topk_w"] - full["topk_w"]).max() <= 1e-6
        want = _expected_shard_grouping(full, lo, hi, E)
        for key in ("counts", "offsets", "unique"):
            assert np.array_equal(r[key], want[key]), (g, key)
        S = int(want["offsets"][-1])
        assert np.array_equal(r["slot_token"][:S], want["slot_token"]), g
        assert np.array_equal(r["slot_k"][:S], want["slot_k"]), g
        assert r["U"] == want["U"]
        pref = run_oracle(lay, x, planes=planes_owned(lay, lo, hi))
        err = float(np.abs(part.cpu().numpy().astype(np.float64) - pref["out"]).max())
        assert err <= tol * scale, (g, err / scale)
    err = float(np.abs(total.cpu().numpy().astype(np.float64) - full["out"]).max())
    assert err <= tol * scale, err / scale
