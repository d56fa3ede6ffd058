"""The prefill path: cohorts of more than 64 tokens (a grouped GEMM per expert).

Routing is bit-exact against the oracle, grouping too (token bitmaps per
expert give the oracle's order: experts ascending, tokens ascending), and the
outputs are within the bf16 tolerance (the tcgen05 GEMMs for experts with at
least mma_min_tokens tokens, looping over each expert's tokens in blocks of
64) or the f32 tolerance (the f32 check path). Sizes span several token
blocks per expert and ragged tails.
"""
import numpy as np
import pytest

import quantized_moe_decode_softmax_gb300 as q
from gpu_cases import (TOL_BF16, TOL_F32, assert_out_close, assert_routing_equal, case,
                       device_layer, make_plan, planes_owned, record_margin, rms, run_gpu,
                       run_oracle)

pytestmark = pytest.mark.gpu


def _check(shape_name, seed, n, kind="independent", full=False, flags=0, out_dtype=None,
           experts=None):
    import os
    lay, x = case(shape_name, seed, n, kind, full=full)
    shape = lay.shape
    ref = run_oracle(lay, x)
    plan = make_plan(shape, flags=flags, out_dtype=out_dtype, max_tokens=max(n, 64))
    launches = []
    out, routing = run_gpu(plan, device_layer(lay), shape, x, launches)
    assert_routing_equal(routing, ref)
    tol = TOL_F32 if flags & q.MOE_FLAG_F32_DEBUG else TOL_BF16
    err_rel = float(np.abs(out.astype(np.float64) - ref["out"]).max()) / max(rms(ref["out"]), 1e-30)
    record_margin(os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], shape_name, n, kind,
                  "prefill (grouped GEMM)" + (", f32 check path" if flags & q.MOE_FLAG_F32_DEBUG else ""),
                  out_dtype, tol, err_rel)
    assert_out_close(out, ref["out"], tol)
    return launches[0]


@pytest.mark.parametrize("n,kind", [(65, "independent"), (128, "independent"), (300, "independent"),
                                    (256, "shared")])
def test_prefill_qwen3(n, kind):
    _check("qwen3", 2, n, kind)


def test_prefill_small_layer_many_tokens_per_expert():
    # E=8, top-2: about 250 tokens per expert, four token blocks each
    _check("tiny", 0, 1000, full=True)
    _check("tiny", 0, 1000, full=True, flags=q.MOE_FLAG_F32_DEBUG, out_dtype="f32")


def test_prefill_many_experts_and_slots():
    _check("e1024", 5, 200, full=True)   # 3200 slots over 1024 experts


def test_prefill_six_bit_down_and_activation():
    lay, x = case("dots", 5, 160, full=True)
    shape = lay.shape
    ref = run_oracle(lay, x, activation=q.MOE_ACT_GEGLU)
    plan = make_plan(shape, max_tokens=160, activation=q.MOE_ACT_GEGLU)
    out, routing = run_gpu(plan, device_layer(lay), shape, x)
    assert_routing_equal(routing, ref)
    assert_out_close(out, ref["out"], TOL_BF16)


def test_prefill_expert_shards_sum_to_the_step():
    import torch
    lay, x = case("qwen3", 2, 96)
    shape = lay.shape
    dl = device_layer(lay)
    full = run_oracle(lay, x)
    total = np.zeros_like(full["out"], dtype=np.float64)
    for lo, hi in ((0, 64), (64, 128)):
        plan = make_plan(shape, out_dtype="f32", max_tokens=96, experts=(lo, hi))
        out, r = run_gpu(plan, dl, shape, x)
        assert np.array_equal(r["topk_idx"], full["topk_idx"])
        part = run_oracle(lay, x, planes=planes_owned(lay, lo, hi))
        assert np.abs(out - part["out"]).max() <= TOL_BF16 * rms(full["out"])
        total += out
    assert np.abs(total - full["out"]).max() <= TOL_BF16 * rms(full["out"])
    torch.cuda.synchronize()


def test_prefill_plan_runs_decode_cohorts_on_the_decode_paths():
    """A plan sized for prefill still runs n <= 8 as one single launch."""
    import torch
    lay, x = case("qwen3", 2, 4)
    shape = lay.shape
    plan = make_plan(shape, max_tokens=512)
    c0 = q.moe_plan_launch_count(plan.plan)
    out, routing = run_gpu(plan, device_layer(lay), shape, x)
    assert q.moe_plan_launch_count(plan.plan) - c0 == 1
    assert_out_close(out, run_oracle(lay, x)["out"], TOL_BF16)
    torch.cuda.synchronize()
