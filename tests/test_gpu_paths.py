"""Which path runs, and the device-side timeout (GPU)."""
import time

import numpy as np
import pytest

import quantized_moe_decode_softmax_gb300 as q
from gpu_cases import (TOL_BF16, assert_out_close, assert_routing_equal, case, device_layer,
                       make_plan, run_gpu, run_oracle, x_tensor)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,flags,launches", [(1, 0, 1), (4, 0, 1), (8, 0, 1), (9, 0, 3), (16, 0, 3),
                                               (17, 0, 6), (64, 0, 6),
                                               (9, q.MOE_FLAG_GROUPED_COHORTS, 6)])
def test_launches_per_step(n, flags, launches):
    """Cohorts of up to 8 tokens run as one fused launch; 9..16 tokens as
    chunks of at most 8 plus one grouping kernel; larger cohorts (or any
    cohort above 8 with the grouped flag) take the multi-kernel path (router,
    grouping, x to f16, the tcgen05 gate/up and down GEMMs, combine; with the
    default threshold of one token no expert is left for the GEMV kernels)."""
    import torch
    lay, x = case("qwen3", 2, n)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, flags=flags)
    c0 = q.moe_plan_launch_count(plan.plan)
    plan.forward(x_tensor(shape, x), dl)
    torch.cuda.synchronize()
    assert q.moe_plan_launch_count(plan.plan) - c0 == launches


def test_chunked_matches_grouped_path():
    """The same 13-token cohort through chunks of the single-launch kernel and
    through the grouped path: identical routing tables, outputs within the
    bf16 tolerance."""
    lay, x = case("qwen3", 2, 13)
    shape = lay.shape
    dl = device_layer(lay)
    a, r_a = run_gpu(make_plan(shape, out_dtype="f32"), dl, shape, x)
    b, r_b = run_gpu(make_plan(shape, flags=q.MOE_FLAG_GROUPED_COHORTS, out_dtype="f32"), dl, shape, x)
    assert_routing_equal(r_a, r_b)
    assert_out_close(a, b, TOL_BF16)


def test_fused_matches_f32_check_path():
    """The fused path and the f32 check path agree on one cohort."""
    lay, x = case("qwen3", 2, 6)
    shape = lay.shape
    dl = device_layer(lay)
    fast, r_fast = run_gpu(make_plan(shape, out_dtype="f32"), dl, shape, x)
    slow, r_slow = run_gpu(make_plan(shape, flags=q.MOE_FLAG_F32_DEBUG, out_dtype="f32"), dl, shape, x)
    assert_routing_equal(r_fast, r_slow)
    assert_out_close(fast, slow, TOL_BF16)


def test_device_wait_times_out_and_context_stays_usable():
    """A grid barrier that one CTA reaches only after the others' bounded waits
    gave up: moe_plan_check reports MOE_ERR_TIMEOUT, and the NEXT step on the
    SAME plan (whose barrier counter the stalled step left behind) matches the
    oracle. No GPU fault or hang is involved: every wait is bounded."""
    import torch
    lay, x = case("qwen3", 2, 2)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, flags=q.MOE_FLAG_TEST_STALL)
    t0 = time.time()
    plan.forward(x_tensor(shape, x), dl)
    with pytest.raises(q.MoeError) as ei:
        plan.check()
    assert ei.value.status == q.MOE_ERR_TIMEOUT
    assert time.time() - t0 < 30
    ref = run_oracle(lay, x)
    for _ in range(2):  # the same plan, twice
        out, routing = run_gpu(plan, dl, shape, x)
        assert_routing_equal(routing, ref)
        assert_out_close(out, ref["out"], TOL_BF16)
    torch.cuda.synchronize()


def test_timeout_is_reported_by_the_next_forward_call():
    """The stalled step has finished on the device: the next forward call on the
    plan returns MOE_ERR_TIMEOUT without launching, and the call after it runs
    normally and matches the oracle (no moe_plan_check in between)."""
    import torch
    lay, x = case("qwen3", 2, 3)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, flags=q.MOE_FLAG_TEST_STALL)
    xt = x_tensor(shape, x)
    plan.forward(xt, dl)
    torch.cuda.synchronize()
    c0 = q.moe_plan_launch_count(plan.plan)
    with pytest.raises(q.MoeError) as ei:
        plan.forward(xt, dl)
    assert ei.value.status == q.MOE_ERR_TIMEOUT
    assert q.moe_plan_launch_count(plan.plan) == c0
    ref = run_oracle(lay, x)
    out, routing = run_gpu(plan, dl, shape, x)  # also runs moe_plan_check: clear
    assert_routing_equal(routing, ref)
    assert_out_close(out, ref["out"], TOL_BF16)


def test_phase_times_are_ordered():
    """Per-CTA timestamps of the fused step's phases are non-decreasing."""
    import torch
    lay, x = case("qwen3", 2, 4)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, flags=q.MOE_FLAG_PHASE_TIMES)
    plan.forward(x_tensor(shape, x), dl)
    torch.cuda.synchronize()
    t = q.moe_get_phase_times(plan.plan)
    assert t.shape[0] >= 1 and t.shape[1] == 16
    assert np.all(np.diff(t[:, :8], axis=1) >= 0)
    assert np.all(t[:, 0] > 0)


@pytest.mark.parametrize("n", [1, 4, 24])
def test_layer_chain_matches_the_oracle_per_layer(n):
    """moe_decode_forward_layers over three layers with their own weights and
    cohorts: each layer's output matches the oracle (single launch for n <= 8,
    the grouped path for 24), and the chain launches what the three separate
    calls would."""
    import torch
    import moe_synth as ms
    shape = ms.SHAPES["qwen3"]
    steps, refs = [], []
    for l in range(3):
        router_w, bias = ms.draw_router(shape, 70 + l, 0)
        x = ms.draw_tokens(shape, router_w, bias, 70 + l, 0, n)
        lay = ms.make_layer(shape, 70 + l, 0, ms.routed_experts(x, router_w, bias, shape.top_k))
        refs.append(run_oracle(lay, x))
        out = torch.empty((n, shape.D), dtype=torch.bfloat16, device="cuda")
        steps.append((x_tensor(shape, x), device_layer(lay), out))
    plan = make_plan(shape)
    c0 = q.moe_plan_launch_count(plan.plan)
    plan.forward_layers(steps)
    torch.cuda.synchronize()
    plan.check()
    chain_launches = q.moe_plan_launch_count(plan.plan) - c0
    for (_, _, out), ref in zip(steps, refs):
        assert_out_close(out.float().cpu().numpy(), ref["out"], TOL_BF16)
    assert_routing_equal(plan.routing(n), refs[-1])
    c1 = q.moe_plan_launch_count(plan.plan)
    for x, dl, out in steps:
        plan.forward(x, dl, out)
    torch.cuda.synchronize()
    assert q.moe_plan_launch_count(plan.plan) - c1 == chain_launches


def test_layer_chain_checks_every_layer_before_launching():
    import torch
    lay, x = case("qwen3", 2, 2)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape)
    xt = x_tensor(shape, x)
    out = torch.empty((2, shape.D), dtype=torch.bfloat16, device="cuda")
    c0 = q.moe_plan_launch_count(plan.plan)
    with pytest.raises(q.MoeError) as ei:  # the third layer's out aliases its x
        plan.forward_layers([(xt, dl, out), (xt, dl, out.clone()), (xt, dl, xt)])
    assert ei.value.status == q.MOE_ERR_INVALID_ARG
    assert q.moe_plan_launch_count(plan.plan) == c0
