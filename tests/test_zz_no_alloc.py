"""The allocation-free entry point (moe_decode_forward_noalloc) against the
plan-based one, through the C ABI.

Callers that cannot allocate device memory (for example code running during
CUDA graph capture, or runtimes that own the device memory pool) use
moe_decode_forward_noalloc, whose scratch is a static device array of the
library. It runs the same kernel on the same inputs as moe_decode_forward, so
its output must equal that entry point's output bit for bit (which is within
the bf16 tolerance of the parity tests), on two calls in a row (the second
call reuses the array the first one left behind). This file is collected last
on purpose.
"""
import numpy as np
import pytest

import quantized_moe_decode_softmax_gb300 as q
from gpu_cases import TOL_BF16, assert_out_close, case, device_layer, make_plan, run_gpu, x_tensor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [1, 4])
def test_noalloc_matches_plan_entry_point_twice(n):
    import torch
    lay, x = case("qwen3", 2, n)
    shape = lay.shape
    dl = device_layer(lay)
    ref, _ = run_gpu(make_plan(shape), dl, shape, x)
    cfg = q.make_config(shape.E, shape.top_k, shape.D, shape.F, max_tokens=n)
    xt = x_tensor(shape, x)
    for _ in range(2):
        out = torch.full((n, shape.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        q.moe_decode_forward_noalloc(cfg, xt, dl.router_w, dl.router_bias, dl.c_planes, n, shape.top_k, out)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_out_close(got, ref, TOL_BF16)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), "bits differ from the plan path" 


def test_noalloc_declines_what_its_kernel_cannot_run():
    import torch
    lay, x = case("qwen3", 2, 1)
    shape = lay.shape
    dl = device_layer(lay)
    xt = x_tensor(shape, np.repeat(x, 9, axis=0))
    out = torch.empty((9, shape.D), dtype=torch.bfloat16, device="cuda")
    cfg = q.make_config(shape.E, shape.top_k, shape.D, shape.F, max_tokens=9)
    with pytest.raises(q.MoeError) as ei:  # more than 8 tokens
        q.moe_decode_forward_noalloc(cfg, xt, dl.router_w, dl.router_bias, dl.c_planes, 9, shape.top_k, out)
    assert ei.value.status == q.MOE_ERR_UNSUPPORTED


def test_noalloc_with_a_layer_variant_and_an_expert_range():
    """The allocation-free entry point takes the same variant fields."""
    import torch
    lay, x = case("qwen3", 2, 3)
    shape = lay.shape
    dl = device_layer(lay)
    xt = x_tensor(shape, x)
    ref_plan = make_plan(shape, activation=q.MOE_ACT_GEGLU, experts=(0, 64))  # plan path
    ref = ref_plan.forward(xt, dl).clone()
    torch.cuda.synchronize()
    cfg = q.make_config(shape.E, shape.top_k, shape.D, shape.F, max_tokens=3,
                        activation=q.MOE_ACT_GEGLU, expert_begin=0, expert_end=64)
    out = torch.empty_like(ref)
    q.moe_decode_forward_noalloc(cfg, xt, dl.router_w, dl.router_bias, dl.c_planes, 3, shape.top_k, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
