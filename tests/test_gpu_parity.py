"""GPU path (through the C ABI) against the CPU oracle, element by element.

Routing and grouping must match bit for bit (inputs are drawn with top-k
logit margins of at least 1e-2). Outputs must be within 2e-2 * RMS(out) on
the default path and within 1e-4 * RMS(out) on the f32 check path.
"""
import numpy as np
import pytest

import moe_synth as ms
from gpu_cases import (TOL_BF16, TOL_F32, assert_out_close, assert_routing_equal, case,
                       device_layer, make_plan, path_name, record_margin, run_gpu, run_oracle,
                       x_tensor)

pytestmark = pytest.mark.gpu

F32_DEBUG = 1
GROUPED = 1 << 3  # MOE_FLAG_GROUPED_COHORTS


def _check(shape_name, seed, n, kind="independent", full=False, flags=0, out_dtype=None,
           tol=None, mma_min_tokens=0, max_tokens=64):
    import os
    lay, x = case(shape_name, seed, n, kind, full=full)
    shape = lay.shape
    ref = run_oracle(lay, x)
    plan = make_plan(shape, flags=flags, out_dtype=out_dtype, mma_min_tokens=mma_min_tokens,
                     max_tokens=max_tokens)
    launches = []
    out, routing = run_gpu(plan, device_layer(lay), shape, x, launches)
    assert_routing_equal(routing, ref)
    if tol is None:
        tol = TOL_F32 if flags & F32_DEBUG else TOL_BF16
    err = float(np.abs(out.astype(np.float64) - ref["out"].astype(np.float64)).max())
    err_rel = err / max(float(np.sqrt(np.mean(np.square(ref["out"].astype(np.float64))))), 1e-30)
    path = path_name(n, launches[0], flags)
    if mma_min_tokens:
        path += f", tensor-core threshold {mma_min_tokens}"
    record_margin(os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], shape_name, n, kind,
                  path, out_dtype, tol, err_rel)
    return assert_out_close(out, ref["out"], tol)


# ---- tiny layer (E=8, top-2, D=256, Dff=128, f32 activations) -------------------
@pytest.mark.parametrize("flags", [0, F32_DEBUG])
def test_tiny(flags):
    _check("tiny", 0, 1, full=True, flags=flags)


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_tiny_cohorts(n):
    _check("tiny", 0, n, full=True, flags=F32_DEBUG)
    _check("tiny", 0, n, full=True)


# ---- 128-expert top-8 layer (D=2048, Dff=768) -------------------------------------
def test_qwen3_n1_full_layer():
    _check("qwen3", 1, 1, full=True)


def test_qwen3_n1_f32_check_path():
    _check("qwen3", 1, 1, full=True, flags=F32_DEBUG, out_dtype="f32")


@pytest.mark.parametrize("n", [2, 4, 8])
@pytest.mark.parametrize("kind", ["independent", "shared", "disjoint"])
def test_qwen3_ladder(n, kind):
    _check("qwen3", 2, n, kind)


@pytest.mark.parametrize("n", [9, 16, 17, 32, 64])
def test_qwen3_large_cohorts(n):
    # 9..16: chunks of the single-launch kernel; 17 and up: the grouped path
    _check("qwen3", 2, n)


@pytest.mark.parametrize("n,kind", [(12, "independent"), (24, "shared")])
def test_qwen3_grouped_path_below_the_chunk_limit(n, kind):
    _check("qwen3", 2, n, kind, flags=GROUPED)


def test_qwen3_shared_64_tokens_single_expert_set():
    # every token routes to the same 8 experts: per-expert count 64
    _check("qwen3", 2, 64, "shared")


@pytest.mark.parametrize("shape_name,seed,n,full", [("qwen3", 2, 16, False), ("e256", 3, 16, False),
                                                   ("tiny", 0, 12, True)])
def test_tensor_core_gemms_for_every_expert(shape_name, seed, n, full):
    # mma_min_tokens = 1 on the grouped path: every selected expert takes the
    # tcgen05 GEMMs (weights dequantised into tensor memory, its tokens in
    # blocks of 64)
    _check(shape_name, seed, n, full=full, flags=GROUPED, mma_min_tokens=1)


def test_tensor_core_gemms_with_mixed_counts():
    # threshold 3 on a 64-token cohort: experts with at least 3 tokens take the
    # tcgen05 GEMMs, the others the GEMV kernels, in the same step
    _check("qwen3", 2, 64, mma_min_tokens=3)


@pytest.mark.parametrize("n,kind", [(3, "independent"), (24, "independent"), (64, "shared"),
                                    (200, "independent")])
def test_shape_outside_the_tcgen05_rule_runs_on_the_gemv(n, kind):
    # Dff = 192 (a multiple of 64, not of 128): the single launch and the
    # tcgen05 GEMMs decline the shape, so every cohort takes the grouped (or
    # prefill) path with every expert on the f32 GEMV kernels
    _check("f192", 7, n, kind, full=True, tol=TOL_BF16, max_tokens=max(n, 64))


# ---- 256-expert top-6 layer (D=4096, Dff=2048, Zipf router bias) ------------------
@pytest.mark.parametrize("n", [1, 4, 16])
def test_e256(n):
    _check("e256", 3, n)


def test_e256_chunks_of_unequal_size():
    # 15 tokens run as chunks of 7 and 8 tokens
    _check("e256", 3, 15)


def test_e256_f32_check_path():
    _check("e256", 3, 4, flags=F32_DEBUG, out_dtype="f32")


# ---- edge shapes -------------------------------------------------------------------
@pytest.mark.parametrize("shape_name,n,flags", [
    ("k16", 1, 0),           # top-16 on the single launch
    ("k16", 8, 0),           # 128 slots, the single launch's maximum
    ("k16", 12, 0),          # chunks of 6 and 6
    ("k16", 12, GROUPED),
    ("kall", 3, 0),          # top-k = E: every expert selected, weights = softmax
    ("k1", 5, 0),            # top-1, f32 activations on the single launch
    ("e1024", 4, 0),         # 1024 experts (multi-kernel path), top-16
    ("e1024", 64, 0),        # 64 tokens x top-16 = 1024 slots, the largest cohort
])
def test_edge_shapes(shape_name, n, flags):
    _check(shape_name, 5, n, full=True, flags=flags)


def test_edge_shapes_f32_check_path():
    _check("k16", 5, 8, full=True, flags=F32_DEBUG, out_dtype="f32")
    _check("e1024", 5, 16, full=True, flags=F32_DEBUG, out_dtype="f32")


# ---- properties --------------------------------------------------------------------
def test_deterministic_and_identical_tokens():
    import torch
    lay, x = case("qwen3", 2, 4)
    x = np.repeat(x[1:2], 4, axis=0)  # four identical tokens
    shape = lay.shape
    lay = ms.make_layer(shape, 2, 0, ms.routed_experts(x, lay.router_w, None, shape.top_k))
    dl = device_layer(lay)
    plan = make_plan(shape)
    xt = x_tensor(shape, x)
    outs = []
    for _ in range(10):
        outs.append(plan.forward(xt, dl).clone())
    torch.cuda.synchronize()
    ref = outs[0].view(torch.int16)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), ref), "run-to-run bits differ"
    for t in range(1, 4):
        assert torch.equal(outs[0][t].view(torch.int16), outs[0][0].view(torch.int16))


def test_cohort_size_changes_between_calls():
    """One plan, n varying call to call (no re-specialisation per n)."""
    lay, x = case("qwen3", 2, 8)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape)
    for n in (3, 1, 8, 5):
        ref = run_oracle(lay, x[:n])
        out, routing = run_gpu(plan, dl, shape, x[:n])
        assert_routing_equal(routing, ref)
        assert_out_close(out, ref["out"], TOL_BF16)


def test_host_entry_point_matches_device_entry_point():
    import torch
    lay, x = case("qwen3", 2, 4)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape)
    xt = x_tensor(shape, x)
    dev = plan.forward(xt, dl)
    torch.cuda.synchronize()
    x_host = xt.cpu().pin_memory()
    out_host = torch.empty((4, shape.D), dtype=torch.bfloat16).pin_memory()
    plan.forward_host(x_host, dl, out_host)
    assert torch.equal(out_host.view(torch.int16), dev.cpu().view(torch.int16))


def test_host_entry_point_for_a_chunked_cohort():
    """12 tokens through the host entry point (chunks of the single launch):
    the same bits as the device entry point."""
    import torch
    lay, x = case("qwen3", 2, 12)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape)
    xt = x_tensor(shape, x)
    dev = plan.forward(xt, dl)
    torch.cuda.synchronize()
    out_host = torch.empty((12, shape.D), dtype=torch.bfloat16).pin_memory()
    plan.forward_host(xt.cpu().pin_memory(), dl, out_host)
    assert torch.equal(out_host.view(torch.int16), dev.cpu().view(torch.int16))


def test_zero_input():
    import torch
    lay, _ = case("qwen3", 2, 2)
    shape = lay.shape
    x = np.zeros((2, shape.D), np.float32)
    lay = ms.make_layer(shape, 2, 0, range(shape.top_k))
    ref = run_oracle(lay, x)
    plan = make_plan(shape)
    out, routing = run_gpu(plan, device_layer(lay), shape, x)
    assert np.array_equal(routing["topk_idx"], np.tile(np.arange(shape.top_k), (2, 1)))
    assert np.all(out == 0.0) and np.all(ref["out"] == 0.0)


def test_runtime_argument_errors_launch_nothing():
    import torch
    import quantized_moe_decode_softmax_gb300 as q
    lay, x = case("tiny", 0, 1, full=True)
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, max_tokens=4)
    xt = x_tensor(shape, np.zeros((8, shape.D), np.float32))
    out = torch.empty((8, shape.D), device="cuda")
    for n, k in ((0, 2), (5, 2), (1, 3)):
        with pytest.raises(q.MoeError) as ei:
            q.moe_decode_forward(plan.plan, xt, dl.router_w, None, dl.c_planes, n, k, out)
        assert ei.value.status == q.MOE_ERR_INVALID_ARG
    with pytest.raises(q.MoeError):
        q.moe_decode_forward(plan.plan, xt, dl.router_w, None, dl.c_planes, 1, 2, xt)  # out aliases x
    plan.check()
