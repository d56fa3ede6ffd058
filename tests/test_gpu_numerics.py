"""Numerics of the tensor-core paths beyond the bf16 tolerance (GPU).

1. Cohort order. A row permutation of x permutes the output rows bit for bit,
   on the single launch and the grouped path (tcgen05 and GEMV variants): every
   token's result is computed independently of its position. On the chunks of
   the single launch (9..16 tokens) this holds for permutations inside each
   chunk; across chunks the rows agree within the bf16 tolerance.

2. A derived error model for the single-launch kernel with f32 output. The
   kernel rounds what the oracle keeps in f32:
     - h' = w * act(g, u) is stored as f16 (round to nearest even): an absolute
       error uniform in +-ulp(h')/2, variance ulp(h')^2 / 12;
     - the down projection accumulates (1024 + q) h' per group of 64 inputs in
       f32 (four k16 steps) and subtracts the MMA row that holds 1024 sum(h'):
       at most eight roundings at the magnitude M = 1024 sum_group |h'|, each
       of variance at most (2^-23 M)^2 / 12, scaled by the group's scale s;
     - gate/up do the same with 1024 + q against x / m: taken as a relative
       error of 2^-13 on h';
     - x enters the MMA as f16: exact for bf16 x inside f16's range, a relative
       error of at most 2^-11 for f32 x (taken as that relative error on h').
   Each output element is out[t, d] = sum_j sum_f Wd_j[d, f] h'_jf, so its error
   is a sum of independent terms with variance
     var[t, d] = sum_j ( sum_f Wd_j[d, f]^2 (ulp(h'_jf)^2 / 12 + (c h'_jf)^2)
                       + sum_g s_j[d, g]^2 (2/3) 2^-26 (sum_{f in g} |h'_jf|)^2 ),
   c^2 = 2^-26 (+ 2^-22 / 3 for f32 x). The test requires every element within
   6 standard deviations (one element of a few ten thousand exceeds 6 sigma
   with probability below 1e-4 under the model), with an absolute floor of
   1e-6 RMS(out).

3. f16 range. Activations far below or beyond f16's range take a per-token
   power-of-two scale on the single launch and still match the oracle; an
   intermediate h beyond f16's range is reported as MOE_ERR_RANGE (single
   launch and the tcgen05 GEMMs), and the f32 check path computes the same layer.
"""
import numpy as np
import pytest

import moe_synth as ms
import oracle
from gpu_cases import (TOL_BF16, assert_out_close, case, device_layer, make_plan, path_name,
                       record_margin, rms, run_gpu, run_oracle, x_tensor)

pytestmark = pytest.mark.gpu

GROUPED = 1 << 3  # MOE_FLAG_GROUPED_COHORTS


@pytest.mark.parametrize("shape_name,n,kind,flags,mma_min", [
    ("qwen3", 8, "independent", 0, 0),        # single launch
    ("qwen3", 12, "independent", 0, 0),       # two chunks of the single launch
    ("qwen3", 24, "independent", 0, 0),       # grouped: GEMV variant
    ("qwen3", 24, "shared", GROUPED, 0),      # grouped: tile variant (24 tokens per expert)
    ("tiny", 5, "independent", 0, 0),         # grouped (shape the single launch declines)
])
def test_row_permutation_permutes_output_rows_bitwise(shape_name, n, kind, flags, mma_min):
    import torch
    lay, x = case(shape_name, 2 if shape_name == "qwen3" else 0, n, kind,
                  full=shape_name == "tiny")
    shape = lay.shape
    dl = device_layer(lay)
    plan = make_plan(shape, flags=flags, mma_min_tokens=mma_min)
    xt = x_tensor(shape, x)
    a = plan.forward(xt, dl).clone()
    bits = torch.int16 if a.dtype == torch.bfloat16 else torch.int32
    rng = np.random.default_rng(n)
    chunked = shape_name == "qwen3" and 9 <= n <= 16 and not flags
    if chunked:
        # Chunks of the single launch: a token's result depends, at the rounding
        # level, on which experts share its chunk (the down projection's sum
        # order over a chunk's expert set). A permutation inside each chunk
        # keeps every chunk's token set and must permute rows bit for bit; a
        # permutation across chunks stays within the bf16 tolerance.
        half = n // 2  # two chunks of n/2 tokens (n even here)
        inside = np.concatenate([rng.permutation(half), half + rng.permutation(n - half)])
        b = plan.forward(x_tensor(shape, x[inside]), dl).clone()
        across = rng.permutation(n)
        c = plan.forward(x_tensor(shape, x[across]), dl).clone()
        torch.cuda.synchronize()
        plan.check()
        assert torch.equal(b.view(bits).cpu(), a.view(bits).cpu()[torch.from_numpy(inside)])
        assert_out_close(c.float().cpu().numpy(), a.float().cpu().numpy()[across], TOL_BF16)
        return
    perm = rng.permutation(n)
    b = plan.forward(x_tensor(shape, x[perm]), dl).clone()
    torch.cuda.synchronize()
    plan.check()
    assert torch.equal(b.view(bits).cpu(), a.view(bits).cpu()[torch.from_numpy(perm)])


def _error_sigma(lay, x, ref):
    """Per-element standard deviation of the single-launch kernel's f32 output
    error under the model in the module docstring."""
    shape = lay.shape
    n, D = x.shape
    c2 = 2.0 ** -26 + (2.0 ** -22 / 3.0 if shape.act_dtype == "f32" else 0.0)
    var = np.zeros((n, D), np.float64)
    deq = {}
    for t in range(n):
        for j in range(shape.top_k):
            e = int(ref["topk_idx"][t, j])
            if e not in deq:
                p = lay.planes
                deq[e] = (oracle.dequant(p.down_q[e], p.down_s[e], p.down_b[e]).astype(np.float64),
                          ms.bf16_to_f32(p.down_s[e]).astype(np.float64))
            h, _ = oracle.expert_mlp(x[t], lay.planes, e)
            hp = float(ref["topk_w"][t, j]) * h.astype(np.float64)
            _, ex = np.frexp(hp)  # |hp| in [2^(ex-1), 2^ex)
            ulp = np.where(hp != 0.0, np.ldexp(1.0, np.maximum(ex - 1, -14) - 10), 0.0)  # f16
            per_f = ulp ** 2 / 12.0 + c2 * hp ** 2
            var[t] += np.square(deq[e][0]) @ per_f
            hg = np.abs(hp).reshape(-1, 64).sum(axis=1)          # sum |h'| per group
            var[t] += np.square(deq[e][1]) @ (hg ** 2) * (2.0 / 3.0) * 2.0 ** -26
    return np.sqrt(var)


@pytest.mark.parametrize("shape_name,seed,n,kind", [
    ("qwen3", 2, 1, "independent"),
    ("qwen3", 2, 4, "independent"),
    ("qwen3", 2, 8, "shared"),
    ("k1", 5, 5, "independent"),   # f32 activations on the single launch
    ("e256", 3, 1, "independent"),
])
def test_single_launch_f32_output_within_the_derived_error_model(shape_name, seed, n, kind):
    lay, x = case(shape_name, seed, n, kind, full=shape_name == "k1")
    shape = lay.shape
    ref = run_oracle(lay, x)
    plan = make_plan(shape, out_dtype="f32")
    launches = []
    out, _ = run_gpu(plan, device_layer(lay), shape, x, launches)
    assert launches[0] == 1, "this case must run on the single launch"
    sigma = _error_sigma(lay, x, ref)
    r = rms(ref["out"])
    err = np.abs(out.astype(np.float64) - ref["out"].astype(np.float64))
    z = err / np.maximum(sigma, 1e-6 * r)
    record_margin(f"model z max {z.max():.2f} (bound 6)", shape_name, n, kind,
                  path_name(n, launches[0]), "f32", TOL_BF16, float(err.max()) / r)
    assert z.max() <= 6.0, f"max |err| / sigma = {z.max():.2f}"
    assert_out_close(out, ref["out"], TOL_BF16)


def _range_layer():
    """A small layer whose expert weights are tiny (std 1e-6), so that very
    large activations still give gate, up and h values of order one."""
    shape = ms.LayerShape(E=16, top_k=2, D=512, F=256, act_dtype="bf16",
                          router_std=1.0 / 512 ** 0.5, expert_std=1e-6)
    lay = ms.make_layer(shape, 61, 0)
    x = ms.draw_tokens(shape, lay.router_w, None, 61, 0, 3)
    return shape, lay, x


@pytest.mark.parametrize("scale_exp", [17, -14])
def test_single_launch_scales_tokens_outside_f16_range(scale_exp):
    """x times 2^17 (beyond f16's largest value) or 2^-14 (where most values
    would be f16 subnormals): the single launch scales each token by a power of
    two and matches the oracle as for ordinary activations."""
    shape, lay, x = _range_layer()
    if scale_exp < 0:  # ordinary weights: the output is then small but not tiny
        shape = ms.LayerShape(E=16, top_k=2, D=512, F=256, act_dtype="bf16",
                              router_std=1.0 / 512 ** 0.5)
        lay = ms.make_layer(shape, 62, 0)
        x = ms.draw_tokens(shape, lay.router_w, None, 62, 0, 3)
    xs = np.ldexp(x, scale_exp).astype(np.float32)  # exact: bf16 values times 2^k
    # the router scaled the other way keeps the logits (and their margins)
    lay.router_w = np.ldexp(lay.router_w, -scale_exp).astype(np.float32)
    ref = run_oracle(lay, xs)
    plan = make_plan(shape)
    launches = []
    out, routing = run_gpu(plan, device_layer(lay), shape, xs, launches)
    assert launches[0] == 1, "this case must run on the single launch"
    assert np.array_equal(routing["topk_idx"], ref["topk_idx"])
    err_rel = assert_out_close(out, ref["out"], TOL_BF16)
    record_margin(f"x scaled by 2^{scale_exp}", "range", 3, "independent", "single launch", None,
                  TOL_BF16, err_rel)


def test_h_beyond_f16_range_is_reported():
    """Activations of order 2^12 on the 128-expert layer make h of order 10^6:
    the single launch reports MOE_ERR_RANGE (on moe_plan_check and on the next
    forward call), the tcgen05 GEMMs too, and the f32 check path computes the
    step."""
    import torch
    import quantized_moe_decode_softmax_gb300 as q
    lay, x = case("qwen3", 2, 2)
    shape = lay.shape
    xs = np.ldexp(x, 12).astype(np.float32)
    dl = device_layer(lay)
    plan = make_plan(shape)
    plan.forward(x_tensor(shape, xs), dl)
    with pytest.raises(q.MoeError) as ei:
        plan.check()
    assert ei.value.status == q.MOE_ERR_RANGE
    plan.forward(x_tensor(shape, xs), dl)
    torch.cuda.synchronize()
    with pytest.raises(q.MoeError) as ei:  # reported by the next forward call
        plan.forward(x_tensor(shape, xs), dl)
    assert ei.value.status == q.MOE_ERR_RANGE
    # the same plan, ordinary activations: correct again
    ref = run_oracle(lay, x)
    out, _ = run_gpu(plan, dl, shape, x)
    assert_out_close(out, ref["out"], TOL_BF16)
    # grouped path (every expert on the tcgen05 GEMMs)
    tplan = make_plan(shape, flags=q.MOE_FLAG_GROUPED_COHORTS, mma_min_tokens=1)
    lay16, x16 = case("qwen3", 2, 16)
    dl16 = device_layer(lay16)
    tplan.forward(x_tensor(shape, np.ldexp(x16, 12).astype(np.float32)), dl16)
    with pytest.raises(q.MoeError) as ei:
        tplan.check()
    assert ei.value.status == q.MOE_ERR_RANGE
    # the f32 check path computes the large activations
    fplan = make_plan(shape, flags=q.MOE_FLAG_F32_DEBUG, out_dtype="f32")
    ref = run_oracle(lay, xs)
    out, _ = run_gpu(fplan, dl, shape, xs)
    assert_out_close(out, ref["out"], 1e-4)
