"""Checks that pin the CPU oracle to things other than itself.

Each check raises AssertionError on failure. They are run by
test_oracle_pins.py against the oracle as built, and by
test_oracle_mutants.py against copies of the oracle with a planted mistake
(each such copy must fail at least one check).

Independent references used here: the generator's original float weights
(quantiser round trip), hand-built planes with known codes, numpy matmul and
argsort, scipy softmax and expit in float64, a stable sort for grouping, the
closed-form example under tests/golden/, and invariants of the definition.
"""
from __future__ import annotations

import os

import numpy as np
from scipy import special

import moe_synth as ms
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# a small shape that still has several groups per row and several experts
SMALL = ms.LayerShape(E=16, top_k=4, D=256, F=128, act_dtype="f32", router_std=0.08)


def _rms(a):
    return float(np.sqrt(np.mean(np.square(a.astype(np.float64)))))


# ---------------------------------------------------------------------------
# dequantisation
# ---------------------------------------------------------------------------
def check_quant_roundtrip():
    """Dequantised codes stay within half a step of the original weights."""
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    w[3, 64:128] = 0.0125  # a constant group: s == 0
    q, s, b = ms.quantize_affine4(w)
    deq = oracle.dequant(q, s, b)
    g = w.reshape(8, 4, 64).astype(np.float64)
    lo, hi = g.min(-1), g.max(-1)
    sf = ms.bf16_to_f32(s).astype(np.float64)
    bf = ms.bf16_to_f32(b).astype(np.float64)
    bound = sf / 2 + np.abs(bf - lo) + 15 * np.abs(sf - (hi - lo) / 15) + 1e-7
    err = np.abs(deq.reshape(8, 4, 64) - g).max(-1)
    assert np.all(err <= bound), (err, bound)
    # the constant group dequantises to its (rounded) bias exactly
    assert np.all(deq[3, 64:128] == ms.bf16_to_f32(b)[3, 1])


def check_dequant_known_codes():
    """Hand-packed codes: input j of row r carries code (j + r) mod 16,
    scale 2^-(g+1) and bias g for group g. The value is known in closed form."""
    rows, cols = 4, 192
    codes = (np.arange(cols)[None, :] + np.arange(rows)[:, None]) % 16
    q = ms.pack_nibbles(codes.astype(np.uint32))
    groups = cols // 64
    s = np.zeros((rows, groups), np.float32)
    b = np.zeros((rows, groups), np.float32)
    for g in range(groups):
        s[:, g] = 2.0 ** -(g + 1)
        b[:, g] = float(g)
    deq = oracle.dequant(q, ms.bf16_bits(s), ms.bf16_bits(b))
    grp = np.arange(cols) // 64
    want = codes * (2.0 ** -(grp + 1))[None, :] + grp[None, :]
    assert np.array_equal(deq, want.astype(np.float32)), np.argwhere(deq != want)[:5]
    # all-zero codes with zero bias dequantise to exactly zero
    z = oracle.dequant(np.zeros((2, 8), np.uint32), ms.bf16_bits(np.ones((2, 1), np.float32)),
                       np.zeros((2, 1), np.uint16))
    assert np.all(z == 0.0)


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------
def _small_router_case(seed=5, n=6):
    w, _ = ms.draw_router(SMALL, seed, 0)
    x = ms.draw_tokens(SMALL, w, None, seed, 0, n)
    return x, w


def check_router_vs_library():
    x, w = _small_router_case()
    k = SMALL.top_k
    idx, tw, lg, pr = oracle.route(x, w, None, k)
    lg64 = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.allclose(lg, lg64, rtol=0, atol=1e-5)
    want_idx = np.argsort(-lg64, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, want_idx)
    sel = np.take_along_axis(lg64, want_idx, axis=1)
    want_w = special.softmax(sel, axis=1)  # softmax of the selected logits
    assert np.allclose(tw, want_w, rtol=0, atol=1e-6)
    assert np.allclose(pr, special.softmax(lg64, axis=1), rtol=0, atol=1e-6)
    assert np.allclose(tw.sum(1), 1.0, rtol=0, atol=1e-6)


def check_router_bias():
    w, _ = ms.draw_router(SMALL, 6, 0)
    bias = np.linspace(-2, 2, SMALL.E).astype(np.float32)
    x = ms.draw_tokens(SMALL, w, bias, 6, 0, 4)
    idx, tw, lg, _ = oracle.route(x, w, bias, SMALL.top_k)
    lg64 = x.astype(np.float64) @ w.astype(np.float64).T + bias[None, :]
    assert np.allclose(lg, lg64, atol=1e-5)
    assert np.array_equal(idx, np.argsort(-lg64, axis=1, kind="stable")[:, :SMALL.top_k])


def check_router_special_k():
    x, w = _small_router_case(seed=7, n=3)
    lg64 = x.astype(np.float64) @ w.astype(np.float64).T
    idx1, w1, _, _ = oracle.route(x, w, None, 1)   # k = 1: weight exactly 1
    assert np.all(w1 == 1.0)
    assert np.array_equal(idx1[:, 0], np.argmax(lg64, axis=1))
    E = SMALL.E                                        # k = E: the full softmax
    idxE, wE, _, _ = oracle.route(x, w, None, E)
    full = special.softmax(lg64, axis=1)
    got = np.zeros_like(full)
    np.put_along_axis(got, idxE.astype(np.int64), wE.astype(np.float64), axis=1)
    assert np.allclose(got, full, rtol=0, atol=1e-6)


def check_router_zero_input_ties():
    """x = 0: every logit ties; ties go to the lower index, weights are 1/k."""
    w, _ = ms.draw_router(SMALL, 8, 0)
    x = np.zeros((2, SMALL.D), np.float32)
    idx, tw, _, _ = oracle.route(x, w, None, 3)
    assert np.array_equal(idx, np.tile(np.arange(3), (2, 1)))
    assert np.allclose(tw, 1.0 / 3.0, rtol=0, atol=1e-7)


# ---------------------------------------------------------------------------
# grouping
# ---------------------------------------------------------------------------
def check_grouping_vs_sort():
    rng = np.random.default_rng(3)
    E, n, k = 12, 9, 3
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(n)]).astype(np.int32)
    g = oracle.group(idx, E)
    tok = np.repeat(np.arange(n), k)
    rank = np.tile(np.arange(k), n)
    ex = idx.reshape(-1)
    order = np.lexsort((tok, ex))  # by expert, then token
    assert np.array_equal(g["slot_token"], tok[order])
    assert np.array_equal(g["slot_k"], rank[order])
    assert np.array_equal(g["counts"], np.bincount(ex, minlength=E))
    assert np.array_equal(g["offsets"], np.concatenate([[0], np.cumsum(np.bincount(ex, minlength=E))]))
    assert np.array_equal(g["unique"], np.unique(ex))
    assert g["U"] == len(np.unique(ex))


# ---------------------------------------------------------------------------
# expert MLP and the whole step
# ---------------------------------------------------------------------------
def _dense_f64(planes, e):
    """One expert's dequantised matrices in float64 (through the pinned dequant)."""
    wg = oracle.dequant(planes.gate_q[e], planes.gate_s[e], planes.gate_b[e]).astype(np.float64)
    wu = oracle.dequant(planes.up_q[e], planes.up_s[e], planes.up_b[e]).astype(np.float64)
    wd = oracle.dequant(planes.down_q[e], planes.down_s[e], planes.down_b[e]).astype(np.float64)
    return wg, wu, wd


def _swiglu64(wg, wu, wd, x):
    g = x @ wg.T
    u = x @ wu.T
    return (g * special.expit(g) * u) @ wd.T


def check_single_expert_is_dense_swiglu():
    """E = 1, k = 1: the step is a textbook dense SwiGLU with weight 1."""
    shp = ms.LayerShape(E=1, top_k=1, D=256, F=192, act_dtype="f32", router_std=0.05)
    lay = ms.make_layer(shp, 21, 0)
    x = np.random.default_rng(21).standard_normal((3, shp.D)).astype(np.float32)
    r = oracle.moe_forward(x, lay.router_w, None, lay.planes, 1)
    assert np.all(r["topk_idx"] == 0) and np.all(r["topk_w"] == 1.0)
    want = _swiglu64(*_dense_f64(lay.planes, 0), x.astype(np.float64))
    assert np.abs(r["out"] - want).max() <= 1e-5 * _rms(want)
    # the per-expert routine agrees
    h, y = oracle.expert_mlp(x[1], lay.planes, 0)
    assert np.abs(y - want[1]).max() <= 1e-5 * _rms(want)


def check_brute_force_dense():
    """Every expert on every token, a dense gate matrix from a full sort and a
    softmax of the selected logits, summed over all experts (float64)."""
    lay = ms.make_layer(SMALL, 4, 0)
    x = ms.draw_tokens(SMALL, lay.router_w, None, 4, 0, 4)
    k = SMALL.top_k
    r = oracle.moe_forward(x, lay.router_w, None, lay.planes, k)
    x64 = x.astype(np.float64)
    lg = x64 @ lay.router_w.astype(np.float64).T
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    G = np.zeros((x.shape[0], SMALL.E))
    sel = np.take_along_axis(lg, order, axis=1)
    np.put_along_axis(G, order, special.softmax(sel, axis=1), axis=1)
    out = np.zeros((x.shape[0], SMALL.D))
    for e in range(SMALL.E):
        out += G[:, e:e + 1] * _swiglu64(*_dense_f64(lay.planes, e), x64)
    assert np.array_equal(r["topk_idx"], order)
    assert np.abs(r["out"] - out).max() <= 1e-5 * _rms(out), (np.abs(r["out"] - out).max(), _rms(out))


def check_closed_form_golden():
    """The worked example in tests/golden/closed_form_swiglu.txt."""
    spec = {}
    with open(os.path.join(GOLDEN, "closed_form_swiglu.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split("=", 1)
                spec[key.strip()] = float(val)
    D, F, E = int(spec["D"]), int(spec["F"]), 2

    def plane(rows, cols, code, scale):
        q = ms.pack_nibbles(np.full((rows, cols), code, np.uint32))
        s = ms.bf16_bits(np.full((rows, cols // 64), scale, np.float32))
        b = np.zeros((rows, cols // 64), np.uint16)
        return q, s, b

    per_expert = {
        # expert 0: gate codes 0 -> g = 0 -> h = 0 -> y = 0
        0: [plane(F, D, 0, 1.0 / D), plane(F, D, 2, 1.0 / D), plane(D, F, 1, 0.5 / F)],
        # expert 1: g = 1, u = 2, h = 2*sigmoid(1), y = h/2 = sigmoid(1)
        1: [plane(F, D, 1, 1.0 / D), plane(F, D, 2, 1.0 / D), plane(D, F, 1, 0.5 / F)],
    }
    arrays = {}
    for mi, m in enumerate(("gate", "up", "down")):
        for ci, c in enumerate(("q", "s", "b")):
            arrays[f"{m}_{c}"] = np.stack([per_expert[e][mi][ci] for e in range(E)])
    planes = ms.ExpertPlanes(**arrays)
    router = np.zeros((E, D), np.float32)
    router[1, :] = 1.0 / D  # logits: expert 0 -> 0, expert 1 -> sum(x)/D = 1
    x = np.ones((1, D), np.float32)
    r1 = oracle.moe_forward(x, router, None, planes, 1)
    assert r1["topk_idx"][0, 0] == 1 and r1["topk_w"][0, 0] == 1.0
    # f32 arithmetic: a 64-term sum of equal terms plus expf; 1e-6 is ~16 ulp
    assert np.allclose(r1["out"], spec["out_k1"], rtol=1e-6, atol=0)
    r2 = oracle.moe_forward(x, router, None, planes, 2)
    assert list(r2["topk_idx"][0]) == [1, 0]
    assert np.allclose(r2["topk_w"][0], [spec["w0_k2"], spec["w1_k2"]], rtol=1e-6, atol=0)
    assert np.allclose(r2["out"], spec["out_k2"], rtol=2e-6, atol=0)


# ---------------------------------------------------------------------------
# invariants of the definition
# ---------------------------------------------------------------------------
def check_invariants():
    lay = ms.make_layer(SMALL, 9, 0)
    x = ms.draw_tokens(SMALL, lay.router_w, None, 9, 0, 5)
    k = SMALL.top_k
    base = oracle.moe_forward(x, lay.router_w, None, lay.planes, k, want_bf16=True)
    assert np.allclose(base["topk_w"].sum(1), 1.0, atol=1e-6)

    # expert storage order: permute planes and router rows
    perm = np.random.default_rng(1).permutation(SMALL.E)
    inv = np.argsort(perm)
    pp = ms.ExpertPlanes(*[a[perm] for a in lay.planes.arrays()])
    rp = oracle.moe_forward(x, lay.router_w[perm], None, pp, k)
    # the softmax denominator is summed over experts in storage order, so the
    # weights (and out) move by f32 rounding only; the selection is exact
    assert np.abs(rp["out"] - base["out"]).max() <= 1e-6 * _rms(base["out"])
    assert np.allclose(rp["topk_w"], base["topk_w"], rtol=0, atol=1e-7)
    assert np.array_equal(perm[rp["topk_idx"]], base["topk_idx"])
    assert np.array_equal(inv[base["topk_idx"]], rp["topk_idx"])

    # token order: a row permutation of x permutes the output rows
    tp = np.array([3, 0, 4, 1, 2])
    rt = oracle.moe_forward(x[tp], lay.router_w, None, lay.planes, k)
    assert np.array_equal(rt["out"], base["out"][tp])

    # identical tokens give identical rows
    xi = np.repeat(x[2:3], 4, axis=0)
    ri = oracle.moe_forward(xi, lay.router_w, None, lay.planes, k)
    assert all(np.array_equal(ri["out"][t], ri["out"][0]) for t in range(4))
    assert np.array_equal(ri["out"][0], base["out"][2])
    assert ri["U"] == k and list(ri["counts"][ri["unique"]]) == [4] * k

    # x = 0 gives exactly zero output
    r0 = oracle.moe_forward(np.zeros((2, SMALL.D), np.float32), lay.router_w, None, lay.planes, k)
    assert np.all(r0["out"] == 0.0)
    assert np.array_equal(r0["topk_idx"], np.tile(np.arange(k), (2, 1)))

    # the single final rounding is round-to-nearest-even of the f32 result
    assert np.array_equal(base["out_bf16"], ms.bf16_bits(base["out"]))


def check_expert_shards_sum_to_the_step():
    """Expert-parallel split, done with virtual shards on the CPU: shard g keeps the
    planes of its experts and zeroes the scales and biases of all others. All
    weights of a zeroed expert are then 0, so its SwiGLU output is exactly 0 while
    routing is unchanged. The shards' f32 outputs must sum to the unsharded output
    (up to f32 rounding of the two summation orders), for 2 and 3 shards."""
    lay = ms.make_layer(SMALL, 13, 0)
    x = ms.draw_tokens(SMALL, lay.router_w, None, 13, 0, 6)
    k = SMALL.top_k
    full = oracle.moe_forward(x, lay.router_w, None, lay.planes, k)
    owner = np.random.default_rng(4).permutation(SMALL.E)
    for G in (2, 3):
        total = np.zeros_like(full["out"], dtype=np.float64)
        for g in range(G):
            mine = np.zeros(SMALL.E, bool)
            mine[owner[g::G]] = True
            arrs = []
            for name, a in zip(ms.ExpertPlanes.FIELDS, lay.planes.arrays()):
                a = a.copy()
                if not name.endswith("_q"):
                    a[~mine] = 0  # bf16 +0
                arrs.append(a)
            part = oracle.moe_forward(x, lay.router_w, None, ms.ExpertPlanes(*arrs), k)
            assert np.array_equal(part["topk_idx"], full["topk_idx"])
            total += part["out"]
        assert np.abs(total - full["out"]).max() <= 1e-6 * _rms(full["out"]), G


def _bf16_by_definition(u: int) -> int:
    """bf16 bits of the f32 with bits u, rounded to nearest with ties to an even
    last mantissa bit (IEEE 754 roundTiesToEven), taken from the definition: the
    two bf16 values that bracket the input are compared by exact rational
    distance. A magnitude that rounds past the largest finite bf16 goes to
    infinity, as if the exponent range were unbounded (IEEE overflow rule)."""
    from fractions import Fraction

    def value(bits32):
        sign = -1 if bits32 >> 31 else 1
        exp = (bits32 >> 23) & 0xFF
        man = bits32 & 0x7FFFFF
        if exp == 0:
            return sign * Fraction(man, 1 << 149)
        return sign * Fraction((1 << 23) | man, 1 << 23) * Fraction(2) ** (exp - 127)

    sign = u & 0x80000000
    mag = u & 0x7FFFFFFF
    if mag >= 0x7F800000:
        return (u >> 16) & 0xFFFF  # infinities pass through (NaN is checked apart)
    lo = mag & 0xFFFF0000          # the bf16 at or below |v|
    hi = lo + 0x10000              # the next bf16 up (0x7F800000 is infinity)
    v = value(mag)
    d_lo = v - value(lo)
    d_hi = (Fraction(2) ** 128 if hi == 0x7F800000 else value(hi)) - v
    if d_lo < d_hi:
        pick = lo
    elif d_hi < d_lo:
        pick = hi
    else:
        pick = lo if ((lo >> 16) & 1) == 0 else hi
    return ((sign | pick) >> 16) & 0xFFFF


def check_final_rounding_vs_library():
    """The single final rounding (f32 -> bf16, round to nearest even) against two
    references that do not share the oracle's bit formula: PyTorch's CPU
    float32 -> bfloat16 conversion, and the definition above on exact rational
    distances. Cases: exact ties with an even and with an odd lower neighbour,
    one ulp either side of a tie, carries into the exponent, +-0, subnormals,
    the largest finite values (overflow to infinity), infinities, NaN, and
    random bit patterns."""
    import torch
    rng = np.random.default_rng(23)
    special_u = [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x00008000, 0x00018000,
                 0x00007FFF, 0x00008001, 0x007FFFFF, 0x807FFFFF, 0x00800000, 0x3F7FFFFF,
                 0x3FFFFFFF, 0xBFFFFFFF, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001,
                 0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0x7F7E8000, 0x7F800000,
                 0xFF800000, 0x7FC00000, 0x7F800001, 0xFFFFFFFF, 0x7F7F0000]
    ties = [(int(b) << 16) | 0x8000 for b in rng.integers(0, 0x7F7F, 64)]
    near = [t + d for t in ties[:16] for d in (-1, 1)]
    rand = [int(v) for v in rng.integers(0, 1 << 32, 4096, dtype=np.uint64)]
    normals = [int(v) for v in (rng.standard_normal(2048).astype(np.float32) *
                                np.float32(3.0)).view(np.uint32)]
    u = np.array(special_u + ties + near + rand + normals, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    got = oracle.round_bf16(f)
    lib_bits = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    got_nan = (got & 0x7F80) == 0x7F80
    got_nan &= (got & 0x7F) != 0
    assert np.array_equal(got_nan, nan), "NaN inputs must give NaN, and only they"
    assert np.array_equal(got[~nan], lib_bits[~nan]), "final rounding differs from torch's bf16 cast"
    by_def = np.array([_bf16_by_definition(int(v)) for v in u[~nan]], dtype=np.uint16)
    assert np.array_equal(got[~nan], by_def), "final rounding differs from round-to-nearest-even"


# ---------------------------------------------------------------------------
# layer variants: GeGLU, clamped SwiGLU, 6-bit down planes
# ---------------------------------------------------------------------------
def _act64(kind, g, u, limit):
    """The activations in float64 from library routines (scipy erf and expit,
    numpy tanh and clip)."""
    if kind == oracle.ACT_GEGLU:
        return 0.5 * g * (1.0 + special.erf(g / np.sqrt(2.0))) * u
    if kind == oracle.ACT_GEGLU_TANH:
        return 0.5 * g * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (g + 0.044715 * g ** 3))) * u
    if kind == oracle.ACT_SWIGLU_CLAMPED:
        gc = np.minimum(g, limit)
        return gc * special.expit(gc) * np.clip(u, -limit, limit)
    return g * special.expit(g) * u


def check_activation_variants_vs_library():
    """Each activation kind of the oracle's expert MLP against a float64 dense
    formulation from library routines, on one expert; for the clamp, a limit
    below the largest |gate| and |up| so that both bounds act. Then the whole
    step with GeGLU against the brute-force dense gate formulation, and the
    clamp with a limit above every |gate| and |up| equal to SwiGLU bit for bit."""
    shp = ms.LayerShape(E=1, top_k=1, D=256, F=192, act_dtype="f32", router_std=0.05,
                        expert_std=0.08)
    lay = ms.make_layer(shp, 31, 0)
    x = np.random.default_rng(31).standard_normal((2, shp.D)).astype(np.float32)
    wg, wu, wd = _dense_f64(lay.planes, 0)
    for t in range(2):
        x64 = x[t].astype(np.float64)
        g, u = wg @ x64, wu @ x64
        limit = float(np.quantile(np.abs(np.concatenate([g, u])), 0.6))
        assert (g > limit).any() and (g < -limit).any() and (np.abs(u) > limit).any()
        for kind in (oracle.ACT_SWIGLU, oracle.ACT_GEGLU, oracle.ACT_GEGLU_TANH,
                     oracle.ACT_SWIGLU_CLAMPED):
            h, y = oracle.expert_mlp(x[t], lay.planes, 0, activation=kind, limit=limit)
            h64 = _act64(kind, g, u, limit)
            y64 = wd @ h64
            assert np.abs(h - h64).max() <= 1e-5 * _rms(h64), kind
            assert np.abs(y - y64).max() <= 1e-5 * _rms(y64), kind

    lay = ms.make_layer(SMALL, 4, 0)
    xs = ms.draw_tokens(SMALL, lay.router_w, None, 4, 0, 4)
    k = SMALL.top_k
    r = oracle.moe_forward(xs, lay.router_w, None, lay.planes, k, activation=oracle.ACT_GEGLU)
    x64 = xs.astype(np.float64)
    lg = x64 @ lay.router_w.astype(np.float64).T
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    G = np.zeros((xs.shape[0], SMALL.E))
    np.put_along_axis(G, order, special.softmax(np.take_along_axis(lg, order, axis=1), axis=1), axis=1)
    out = np.zeros((xs.shape[0], SMALL.D))
    for e in range(SMALL.E):
        wg, wu, wd = _dense_f64(lay.planes, e)
        out += G[:, e:e + 1] * (_act64(oracle.ACT_GEGLU, x64 @ wg.T, x64 @ wu.T, 0.0) @ wd.T)
    assert np.abs(r["out"] - out).max() <= 1e-5 * _rms(out)

    base = oracle.moe_forward(xs, lay.router_w, None, lay.planes, k)
    wide = oracle.moe_forward(xs, lay.router_w, None, lay.planes, k,
                              activation=oracle.ACT_SWIGLU_CLAMPED, limit=1e30)
    assert np.array_equal(wide["out"], base["out"])


def _pack6_by_int(codes):
    """6-bit codes of one row packed through a Python integer: code j shifted
    to bit 6j, written out as little-endian bytes."""
    v = 0
    for j, c in enumerate(codes):
        v |= int(c) << (6 * j)
    return np.frombuffer(v.to_bytes(3 * len(codes) // 4, "little"), dtype=np.uint8)


def check_dequant6_known_codes():
    """A 6-bit row with known codes, packed through a Python integer (not the
    generator's packer), dequantises to s*q + b exactly; the generator's packer
    gives the same bytes."""
    cols = 256
    rows = 3
    codes = np.array([[(7 * j + 3 * r + 1) % 64 for j in range(cols)] for r in range(rows)], np.uint32)
    q = np.stack([_pack6_by_int(codes[r]) for r in range(rows)])
    assert np.array_equal(q, ms.pack_6bit(codes))
    s = np.array([[0.5, 0.25, 2.0, 1.0]] * rows, np.float32)
    b = np.array([[-3.0, 1.0, -0.5, 0.0]] * rows, np.float32)
    got = oracle.dequant6(q, ms.bf16_bits(s), ms.bf16_bits(b))
    want = np.repeat(s, 64, axis=1) * codes.astype(np.float32) + np.repeat(b, 64, axis=1)
    assert np.array_equal(got, want)


def check_quant6_roundtrip():
    """6-bit codes dequantise to within half a step of the original weights."""
    rng = np.random.default_rng(12)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    q, sb, bb = ms.quantize_affine6(w)
    deq = oracle.dequant6(q, sb, bb).astype(np.float64)
    step = np.repeat(ms.bf16_to_f32(sb).astype(np.float64), 64, axis=1)
    bias = np.repeat(ms.bf16_to_f32(bb).astype(np.float64), 64, axis=1)
    # half a step, plus the rounding of the bias to bf16 (2^-8 relative)
    assert np.all(np.abs(deq - w) <= 0.5 * step + np.abs(bias) * 2.0 ** -8 + 1e-9)
    assert np.abs(deq - w).max() < np.abs(w).max() / 40


def check_down6_layer_vs_dense():
    """A layer with 4-bit gate/up and 6-bit down planes: the whole step against
    the brute-force dense formulation (every expert, dense gate from a full
    sort, float64), the 6-bit planes dequantised through the pinned routine."""
    shp = ms.SHAPES["dots"]
    lay = ms.make_layer(shp, 7, 0)
    x = ms.draw_tokens(shp, lay.router_w, None, 7, 0, 3)
    k = shp.top_k
    r = oracle.moe_forward(x, lay.router_w, None, lay.planes, k, down_bits=6)
    x64 = x.astype(np.float64)
    lg = x64 @ lay.router_w.astype(np.float64).T
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    G = np.zeros((x.shape[0], shp.E))
    np.put_along_axis(G, order, special.softmax(np.take_along_axis(lg, order, axis=1), axis=1), axis=1)
    out = np.zeros((x.shape[0], shp.D))
    p = lay.planes
    for e in range(shp.E):
        wg = oracle.dequant(p.gate_q[e], p.gate_s[e], p.gate_b[e]).astype(np.float64)
        wu = oracle.dequant(p.up_q[e], p.up_s[e], p.up_b[e]).astype(np.float64)
        wd = oracle.dequant6(p.down_q[e], p.down_s[e], p.down_b[e]).astype(np.float64)
        out += G[:, e:e + 1] * _swiglu64(wg, wu, wd, x64)
    assert np.array_equal(r["topk_idx"], order)
    assert np.abs(r["out"] - out).max() <= 1e-5 * _rms(out)


ALL_CHECKS = [
    check_quant_roundtrip,
    check_dequant_known_codes,
    check_router_vs_library,
    check_router_bias,
    check_router_special_k,
    check_router_zero_input_ties,
    check_grouping_vs_sort,
    check_single_expert_is_dense_swiglu,
    check_brute_force_dense,
    check_closed_form_golden,
    check_invariants,
    check_expert_shards_sum_to_the_step,
    check_final_rounding_vs_library,
    check_activation_variants_vs_library,
    check_dequant6_known_codes,
    check_quant6_roundtrip,
    check_down6_layer_vs_dense,
]
