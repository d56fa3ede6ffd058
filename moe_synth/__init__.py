"""Seeded synthetic inputs for one quantized MoE decode layer.

This module is the only code shared by the CUDA path, the oracle and the
benchmark. It draws weights and tokens, rounds them to bf16, and packs
expert weights into the affine 4-bit, group-64 format (MLX layout).
It holds none of the decode step's arithmetic: no dequantisation, no
routing, no expert MLP, no combine.

Two pieces of input conditioning need a value derived from the inputs:

* The quantiser (the inverse of the format) picks a per-group scale and
  bias from the group's min and max.
* The routing-margin rule redraws a token until the gaps among its
  top-(k+1) router logits are at least 1e-2. It computes those logits in
  float64 with numpy's matmul, from the stored (rounded) values. This is
  the condition a workload must meet, checked before either side runs.

Every array comes from a numpy PCG64 stream keyed by
(seed, layer, role, index). An expert's planes therefore do not depend on
which other experts are materialised.

Format (MLX-style affine quantisation, 4 bits, group 64):
  plane q  : uint32 [E, out, in/8]; nibble j (bits 4j..4j+3) of word i holds
             the code of input index 8*i + j (lowest input in the low nibble)
  scale s  : bf16 bits (uint16) [E, out, in/64]
  bias  b  : bf16 bits (uint16) [E, out, in/64]
  the weight a code stands for is s*q + b.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

GROUP = 64
BITS = 4
MARGIN = 1e-2

# role tags for the seeded streams
_ROUTER, _EXPERT, _TOKENS, _BIAS = 0, 1, 2, 3


# ----------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ----------------------------------------------------------------------------
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16, round-to-nearest-even; return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# configurations
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class LayerShape:
    E: int          # experts
    top_k: int
    D: int          # hidden size (input of gate/up, output of down)
    F: int          # expert intermediate size (Dff)
    act_dtype: str  # "f32" or "bf16": dtype of x, router weights and out
    router_std: float
    expert_std: float = 0.02
    zipf_s: float = 0.0  # >0: add a Zipf log-prior router bias
    down_bits: int = 4   # 4: down codes as uint32 words; 6: a byte stream of 6-bit codes

    @property
    def plane_bytes(self) -> int:
        """HBM bytes of one expert's three planes with scales and biases."""
        sb = 4 * self.D * self.F // GROUP
        return 2 * (self.D * self.F // 2 + sb) + self.D * self.F * self.down_bits // 8 + sb


TINY = LayerShape(E=8, top_k=2, D=256, F=128, act_dtype="f32", router_std=0.05)
QWEN3 = LayerShape(E=128, top_k=8, D=2048, F=768, act_dtype="bf16", router_std=0.02)
E256 = LayerShape(E=256, top_k=6, D=4096, F=2048, act_dtype="bf16",
                  router_std=1.0 / 64.0, zipf_s=1.1)

# edge shapes for parity tests: the largest top-k (16) on the single-launch
# path, the largest expert count (1024, multi-kernel path), top-k equal to the
# expert count, and top-1 with f32 activations. Router deviations put the
# logits' standard deviation near 1-2 so the margin rule is met quickly.
K16 = LayerShape(E=64, top_k=16, D=512, F=256, act_dtype="bf16", router_std=2.0 / 512 ** 0.5)
E1024 = LayerShape(E=1024, top_k=16, D=256, F=128, act_dtype="bf16", router_std=2.0 / 256 ** 0.5)
KALL = LayerShape(E=8, top_k=8, D=512, F=256, act_dtype="bf16", router_std=1.0 / 512 ** 0.5)
K1 = LayerShape(E=16, top_k=1, D=512, F=256, act_dtype="f32", router_std=1.0 / 512 ** 0.5)
# mixed widths: 4-bit gate/up with 6-bit down (a small layer, and the
# 128-expert top-8 shape with 6-bit down)
DOTS = LayerShape(E=16, top_k=4, D=512, F=256, act_dtype="bf16", router_std=1.0 / 512 ** 0.5,
                  down_bits=6)
QWEN3_D6 = LayerShape(E=128, top_k=8, D=2048, F=768, act_dtype="bf16", router_std=0.02, down_bits=6)
# Dff a multiple of 64 but not of 128: outside the single launch's and the
# tensor-core GEMMs' shape rules (every expert on the f32 GEMV)
F192 = LayerShape(E=16, top_k=4, D=512, F=192, act_dtype="bf16", router_std=1.0 / 512 ** 0.5)

SHAPES: Dict[str, LayerShape] = {"tiny": TINY, "qwen3": QWEN3, "e256": E256, "k16": K16,
                                 "e1024": E1024, "kall": KALL, "k1": K1, "dots": DOTS,
                                 "qwen3_d6": QWEN3_D6, "f192": F192}

# named workloads: shape, seed, cohort sizes and cohort kinds
WORKLOADS = {
    "tiny": dict(shape="tiny", seed=0, n=[1]),
    "qwen3_n1": dict(shape="qwen3", seed=1, n=[1]),
    "qwen3_ladder": dict(shape="qwen3", seed=2, n=[2, 4, 8]),
    "e256": dict(shape="e256", seed=3, n=[1, 4, 16]),
    "stack48": dict(shape="qwen3", seed=100, n=[1, 2, 4, 8, 16, 32, 64], layers=48),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


# ----------------------------------------------------------------------------
# quantiser (input generation)
# ----------------------------------------------------------------------------
def quantize_affine4(w: np.ndarray):
    """Quantise float32 w [rows, cols] to 4-bit codes, group 64 along cols.

    Per group: lo = min, hi = max, s = bf16((hi - lo) / 15), b = bf16(lo),
    q = clamp(rint((w - b) / s), 0, 15) computed with the rounded s and b
    (q = 0 where s == 0). Returns (q_packed uint32 [rows, cols/8],
    s_bits uint16 [rows, cols/64], b_bits uint16 [rows, cols/64]).
    """
    q, s_bits, b_bits = _quantize_codes(w, 15)
    return pack_nibbles(q), s_bits, b_bits


def quantize_affine6(w: np.ndarray):
    """The same affine rule with 6-bit codes (63 steps per group). Returns
    (q_packed uint8 [rows, 3*cols/4], s_bits, b_bits); see pack_6bit."""
    q, s_bits, b_bits = _quantize_codes(w, 63)
    return pack_6bit(q), s_bits, b_bits


def _quantize_codes(w: np.ndarray, qmax: int):
    rows, cols = w.shape
    assert cols % GROUP == 0
    g = w.reshape(rows, cols // GROUP, GROUP).astype(np.float32)
    lo = g.min(axis=2)
    hi = g.max(axis=2)
    s_bits = bf16_bits((hi - lo) / np.float32(qmax))
    b_bits = bf16_bits(lo)
    s = bf16_to_f32(s_bits)[..., None]
    b = bf16_to_f32(b_bits)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint((g - b) / np.where(s == 0, np.float32(1.0), s))
    qf = np.where(s == 0, 0.0, qf)
    q = np.clip(qf, 0, qmax).astype(np.uint32).reshape(rows, cols)
    return q, s_bits, b_bits


def pack_6bit(q: np.ndarray) -> np.ndarray:
    """Pack 6-bit codes [rows, cols] as one little-endian bit stream per row:
    code j occupies bits 6j..6j+5, so four codes fill three bytes. Returns
    uint8 [rows, 3*cols/4]."""
    rows, cols = q.shape
    q4 = q.reshape(rows, cols // 4, 4).astype(np.uint32)
    v = q4[..., 0] | (q4[..., 1] << 6) | (q4[..., 2] << 12) | (q4[..., 3] << 18)
    out = np.stack([v & 0xFF, (v >> 8) & 0xFF, (v >> 16) & 0xFF], axis=-1).astype(np.uint8)
    return out.reshape(rows, 3 * cols // 4)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Pack codes [rows, cols] (0..15) as uint32 [rows, cols/8], low nibble first."""
    rows, cols = q.shape
    q8 = q.reshape(rows, cols // 8, 8).astype(np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    return np.bitwise_or.reduce(q8 << shifts, axis=2).astype(np.uint32)


def unpack_nibbles(p: np.ndarray) -> np.ndarray:
    """Inverse of pack_nibbles: uint32 [rows, words] -> uint8 codes [rows, 8*words]."""
    rows, words = p.shape
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    return ((p[:, :, None] >> shifts) & 0xF).astype(np.uint8).reshape(rows, words * 8)


# ----------------------------------------------------------------------------
# layer weights
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class ExpertPlanes:
    """Quantised planes of E experts (numpy, host)."""
    gate_q: np.ndarray   # uint32 [E, F, D/8]
    gate_s: np.ndarray   # uint16 [E, F, D/64]
    gate_b: np.ndarray
    up_q: np.ndarray     # uint32 [E, F, D/8]
    up_s: np.ndarray
    up_b: np.ndarray
    down_q: np.ndarray   # uint32 [E, D, F/8] (4-bit), or uint8 [E, D, 3F/4] (6-bit)
    down_s: np.ndarray   # uint16 [E, D, F/64]
    down_b: np.ndarray

    FIELDS = ("gate_q", "gate_s", "gate_b", "up_q", "up_s", "up_b",
              "down_q", "down_s", "down_b")

    def arrays(self):
        return [getattr(self, f) for f in self.FIELDS]


@dataclasses.dataclass
class Layer:
    shape: LayerShape
    seed: int
    layer: int
    router_w: np.ndarray           # f32 values [E, D] (bf16-representable for bf16 shapes)
    router_bias: Optional[np.ndarray]  # f32 [E] or None
    planes: ExpertPlanes
    materialised: np.ndarray       # bool [E]: experts whose planes were drawn


def draw_expert_weights(shape: LayerShape, seed: int, layer: int, e: int):
    """Unquantised float32 weights of expert e: (gate [F,D], up [F,D], down [D,F])."""
    r = _rng(seed, layer, _EXPERT, e)
    std = np.float32(shape.expert_std)
    gate = r.standard_normal((shape.F, shape.D), dtype=np.float32) * std
    up = r.standard_normal((shape.F, shape.D), dtype=np.float32) * std
    down = r.standard_normal((shape.D, shape.F), dtype=np.float32) * std
    return gate, up, down


def draw_router(shape: LayerShape, seed: int, layer: int):
    r = _rng(seed, layer, _ROUTER)
    w = r.standard_normal((shape.E, shape.D), dtype=np.float32) * np.float32(shape.router_std)
    if shape.act_dtype == "bf16":
        w = bf16_to_f32(bf16_bits(w))
    bias = None
    if shape.zipf_s > 0:
        rb = _rng(seed, layer, _BIAS)
        ranks = rb.permutation(shape.E) + 1
        bias = (-shape.zipf_s * np.log(ranks.astype(np.float64))).astype(np.float32)
    return w, bias


def expert_planes(shape: LayerShape, seed: int, layer: int, e: int):
    """The nine quantised arrays of expert e (gate q/s/b, up q/s/b, down q/s/b)."""
    gate, up, down = draw_expert_weights(shape, seed, layer, e)
    qd = quantize_affine6 if shape.down_bits == 6 else quantize_affine4
    return (*quantize_affine4(gate), *quantize_affine4(up), *qd(down))


def _expert_planes_job(args):
    return args[3], expert_planes(*args)


def make_layer(shape: LayerShape, seed: int, layer: int = 0,
               experts: Optional[Sequence[int]] = None, workers: int = 1) -> Layer:
    """Draw a layer. If `experts` is given, only those experts' planes are drawn
    and the others are left zero (their bytes are never read by a decode step
    that does not route to them). workers > 1 draws experts in a process pool
    started with the 'spawn' method (safe after CUDA has been initialised)."""
    router_w, router_bias = draw_router(shape, seed, layer)
    E, D, F = shape.E, shape.D, shape.F
    planes = ExpertPlanes(
        gate_q=np.zeros((E, F, D // 8), np.uint32),
        gate_s=np.zeros((E, F, D // GROUP), np.uint16),
        gate_b=np.zeros((E, F, D // GROUP), np.uint16),
        up_q=np.zeros((E, F, D // 8), np.uint32),
        up_s=np.zeros((E, F, D // GROUP), np.uint16),
        up_b=np.zeros((E, F, D // GROUP), np.uint16),
        down_q=(np.zeros((E, D, 3 * F // 4), np.uint8) if shape.down_bits == 6
                else np.zeros((E, D, F // 8), np.uint32)),
        down_s=np.zeros((E, D, F // GROUP), np.uint16),
        down_b=np.zeros((E, D, F // GROUP), np.uint16),
    )
    mat = np.zeros(E, bool)
    todo = list(range(E)) if experts is None else sorted(set(int(e) for e in experts))
    jobs = [(shape, seed, layer, e) for e in todo]
    if workers > 1 and len(jobs) > 1:
        import concurrent.futures as cf
        import multiprocessing as mp
        with cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
            results = ex.map(_expert_planes_job, jobs, chunksize=max(1, len(jobs) // (4 * workers)))
            for e, arrs in results:
                for f, a in zip(ExpertPlanes.FIELDS, arrs):
                    getattr(planes, f)[e] = a
                mat[e] = True
    else:
        for job in jobs:
            e, arrs = _expert_planes_job(job)
            for f, a in zip(ExpertPlanes.FIELDS, arrs):
                getattr(planes, f)[e] = a
            mat[e] = True
    return Layer(shape, seed, layer, router_w, router_bias, planes, mat)


# ----------------------------------------------------------------------------
# tokens and the routing-margin rule
# ----------------------------------------------------------------------------
def router_logits_f64(x: np.ndarray, router_w: np.ndarray, bias) -> np.ndarray:
    """Router logits in float64 from stored values, for the margin rule only."""
    lg = x.astype(np.float64) @ router_w.astype(np.float64).T
    if bias is not None:
        lg = lg + bias.astype(np.float64)[None, :]
    return lg


def margin_ok(logits_row: np.ndarray, k: int, margin: float = MARGIN) -> bool:
    """All adjacent gaps among the top-(k+1) sorted logits are >= margin."""
    srt = np.sort(logits_row)[::-1]
    m = min(k + 1, srt.size)
    return bool(np.all(srt[: m - 1] - srt[1:m] >= margin))


def topk_set_f64(logits_row: np.ndarray, k: int) -> List[int]:
    return [int(i) for i in np.argsort(-logits_row, kind="stable")[:k]]


def _act_round(shape: LayerShape, x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32)
    if shape.act_dtype == "bf16":
        x = bf16_to_f32(bf16_bits(x))
    return x


def draw_tokens(shape: LayerShape, router_w, bias, seed: int, layer: int, n: int,
                kind: str = "independent", cohort: int = 0, max_tries: int = 10000):
    """Draw a cohort x [n, D] (float32 values, bf16-representable for bf16 shapes).

    kind:
      independent - x_t ~ N(0,1) per token, redrawn until the margin rule holds
      shared      - x_t = x_0 + 0.1*N(0,1), redrawn until token t selects the
                    same top-k set as token 0 (all tokens route to k experts)
      disjoint    - x_t = 4*sum_{e in S_t} Wr[e]/|Wr[e]| + N(0,1) over disjoint
                    random sets S_t, redrawn until top-k(t) == S_t
    """
    r = _rng(seed, layer, _TOKENS, cohort, {"independent": 0, "shared": 1, "disjoint": 2}[kind])
    D, k = shape.D, shape.top_k
    xs = np.zeros((n, D), np.float32)

    def draw_ok(make, want=None):
        for _ in range(max_tries):
            x = _act_round(shape, make())
            lg = router_logits_f64(x[None, :], router_w, bias)[0]
            if not margin_ok(lg, k):
                continue
            if want is not None and set(topk_set_f64(lg, k)) != set(want):
                continue
            return x
        raise RuntimeError(f"could not draw a token meeting the routing rule ({kind})")

    if kind == "independent":
        for t in range(n):
            xs[t] = draw_ok(lambda: r.standard_normal(D, dtype=np.float32))
    elif kind == "shared":
        xs[0] = draw_ok(lambda: r.standard_normal(D, dtype=np.float32))
        want = topk_set_f64(router_logits_f64(xs[:1], router_w, bias)[0], k)
        for t in range(1, n):
            xs[t] = draw_ok(lambda: xs[0] + np.float32(0.1) * r.standard_normal(D, dtype=np.float32), want)
    elif kind == "disjoint":
        if n * k > shape.E:
            raise ValueError("disjoint cohort needs n*k <= E")
        perm = r.permutation(shape.E)
        wn = router_w / np.linalg.norm(router_w, axis=1, keepdims=True)
        for t in range(n):
            S = [int(e) for e in perm[t * k:(t + 1) * k]]
            base = np.float32(4.0) * wn[S].sum(axis=0).astype(np.float32)
            xs[t] = draw_ok(lambda: base + r.standard_normal(D, dtype=np.float32), S)
    else:
        raise ValueError(kind)
    return xs


def routed_experts(x, router_w, bias, k) -> List[int]:
    """Experts the cohort selects (by the float64 logits of the margin rule)."""
    lg = router_logits_f64(x, router_w, bias)
    sel = set()
    for t in range(x.shape[0]):
        sel.update(topk_set_f64(lg[t], k))
    return sorted(sel)


def make_case(shape_name: str, seed: int, n: int, kind: str = "independent",
              layer: int = 0, cohort: int = 0, lazy: bool = False, workers: int = 1):
    """A layer and a cohort. lazy=True draws only the experts the cohort routes to."""
    shape = SHAPES[shape_name]
    router_w, bias = draw_router(shape, seed, layer)
    x = draw_tokens(shape, router_w, bias, seed, layer, n, kind, cohort)
    experts = routed_experts(x, router_w, bias, shape.top_k) if lazy else None
    lay = make_layer(shape, seed, layer, experts, workers=workers)
    return lay, x


def x_storage(shape: LayerShape, x: np.ndarray) -> np.ndarray:
    """x in its storage dtype: float32, or bf16 bits (uint16)."""
    return x.astype(np.float32) if shape.act_dtype == "f32" else bf16_bits(x)


def router_storage(shape: LayerShape, w: np.ndarray) -> np.ndarray:
    return w.astype(np.float32) if shape.act_dtype == "f32" else bf16_bits(w)
