// activation.cuh -- the gated activation h = act(g, u) of the expert MLP.
//
// Kinds (MOE_ACT_*): SwiGLU silu(g) u; GeGLU gelu(g) u with the exact GELU
// g/2 (1 + erf(g / sqrt 2)); GeGLU with GELU's tanh form
// g/2 (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))); and the clamped SwiGLU
// silu(min(g, L)) min(max(u, -L), L).
// Sources: mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against
// 3.25x on dense", Implementation Notes (the fused kernel's GeGLU variant, used
// by gemma4, needs the same treatment or a decline), and issue #1859 "perf(moe):
// attribute the MoE decode gap at the M = 1 expert gather", Problem /
// Background (deepseek_v4's limited SwiGLU has a clamp stage). The pages give
// no formulas or bounds; these are the plainest readings, with the bound L a
// plan parameter.
#pragma once

#include "moe_decode.h"

namespace moe {

// PRECISE: expf and an IEEE division (the f32 check path); otherwise the fast
// exponential and division (the tensor-core paths, held to the bf16 tolerance)
template <bool PRECISE>
__device__ __forceinline__ float glu_act(int act, float limit, float g, float u) {
    if (act == MOE_ACT_GEGLU) return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
    if (act == MOE_ACT_GEGLU_TANH) {
        const float inner = 0.79788456080286536f * (g + 0.044715f * g * g * g);
        return 0.5f * g * (1.0f + tanhf(inner)) * u;
    }
    if (act == MOE_ACT_SWIGLU_CLAMPED) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    if (PRECISE) return g / (1.0f + expf(-g)) * u;
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

}  // namespace moe
