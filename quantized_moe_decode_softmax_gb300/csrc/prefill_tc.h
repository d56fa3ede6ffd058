// prefill_tc.h -- entry points of the prefill path's tcgen05 expert GEMMs
// (prefill_tc.cu) and of the expert launcher that uses them.
#pragma once

#include "moe_internal.h"

namespace moe {

// the tcgen05 GEMMs need D and Dff to be multiples of 128 (weight rows per block)
bool tc_variant_supported(const Shape &s);
// gate/up (down = false: h = act(gate, up)) or down (y) for the experts with at
// least `thr` tokens: per block one expert, 128 weight rows, 64 tokens at a time
cudaError_t launch_expert_tc(const StepArgs &a, const Workspace &ws, int thr, bool down, cudaStream_t st,
                             int &launched);
// launch_experts_f32 with the tcgen05 GEMMs in place of the mma.sync tiles for
// the experts with at least tile_thr tokens (the prefill path)
cudaError_t launch_experts_prefill(const StepArgs &a, const Workspace &ws, int tile_thr, cudaStream_t st,
                                   int &launched);

}  // namespace moe
