// prefill_tc.h -- entry points of the tcgen05 expert GEMMs (prefill_tc.cu) and
// of the expert launcher of the grouped and prefill paths.
#pragma once

#include "moe_internal.h"

namespace moe {

// the tcgen05 GEMMs need D and Dff to be multiples of 128 (weight rows per block)
bool tc_variant_supported(const Shape &s);
// gate/up (down = false: h = act(gate, up)) or down (y) for the experts with at
// least `thr` tokens: per block one expert, 128 weight rows, 64 tokens at a time
cudaError_t launch_expert_tc(const StepArgs &a, const Workspace &ws, int thr, bool down, cudaStream_t st,
                             int &launched);
// router logits on the tensor cores (bf16 x and router rows, f32 accumulation):
// logits[t, e] = x[t] . Wr[e] (+ bias[e]) for the grouped and prefill paths
bool router_tc_supported(const Shape &s);
cudaError_t launch_router_tc(const StepArgs &a, const Workspace &ws, cudaStream_t st, int &launched);

// the per-expert MLPs and the combine of the grouped and prefill paths: experts
// with at least mma_thr tokens (mma_thr > 0, shape supported) on the tcgen05
// GEMMs, the others on the f32 GEMV kernels (expert_f32_kernels.cu)
cudaError_t launch_experts(const StepArgs &a, const Workspace &ws, int mma_thr, cudaStream_t st,
                           int &launched);

}  // namespace moe
