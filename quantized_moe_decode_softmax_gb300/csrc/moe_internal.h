// moe_internal.h -- plan, workspace layout and kernel launchers shared by the
// translation units of the CUDA library. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_decode.h"

namespace moe {

constexpr int kGroup = 64;
constexpr int kMaxTokens = 64;
constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 16;
constexpr int kMaxDff = 8192;
constexpr int kMaxD = 16384;
constexpr int kMaxSlots = kMaxTokens * kMaxTopK;

// status word bits written by device code (ws.status[0])
enum : unsigned {
    kDevErrTimeout = 1u << 0,   // a bounded spin-wait gave up
    kDevErrInternal = 1u << 1,  // an impossible index was seen and skipped
};

// Device workspace of one plan (one cudaMalloc, carved in this order).
struct Workspace {
    float *logits;      // [max_n, E]
    int *topk_idx;      // [max_n, k]
    float *topk_w;      // [max_n, k]
    int *counts;        // [E]
    int *offsets;       // [E + 1]
    int *slot_token;    // [max_n * k]  grouped order
    int *slot_k;        // [max_n * k]  grouped order
    int *slot_of;       // [max_n * k]  (t*k + j) -> grouped position
    int *unique;        // [E]
    int *U;             // [1]
    float *h;           // [max_n * k, Dff]  grouped position major
    float *y;           // [max_n * k, D]    grouped position major
    unsigned *status;   // [4]   device error bits
    unsigned *sync;     // [64]  barrier counters (zeroed at plan creation)
    unsigned long long *phase_ns;  // [256] optional phase timestamps
    void *x_stage;      // [max_n, D] host-call staging for x
    void *out_stage;    // [max_n, D] host-call staging for out
};

struct Shape {
    int E, k, D, F, n;
    int x_dtype, w_dtype, out_dtype;
    unsigned flags;  // MOE_FLAG_* of the plan
};

// Arguments of one step, device pointers.
struct StepArgs {
    Shape s;
    const void *x;
    const void *router_w;
    const float *router_bias;
    moe_expert_planes planes;
    void *out;
};

// Shared-memory and work layout of the fused kernel (computed on the host).
struct FusedLayout {
    int G;            // CTAs (one per SM)
    int NS;           // ring slots
    int slot_bytes;   // bytes per ring slot
    int nksA;         // gate/up K-slices (8 groups each) per 16-row tile
    int nksB;         // down K-slices (4 groups each) per 16-row tile
    int SA;           // gate/up row stride in a slot (bytes, padded)
    int SB;           // down row stride in a slot (bytes, padded)
    int hoff;         // offset of the h block area inside a down slot
    int x_tokens;     // tokens the staged-activation area holds
    int x_stride;     // bytes per token row of the staged activations
    int part_bytes;   // gate/up partial-sum buffers (also the final reduction)
    int off_bar, off_route, off_tiles, off_x, off_xsum, off_part, off_sbuf, off_ring;
    int smem_bytes;
};

}  // namespace moe

struct moe_plan {
    moe_config cfg;
    int device;
    int num_sms;
    size_t ws_bytes;
    void *ws_base;
    moe::Workspace ws;
    cudaStream_t last_stream;
    int last_n;
    int mma_min_tokens;
    unsigned long long launches;  // kernels enqueued by this plan since creation
    bool fused_ok;                // the fused kernel can run this shape
    moe::FusedLayout fused;
};

namespace moe {

// routing (route_kernels.cu)
// Each launcher adds the number of kernels it enqueued to `launched`.
cudaError_t launch_router_logits(const StepArgs &a, const Workspace &ws, cudaStream_t st,
                                 int &launched);
cudaError_t launch_topk_group(const StepArgs &a, const Workspace &ws, cudaStream_t st,
                              int &launched);

// exact f32 expert path (expert_f32_kernels.cu)
cudaError_t launch_experts_f32(const StepArgs &a, const Workspace &ws, cudaStream_t st,
                               int &launched);

// fused single-launch path (fused_step.cu)
bool fused_layout(const moe_config &c, int num_sms, int max_smem, FusedLayout *out);
cudaError_t fused_prepare(const FusedLayout &L, int *blocks_per_sm);
int fused_max_tokens();
cudaError_t launch_fused(const StepArgs &a, const Workspace &ws, const FusedLayout &L,
                         cudaStream_t st, int &launched);

}  // namespace moe
