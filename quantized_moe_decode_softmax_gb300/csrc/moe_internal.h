// moe_internal.h -- plan, workspace layout and kernel launchers shared by the
// translation units of the CUDA library. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_decode.h"

namespace moe {

constexpr int kGroup = 64;
constexpr int kMaxTokens = 64;         // decode cohorts (single launch, chunks, grouped path)
constexpr int kMaxPrefillTokens = 8192; // larger cohorts: the prefill path (grouped GEMM)
constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 16;
constexpr int kMaxDff = 8192;
constexpr int kMaxD = 16384;
constexpr int kMaxSlots = kMaxTokens * kMaxTopK;
constexpr int kTagSlots = 256;  // tagged logits per token (the single launch: E <= 256)
// largest cohort that runs as chunks of the single-launch kernel by default
// (larger ones take the grouped multi-kernel path)
constexpr int kChunkMaxTokens = 16;

// status word bits written by device code (ws.status[0])
enum : unsigned {
    kDevErrTimeout = 1u << 0,   // a bounded spin-wait gave up
    kDevErrInternal = 1u << 1,  // an impossible index was seen and skipped
    kDevErrRange = 1u << 2,     // an f16 operand saturated (|h| > 65504)
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
    unsigned *status;   // [4]   [0] device error bits; [2..3] device address of the
                        //       plan's host-mapped error word (0: none)
    unsigned *sync;     // [64]  [0..1] grid-barrier counter; [32] the single launch's
                        //       last launch tag (zeroed at plan creation)
    unsigned long long *tlog;  // [max_n, kTagSlots] logits of the single launch,
                               // each (launch tag << 32 | f32 bits)
    unsigned long long *phase_ns;  // [256] optional phase timestamps
    unsigned *tbits;    // prefill grouping: [E][W] token bitmaps, W = ceil(max_n / 32)
    int *wbase;         // prefill grouping: [E][W] exclusive scan of the words' popcounts
    void *x_stage;      // [max_n, D] host-call staging for x
    void *out_stage;    // [max_n, D] host-call staging for out
};

struct Shape {
    int E, k, D, F, n;
    int x_dtype, w_dtype, out_dtype;
    unsigned flags;  // MOE_FLAG_* of the plan
    int act;         // MOE_ACT_*
    float act_limit; // clamp bound of MOE_ACT_SWIGLU_CLAMPED
    int down_bits;   // 4 or 6
    int e_lo, e_hi;  // owned experts [e_lo, e_hi)
};

// the Shape of a plan's config for a cohort of n tokens
inline Shape shape_of(const moe_config &c, int n, unsigned flags) {
    Shape s{c.E, c.top_k, c.D, c.Dff, n, c.x_dtype, c.router_dtype, c.out_dtype, flags,
            c.activation, c.act_limit, c.down_bits == 6 ? 6 : 4, 0, c.E};
    if (c.expert_begin != 0 || c.expert_end != 0) {
        s.e_lo = c.expert_begin;
        s.e_hi = c.expert_end;
    }
    return s;
}

// Arguments of one step, device pointers.
struct StepArgs {
    Shape s;
    const void *x;
    const void *router_w;
    const float *router_bias;
    moe_expert_planes planes;
    void *out;
    // the next layer's router (rows and bias) to prefetch into L2 during this
    // step, or null (moe_decode_forward_layers)
    const void *next_router_w;
    const float *next_router_bias;
};

// Shared-memory and work layout of the single-launch decode step (host-computed).
struct DecodeLayout {
    int G;            // CTAs (one per SM)
    int NS;           // ring stages
    int stage_bytes;  // bytes per ring stage (multiple of 1024)
    // gate/up stages: one 16-row tile of gate and up rows x KS K-slices of 256 inputs
    int KS;           // K-slices per gate/up stage
    int NKC;          // gate/up stages per tile (K chunks)
    int GDc;          // groups (64 inputs) per K chunk = 4 * KS
    int off_up;       // byte offset of the up box inside a gate/up stage
    int off_sc;       // byte offset of the four scale/bias boxes (1024 bytes apart)
    int sc_w;         // bytes per row of a gate/up scale box (2 * GDc)
    int sc_m;         // swizzle mask of the gate/up scale boxes
    // down stages: P units, a unit = one expert x one D-tile (<= 15 rows) x all Dff
    int kw_d;         // u32 words per down K-slice row (min(32, Dff/8))
    int sl_d;         // down K-slices
    int swz_d;        // swizzle mask of the down box (7: 128-byte rows, 3: 64-byte rows)
    int Hd[2];        // down D-tile heights that occur (even; tensor map per height)
    int dmode;        // down scale copies: 0 bulk rows as stored, 1 TMA row-pair boxes
    int rb_d;         // bytes per row of down scales (Dff/32)
    int sc_md;        // swizzle mask of the down scale boxes (mode 1)
    int unit_w;       // bytes of a unit's weight box area (multiple of 1024)
    int unit_sc;      // offset of a unit's scale block; its bias block follows at +unit_sc_stride
    int unit_sc_stride;
    int unit_bytes;   // bytes per unit (weights + scale/bias block, multiple of 1024)
    int P;            // units per down stage
    int max_tiles;    // gate/up tiles a CTA may own (bound of the tile list)
    // shared memory carve (byte offsets from the 1024-aligned base)
    int off_bar, off_misc, off_route, off_tiles, off_x, off_xsum, off_red, off_ring;
    int x_stride;     // bytes per staged token row of x
    int smem_bytes;   // dynamic shared memory requested (includes alignment slack)
};

// TMA descriptors of one forward call's expert planes (kernel parameters).
struct TMaps {
    CUtensorMap gq, uq;          // gate/up codes: 3-D {32 words, E*Dff rows, D/256 slices}
    CUtensorMap gs, gb, us, ub;  // gate/up scales, biases: 3-D {D/64, E*Dff/2 row pairs, 2}
    CUtensorMap dq[2];           // down codes per D-tile height: {kw_d, E*D rows, sl_d}
    CUtensorMap ds[2], db[2];    // down scales, biases per height (scale mode 1)
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
    unsigned long long forwards;  // moe_decode_forward calls that launched
    // pinned, device-mapped word set by the device on a timeout or internal
    // error (null if the driver could not map host memory)
    volatile unsigned *host_err;
    bool fused_ok;                // the single-launch kernel can run this shape
    moe::DecodeLayout fused;
    // tensor maps of recently used plane sets (a layer stack or replicas cycle
    // through several), replaced round robin
    struct TmEntry {
        moe::TMaps tmaps;             // first: 64-byte aligned members
        moe_expert_planes planes;     // the planes these maps describe
        bool valid;
    };
    static constexpr int kTmCache = 64;
    TmEntry tm_cache[kTmCache];
    int tm_next;
};

namespace moe {

// routing (route_kernels.cu)
// Each launcher adds the number of kernels it enqueued to `launched`.
cudaError_t launch_router_logits(const StepArgs &a, const Workspace &ws, cudaStream_t st,
                                 int &launched);
// refine: the logits came from the tensor-core router; the weights are taken
// from the k selected logits recomputed with the CUDA-core router's sum
cudaError_t launch_topk_group(const StepArgs &a, const Workspace &ws, cudaStream_t st,
                              int &launched, bool refine = false);
// routing and grouping of a prefill cohort (more than kMaxTokens tokens) from
// the logits: top-k per token, per-expert token bitmaps, counts, offsets, slots
cudaError_t launch_prefill_route(const StepArgs &a, const Workspace &ws, int max_n, cudaStream_t st,
                                 int &launched, bool refine = false);

// exact f32 expert path (expert_f32_kernels.cu)

// single-launch path (decode_step.cu)
bool fused_layout(const moe_config &c, int num_sms, int max_smem, DecodeLayout *out);
cudaError_t fused_prepare(const DecodeLayout &L, int *blocks_per_sm);
int fused_max_tokens();
// encode the tensor maps of `planes`; false if the driver rejects them
bool fused_encode_tmaps(const moe_config &c, const DecodeLayout &L, const moe_expert_planes &planes,
                        TMaps *out);
cudaError_t launch_fused(const StepArgs &a, const Workspace &ws, const DecodeLayout &L,
                         const TMaps &tm, cudaStream_t st, int &launched);

}  // namespace moe
