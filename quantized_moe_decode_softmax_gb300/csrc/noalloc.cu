// noalloc.cu -- moe_decode_forward_noalloc: the single-launch decode step for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a CUDA graph
// that is being captured, allocator-free embedded runtimes, or a host process
// whose memory pool belongs to another framework. This entry point runs the
// same kernel as moe_decode_forward (cohorts of up to 8 tokens) with its
// scratch memory -- router logits, routing tables, the h rows exchanged between
// the gate/up and down phases, the grid-barrier counter and the status word --
// in one statically sized device array of this file. Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "moe_internal.h"

using namespace moe;

namespace {

// Maximum scratch of one call (bytes). Every GPU that loads this library holds
// the array until the process exits.
constexpr size_t kNoAllocScratchBytes = 4u << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Per-device set-up, done once by the first call on that device: the device
// address of the scratch array (the host-side symbol is only a handle).
struct DeviceState {
    bool ready = false;
    unsigned char *scratch = nullptr;
};
DeviceState g_state[kMaxDevices];
std::mutex g_state_mu;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Carve the fused path's workspace for n_tokens out of `base` (nullptr: size only).
size_t carve_noalloc(const moe_config &c, int n, unsigned char *base, Workspace *ws) {
    const size_t E = c.E, k = c.top_k, F = c.Dff, S = (size_t)n * k;
    size_t off = 0;
    auto take = [&](size_t bytes) -> unsigned char * {
        unsigned char *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    Workspace w{};
    w.status = (unsigned *)take(4 * 4);
    w.sync = (unsigned *)take(64 * 4);
    w.tlog = (unsigned long long *)take((size_t)n * kTagSlots * 8);
    w.logits = (float *)take((size_t)n * E * 4);
    w.topk_idx = (int *)take(S * 4);
    w.topk_w = (float *)take(S * 4);
    w.counts = (int *)take(E * 4);
    w.offsets = (int *)take((E + 1) * 4);
    w.slot_token = (int *)take(S * 4);
    w.slot_k = (int *)take(S * 4);
    w.slot_of = (int *)take(S * 4);
    w.unique = (int *)take(E * 4);
    w.U = (int *)take(4);
    w.h = (float *)take(S * F * 2);  // bf16 h rows of the fused path
    w.y = nullptr;
    w.phase_ns = (unsigned long long *)take(8);  // unused: phase timing is off here
    w.x_stage = nullptr;
    w.out_stage = nullptr;
    if (ws) *ws = w;
    return off;
}

}  // namespace

extern "C" moe_status moe_decode_forward_noalloc(const moe_config *cfg, const void *x, const void *router_w,
                                                 const float *router_bias, const moe_expert_planes *planes,
                                                 int n_tokens, int top_k, void *out, void *stream) {
    if (!cfg || !planes || !x || !router_w || !out) return MOE_ERR_INVALID_ARG;
    if (cfg->bits != 4 || cfg->group_size != kGroup) return MOE_ERR_UNSUPPORTED;
    if (cfg->E < 1 || cfg->top_k < 1 || cfg->top_k > cfg->E || cfg->D < 1 || cfg->Dff < 1)
        return MOE_ERR_INVALID_ARG;
    if (top_k != cfg->top_k || n_tokens < 1) return MOE_ERR_INVALID_ARG;
    for (int dt : {cfg->x_dtype, cfg->router_dtype, cfg->out_dtype})
        if (dt != MOE_DTYPE_F32 && dt != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (x == out) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)router_w | (uintptr_t)out) & 15u) return MOE_ERR_INVALID_ARG;
    if (router_bias && ((uintptr_t)router_bias & 3u)) return MOE_ERR_INVALID_ARG;
    const void *ptrs[9] = {planes->gate_q, planes->gate_s, planes->gate_b, planes->up_q, planes->up_s,
                           planes->up_b, planes->down_q, planes->down_s, planes->down_b};
    for (const void *p : ptrs)
        if (!p || ((uintptr_t)p & 15u)) return MOE_ERR_INVALID_ARG;
    // only the single-launch kernel runs here: up to 8 tokens, shapes it supports
    if (n_tokens > fused_max_tokens() || (cfg->flags & MOE_FLAG_F32_DEBUG)) return MOE_ERR_UNSUPPORTED;
    if (cfg->E > kMaxE || cfg->top_k > kMaxTopK || cfg->D > kMaxD || cfg->Dff > kMaxDff ||
        cfg->D % kGroup || cfg->Dff % kGroup)
        return MOE_ERR_UNSUPPORTED;
    // the layer variants: activations and the expert range as for a plan; the
    // single-launch kernel reads 4-bit down planes only
    if (cfg->activation < MOE_ACT_SWIGLU || cfg->activation > MOE_ACT_SWIGLU_CLAMPED) return MOE_ERR_UNSUPPORTED;
    if (cfg->activation == MOE_ACT_SWIGLU_CLAMPED && !(cfg->act_limit > 0.0f && cfg->act_limit <= 3.0e38f))
        return MOE_ERR_INVALID_ARG;
    if (cfg->down_bits == 6) return MOE_ERR_UNSUPPORTED;
    if (cfg->down_bits != 0 && cfg->down_bits != 4) return MOE_ERR_UNSUPPORTED;
    if ((cfg->expert_begin != 0 || cfg->expert_end != 0) &&
        (cfg->expert_begin < 0 || cfg->expert_begin >= cfg->expert_end || cfg->expert_end > cfg->E))
        return MOE_ERR_INVALID_ARG;
    // the scratch this call needs must fit the static array
    if (carve_noalloc(*cfg, n_tokens, nullptr, nullptr) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;

    int dev = 0, num_sms = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    moe_config c = *cfg;
    c.max_tokens = n_tokens;
    c.flags = 0;  // no phase timing, no trace, no test hooks on this path
    DecodeLayout L{};
    if (!fused_layout(c, num_sms, max_smem, &L)) return MOE_ERR_UNSUPPORTED;

    unsigned char *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_state_mu);
        DeviceState &ds = g_state[dev];
        if (!ds.ready) {
            // first call on this device (the current one): resolve the device
            // address of the scratch array
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
                cudaGetLastError();
                return MOE_ERR_CUDA;
            }
            ds.scratch = static_cast<unsigned char *>(p);
            ds.ready = true;
        }
        scratch = ds.scratch;
    }
    int per_sm = 0;
    if (fused_prepare(L, &per_sm) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        return MOE_ERR_UNSUPPORTED;
    }
    TMaps tm;
    if (!fused_encode_tmaps(c, L, *planes, &tm)) return MOE_ERR_UNSUPPORTED;

    Workspace ws{};
    carve_noalloc(c, n_tokens, scratch, &ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the status word, the grid-barrier counter, the launch tag and the tagged
    // logits start at zero on every call (the array keeps the previous call's
    // contents)
    if (cudaMemsetAsync(ws.status, 0, (unsigned char *)ws.logits - (unsigned char *)ws.status, st) !=
        cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    StepArgs a{};
    a.s = shape_of(c, n_tokens, 0u);
    a.x = x;
    a.router_w = router_w;
    a.router_bias = router_bias;
    a.planes = *planes;
    a.out = out;
    int launched = 0;
    if (launch_fused(a, ws, L, tm, st, launched) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
