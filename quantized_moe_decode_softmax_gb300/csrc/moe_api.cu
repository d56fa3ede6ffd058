// moe_api.cu -- the C ABI: plan creation and validation, workspace, dispatch.
//
// The shape checks and the decline rule follow mlxcel issue #1616
// "perf(moe): batched decode scales 1.55x against 3.25x on dense",
// Implementation Notes: unsupported configurations decline (here
// MOE_ERR_UNSUPPORTED) instead of failing, shapes are validated before any
// dispatch because a bad shape must never reach a kernel, n_tokens is a
// runtime extent and never a specialisation key.
#include <cuda_runtime.h>
#include <stdio.h>

#include <algorithm>
#include <stdlib.h>
#include <string.h>

#include "moe_internal.h"
#include "prefill_tc.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

size_t elem_size(int dtype) { return dtype == MOE_DTYPE_F32 ? 4 : 2; }

moe_status validate_config(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->bits != 4 || c->group_size != kGroup) return MOE_ERR_UNSUPPORTED;
    if (c->E < 1 || c->top_k < 1 || c->D < 1 || c->Dff < 1 || c->max_tokens < 1)
        return MOE_ERR_INVALID_ARG;
    if (c->top_k > c->E) return MOE_ERR_INVALID_ARG;
    if (c->max_tokens > kMaxPrefillTokens) return MOE_ERR_INVALID_ARG;
    for (int dt : {c->x_dtype, c->router_dtype, c->out_dtype})
        if (dt != MOE_DTYPE_F32 && dt != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->mma_min_tokens < 0) return MOE_ERR_INVALID_ARG;
    if (c->E > kMaxE || c->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (c->D % kGroup || c->Dff % kGroup) return MOE_ERR_UNSUPPORTED;
    if (c->flags & ~(unsigned)(MOE_FLAG_F32_DEBUG | MOE_FLAG_TRACE | MOE_FLAG_PHASE_TIMES |
                               MOE_FLAG_GROUPED_COHORTS | MOE_FLAG_TEST_STALL))
        return MOE_ERR_INVALID_ARG;
    if (c->Dff > kMaxDff || c->D > kMaxD) return MOE_ERR_UNSUPPORTED;
    if (c->activation < MOE_ACT_SWIGLU || c->activation > MOE_ACT_SWIGLU_CLAMPED) return MOE_ERR_UNSUPPORTED;
    if (c->activation == MOE_ACT_SWIGLU_CLAMPED &&
        !(c->act_limit > 0.0f && c->act_limit <= 3.0e38f))  // finite and positive (NaN fails)
        return MOE_ERR_INVALID_ARG;
    if (c->down_bits != 0 && c->down_bits != 4 && c->down_bits != 6) return MOE_ERR_UNSUPPORTED;
    if (c->expert_begin != 0 || c->expert_end != 0) {
        if (c->expert_begin < 0 || c->expert_begin >= c->expert_end || c->expert_end > c->E)
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

// carve the workspace; with base == nullptr only computes the size
size_t carve(const moe_config &c, char *base, Workspace *ws) {
    const size_t n = c.max_tokens, E = c.E, k = c.top_k, D = c.D, F = c.Dff;
    const size_t S = n * k;
    size_t off = 0;
    auto take = [&](size_t bytes) -> char * {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    Workspace w{};
    w.logits = (float *)take(n * E * 4);
    w.topk_idx = (int *)take(S * 4);
    w.topk_w = (float *)take(S * 4);
    w.counts = (int *)take(E * 4);
    w.offsets = (int *)take((E + 1) * 4);
    w.slot_token = (int *)take(S * 4);
    w.slot_k = (int *)take(S * 4);
    w.slot_of = (int *)take(S * 4);
    w.unique = (int *)take(E * 4);
    w.U = (int *)take(4);
    // f32 h of the check path, or the fused path's bf16 h blocks:
    // ceil(F / 256) K-slices x S slots x 512 bytes
    const size_t h_blocks = ((F / 64 + 3) / 4) * S * 512;
    w.h = (float *)take(S * F * 4 > h_blocks ? S * F * 4 : h_blocks);
    w.y = (float *)take(S * D * 4);
    w.status = (unsigned *)take(4 * 4);
    w.sync = (unsigned *)take(64 * 4);
    w.tlog = (unsigned long long *)take((n < 8 ? n : 8) * kTagSlots * 8);  // single launch: <= 8 tokens
    w.phase_ns = (unsigned long long *)take(16 * 1024 * 8);
    const size_t words = n > (size_t)kMaxTokens ? (n + 31) / 32 : 0;  // prefill cohorts only
    w.tbits = (unsigned *)take(E * words * 4);
    w.wbase = (int *)take(E * words * 4);
    w.x_stage = take(n * D * elem_size(c.x_dtype));
    w.out_stage = take(n * D * elem_size(c.out_dtype));
    if (ws) *ws = w;
    return off;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

moe_status check_planes(const moe_expert_planes *p) {
    if (!p) return MOE_ERR_INVALID_ARG;
    const void *ptrs[9] = {p->gate_q, p->gate_s, p->gate_b, p->up_q, p->up_s,
                           p->up_b, p->down_q, p->down_s, p->down_b};
    for (const void *q : ptrs)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool trace_enabled(const moe_plan *p) {
    if (p->cfg.flags & MOE_FLAG_TRACE) return true;
    const char *env = getenv("MOE_TRACE");
    return env && env[0] && env[0] != '0';
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_OOM: return "MOE_ERR_OOM";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status moe_plan_workspace_bytes(const moe_config *cfg, size_t *bytes) {
    moe_status st = validate_config(cfg);
    if (st != MOE_OK) return st;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    *bytes = carve(*cfg, nullptr, nullptr);
    return MOE_OK;
}

moe_status moe_plan_create(const moe_config *cfg, moe_plan **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_status st = validate_config(cfg);
    if (st != MOE_OK) return st;
    // the plan holds 64-byte aligned tensor maps
    const size_t plan_bytes = (sizeof(moe_plan) + 63) / 64 * 64;
    moe_plan *p = (moe_plan *)aligned_alloc(64, plan_bytes);
    if (!p) return MOE_ERR_OOM;
    memset((void *)p, 0, plan_bytes);
    p->cfg = *cfg;
    // default: every selected expert on the tcgen05 GEMMs where they apply (a
    // 128-row weight tile is dequantised once per 64 tokens, whatever the count)
    p->mma_min_tokens = cfg->mma_min_tokens > 0 ? cfg->mma_min_tokens : 1;
    if (const char *env = getenv("MOE_MMA_MIN_TOKENS")) {
        int v = atoi(env);
        if (v > 0) p->mma_min_tokens = v;
    }
    if (cudaGetDevice(&p->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
        cudaGetLastError();
        free(p);
        return MOE_ERR_CUDA;
    }
    p->ws_bytes = carve(*cfg, nullptr, nullptr);
    cudaError_t err = cudaMalloc(&p->ws_base, p->ws_bytes);
    if (err != cudaSuccess) {
        cudaGetLastError();
        free(p);
        return err == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA;
    }
    carve(*cfg, (char *)p->ws_base, &p->ws);
    p->fused_ok = false;
    // the single-launch kernel reads 4-bit down planes only
    if (!(cfg->flags & MOE_FLAG_F32_DEBUG) && cfg->down_bits != 6) {
        int max_smem = 0, per_sm = 0;
        cudaError_t e2 = cudaSuccess;
        if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device) ==
                cudaSuccess &&
            fused_layout(*cfg, p->num_sms, max_smem, &p->fused)) {
            e2 = fused_prepare(p->fused, &per_sm);
            // the cooperative launch needs every CTA resident at once
            p->fused_ok = e2 == cudaSuccess && per_sm >= 1;
        }
        if (trace_enabled(p))
            fprintf(stderr, "[moe] plan: fused=%d smem=%d stages=%d stage_bytes=%d down_units/stage=%d "
                    "heights=%d,%d ctas/sm=%d (%s)\n",
                    (int)p->fused_ok, p->fused.smem_bytes, p->fused.NS, p->fused.stage_bytes, p->fused.P,
                    p->fused.Hd[0], p->fused.Hd[1], per_sm, cudaGetErrorString(e2));
        cudaGetLastError();
    }
    if (cudaMemset(p->ws_base, 0, p->ws_bytes) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->ws_base);
        free(p);
        return MOE_ERR_CUDA;
    }
    // the host-mapped error word: the device writes it on a timeout, so the next
    // forward call can report the error without a synchronisation. Without
    // mapped host memory, errors are reported by moe_plan_check only.
    p->host_err = nullptr;
    {
        void *h = nullptr, *d = nullptr;
        if (cudaHostAlloc(&h, 64, cudaHostAllocMapped) == cudaSuccess) {
            memset(h, 0, 64);
            unsigned long long dev_addr = 0;
            if (cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess && d) {
                dev_addr = (unsigned long long)(uintptr_t)d;
                if (cudaMemcpy(p->ws.status + 2, &dev_addr, sizeof dev_addr, cudaMemcpyHostToDevice) ==
                    cudaSuccess)
                    p->host_err = static_cast<volatile unsigned *>(h);
            }
            if (!p->host_err) cudaFreeHost(h);
        }
        cudaGetLastError();
    }
    p->last_stream = nullptr;
    *out = p;
    return MOE_OK;
}

}  // extern "C"

namespace {

moe_status check_step_args(const moe_plan *plan, const void *x, const void *router_w,
                           const float *router_bias, const moe_expert_planes *planes, int n_tokens,
                           int top_k, const void *out) {
    if (!plan || !x || !router_w || !out) return MOE_ERR_INVALID_ARG;
    if (n_tokens < 1 || n_tokens > plan->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (top_k != plan->cfg.top_k) return MOE_ERR_INVALID_ARG;
    if (x == out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(router_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if (router_bias && ((uintptr_t)router_bias & 3u)) return MOE_ERR_INVALID_ARG;
    return check_planes(planes);
}

// one step, arguments already checked; next_router_w / next_router_bias: the
// next layer's router for the single launch to prefetch (or null)
moe_status forward_checked(moe_plan *plan, const void *x, const void *router_w,
                           const float *router_bias, const moe_expert_planes *planes, int n_tokens,
                           void *out, void *stream, const void *next_router_w,
                           const float *next_router_bias) {
    DeviceGuard guard(plan->device);
    cudaStream_t s = (cudaStream_t)stream;
    // an error a finished earlier step recorded on the device: report it, clear
    // the plan's error state on this stream, and run nothing
    if (plan->host_err && (plan->host_err[0] || plan->host_err[1] || plan->host_err[2])) {
        const moe_status err = plan->host_err[0] ? MOE_ERR_TIMEOUT
                             : plan->host_err[2] ? MOE_ERR_RANGE : MOE_ERR_CUDA;
        plan->host_err[0] = plan->host_err[1] = plan->host_err[2] = 0u;
        // reset the error bits, the barrier counter, the launch tag and the
        // tagged logits (a restarted tag must not meet an old logit)
        if (cudaMemsetAsync(plan->ws.status, 0, sizeof(unsigned), s) != cudaSuccess ||
            cudaMemsetAsync(plan->ws.sync, 0, 64 * sizeof(unsigned), s) != cudaSuccess ||
            cudaMemsetAsync(plan->ws.tlog, 0, (size_t)std::min(plan->cfg.max_tokens, 8) * kTagSlots * 8, s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        return err;
    }
    StepArgs a{};
    // the test hook stalls only the plan's first step
    const unsigned step_flags = plan->forwards == 0 ? plan->cfg.flags : plan->cfg.flags & ~(unsigned)MOE_FLAG_TEST_STALL;
    a.s = shape_of(plan->cfg, n_tokens, step_flags);
    a.x = x;
    a.router_w = router_w;
    a.router_bias = router_bias;
    a.planes = *planes;
    a.out = out;
    a.next_router_w = next_router_w;
    a.next_router_bias = next_router_bias;

    // n <= 8: one single-launch step; 9..kChunkMaxTokens: chunks of at most 8
    // tokens through it (unless the plan asks for the grouped path); else the
    // grouped multi-kernel path
    const int fmax = fused_max_tokens();
    const bool chunked = n_tokens > fmax && n_tokens <= kChunkMaxTokens &&
                         !(plan->cfg.flags & MOE_FLAG_GROUPED_COHORTS);
    bool fused = plan->fused_ok && (n_tokens <= fmax || chunked);
    const moe::TMaps *tm = nullptr;
    if (fused) {
        // tensor maps describe the plane pointers: reuse the cached ones for
        // these planes, else encode into the next cache entry
        for (int i = 0; i < moe_plan::kTmCache && !tm; ++i) {
            const moe_plan::TmEntry &en = plan->tm_cache[i];
            if (en.valid && memcmp(&en.planes, planes, sizeof *planes) == 0) tm = &en.tmaps;
        }
        if (!tm) {
            moe_plan::TmEntry &en = plan->tm_cache[plan->tm_next];
            plan->tm_next = (plan->tm_next + 1) % moe_plan::kTmCache;
            en.valid = fused_encode_tmaps(plan->cfg, plan->fused, *planes, &en.tmaps);
            en.planes = *planes;
            if (en.valid) tm = &en.tmaps;
            else if (trace_enabled(plan)) fprintf(stderr, "[moe] tensor map encoding failed\n");
        }
        fused = tm != nullptr;
    }
    const bool prefill = n_tokens > kMaxTokens;
    const char *path = prefill ? "prefill" : !fused ? "grouped" : n_tokens <= fmax ? "fused" : "fused-chunks";
    if (trace_enabled(plan))
        fprintf(stderr, "[moe] forward n=%d E=%d k=%d D=%d Dff=%d path=%s\n", n_tokens,
                a.s.E, a.s.k, a.s.D, a.s.F, path);
    int launched = 0;
    cudaError_t err = cudaSuccess;
    if (fused && n_tokens <= fmax) {
        err = launch_fused(a, plan->ws, plan->fused, *tm, s, launched);
    } else if (fused) {
        // balanced chunks (sizes differ by at most one token); chunk c reads
        // and writes its own rows of x, out and the logits, and the grouping
        // kernel then routes the whole cohort from those logits for
        // moe_get_routing (the same decisions each chunk took on the device)
        const int nch = (n_tokens + fmax - 1) / fmax;
        const size_t xrow = (size_t)a.s.D * elem_size(plan->cfg.x_dtype);
        const size_t orow = (size_t)a.s.D * elem_size(plan->cfg.out_dtype);
        for (int c = 0, t0 = 0; c < nch && err == cudaSuccess; ++c) {
            const int nc = (int)((long long)n_tokens * (c + 1) / nch) - t0;
            StepArgs ac = a;
            ac.s.n = nc;
            ac.x = static_cast<const char *>(x) + (size_t)t0 * xrow;
            ac.out = static_cast<char *>(out) + (size_t)t0 * orow;
            Workspace wc = plan->ws;
            wc.logits = plan->ws.logits + (size_t)t0 * a.s.E;
            err = launch_fused(ac, wc, plan->fused, *tm, s, launched);
            t0 += nc;
        }
        if (err == cudaSuccess) err = launch_topk_group(a, plan->ws, s, launched);
    } else if (prefill) {
        // more tokens than a decode cohort: token bitmaps for the grouping, and
        // the tcgen05 GEMMs loop over each expert's tokens (a grouped GEMM); the
        // router on the tensor cores too, except on the f32 check path
        const bool rtc = !(plan->cfg.flags & MOE_FLAG_F32_DEBUG) && router_tc_supported(a.s);
        err = rtc ? launch_router_tc(a, plan->ws, s, launched) : launch_router_logits(a, plan->ws, s, launched);
        if (err == cudaSuccess) err = launch_prefill_route(a, plan->ws, plan->cfg.max_tokens, s, launched, rtc);
        const int thr = (plan->cfg.flags & MOE_FLAG_F32_DEBUG) ? 0 : plan->mma_min_tokens;
        if (err == cudaSuccess) err = launch_experts(a, plan->ws, thr, s, launched);
    } else {
        err = launch_router_logits(a, plan->ws, s, launched);
        if (err == cudaSuccess) err = launch_topk_group(a, plan->ws, s, launched);
        // the f32 check path keeps every expert on the exact f32 kernels; the
        // others with at least mma_min_tokens tokens take the tcgen05 GEMMs
        // where the shape allows them
        const int thr = (plan->cfg.flags & MOE_FLAG_F32_DEBUG) ? 0 : plan->mma_min_tokens;
        if (err == cudaSuccess) err = launch_experts(a, plan->ws, thr, s, launched);
    }
    plan->launches += launched;
    plan->forwards += 1;
    plan->last_stream = s;
    plan->last_n = n_tokens;
    if (err != cudaSuccess) {
        fprintf(stderr, "[moe] forward launch failed (%s path): %s\n", path, cudaGetErrorString(err));
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_decode_forward(moe_plan *plan, const void *x, const void *router_w,
                              const float *router_bias, const moe_expert_planes *planes,
                              int n_tokens, int top_k, void *out, void *stream) {
    moe_status st = check_step_args(plan, x, router_w, router_bias, planes, n_tokens, top_k, out);
    if (st != MOE_OK) return st;
    return forward_checked(plan, x, router_w, router_bias, planes, n_tokens, out, stream, nullptr, nullptr);
}

moe_status moe_decode_forward_layers(moe_plan *plan, const moe_layer_io *layers, int n_layers,
                                     int n_tokens, int top_k, void *stream) {
    if (!plan || !layers || n_layers < 1) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        const moe_layer_io &io = layers[l];
        moe_status st = check_step_args(plan, io.x, io.router_w, io.router_bias, &io.planes, n_tokens,
                                        top_k, io.out);
        if (st != MOE_OK) return st;
    }
    for (int l = 0; l < n_layers; ++l) {
        const moe_layer_io &io = layers[l];
        const moe_layer_io *next = l + 1 < n_layers ? &layers[l + 1] : nullptr;
        moe_status st = forward_checked(plan, io.x, io.router_w, io.router_bias, &io.planes, n_tokens,
                                        io.out, stream, next ? next->router_w : nullptr,
                                        next ? next->router_bias : nullptr);
        if (st != MOE_OK) return st;
    }
    return MOE_OK;
}

moe_status moe_decode_forward_host(moe_plan *plan, const void *x_host, const void *router_w,
                                   const float *router_bias, const moe_expert_planes *planes,
                                   int n_tokens, int top_k, void *out_host, void *stream) {
    if (!plan || !x_host || !out_host) return MOE_ERR_INVALID_ARG;
    if (n_tokens < 1 || n_tokens > plan->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t xb = (size_t)n_tokens * plan->cfg.D * elem_size(plan->cfg.x_dtype);
    const size_t ob = (size_t)n_tokens * plan->cfg.D * elem_size(plan->cfg.out_dtype);
    if (cudaMemcpyAsync(plan->ws.x_stage, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    moe_status st = moe_decode_forward(plan, plan->ws.x_stage, router_w, router_bias, planes,
                                       n_tokens, top_k, plan->ws.out_stage, stream);
    if (st != MOE_OK) return st;
    if (cudaMemcpyAsync(out_host, plan->ws.out_stage, ob, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_plan_check(moe_plan *plan) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    unsigned status = 0;
    if (cudaMemcpy(&status, plan->ws.status, sizeof status, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (plan->host_err) plan->host_err[0] = plan->host_err[1] = plan->host_err[2] = 0u;
    if (status) {
        // clear the error bits (words 2..3 keep the host word's address) and the
        // grid-barrier counters
        cudaMemset(plan->ws.status, 0, sizeof(unsigned));
        cudaMemset(plan->ws.sync, 0, 64 * sizeof(unsigned));
        cudaMemset(plan->ws.tlog, 0, (size_t)std::min(plan->cfg.max_tokens, 8) * kTagSlots * 8);
        cudaDeviceSynchronize();
        return (status & kDevErrTimeout) ? MOE_ERR_TIMEOUT
             : (status & kDevErrRange) ? MOE_ERR_RANGE : MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_get_routing(moe_plan *plan, int32_t *topk_idx, float *topk_w, int32_t *counts,
                           int32_t *offsets, int32_t *slot_token, int32_t *slot_k,
                           int32_t *unique, int32_t *U) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (plan->last_n < 1) return MOE_ERR_INVALID_ARG;  // no forward call yet
    DeviceGuard guard(plan->device);
    if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    const Workspace &w = plan->ws;
    const size_t S = (size_t)plan->last_n * plan->cfg.top_k, E = plan->cfg.E;
    struct Copy { void *dst; const void *src; size_t bytes; } copies[] = {
        {topk_idx, w.topk_idx, S * 4}, {topk_w, w.topk_w, S * 4},
        {counts, w.counts, E * 4},     {offsets, w.offsets, (E + 1) * 4},
        {slot_token, w.slot_token, S * 4}, {slot_k, w.slot_k, S * 4},
        {unique, w.unique, E * 4},     {U, w.U, 4},
    };
    for (const Copy &c : copies)
        if (c.dst && cudaMemcpy(c.dst, c.src, c.bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    return MOE_OK;
}

moe_status moe_get_phase_times(moe_plan *plan, uint64_t *times, int max_entries, int *ctas) {
    if (!plan || !times || max_entries < 0 || !ctas) return MOE_ERR_INVALID_ARG;
    if (!plan->fused_ok) return MOE_ERR_UNSUPPORTED;
    DeviceGuard guard(plan->device);
    if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    *ctas = plan->fused.G;
    size_t count = (size_t)plan->fused.G * 16;
    if ((size_t)max_entries < count) count = (size_t)max_entries;
    if (count && cudaMemcpy(times, plan->ws.phase_ns, count * 8, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_plan_launch_count(const moe_plan *plan, uint64_t *count) {
    if (!plan || !count) return MOE_ERR_INVALID_ARG;
    *count = plan->launches;
    return MOE_OK;
}

moe_status moe_plan_free(moe_plan *plan) {
    if (!plan) return MOE_OK;
    moe_status st = MOE_OK;
    {
        DeviceGuard guard(plan->device);
        if (cudaStreamSynchronize(plan->last_stream) != cudaSuccess) {
            cudaGetLastError();
            st = MOE_ERR_CUDA;
        }
        if (cudaFree(plan->ws_base) != cudaSuccess) {
            cudaGetLastError();
            st = MOE_ERR_CUDA;
        }
        if (plan->host_err && cudaFreeHost((void *)plan->host_err) != cudaSuccess) {
            cudaGetLastError();
            st = MOE_ERR_CUDA;
        }
    }
    free(plan);
    return st;
}

}  // extern "C"
