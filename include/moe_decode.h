/*
 * moe_decode.h -- C ABI of the quantized MoE decode library (GB300, sm_103a).
 *
 * One call runs one MoE layer's decode step for a cohort of 1..64 tokens
 * (and, on the prefill path, for cohorts of up to 8192 tokens):
 *   1. router GEMV, softmax over all experts, top-k, renormalise the k weights
 *   2. group the n*k (token, rank) slots by expert, de-duplicated, so every
 *      selected expert's planes are streamed from HBM once per step (once
 *      per chunk for cohorts that run in chunks; see moe_decode_forward)
 *   3. per selected expert: h = act(Wg x, Wu x) on affine 4-bit weights
 *      (SwiGLU silu(g) * u by default; GeGLU and a clamped SwiGLU as options)
 *   4. y = Wd h, and out[t] = sum_j w[t,j] * y[t,j] in rank order j,
 *      f32 partials with a single final rounding
 *
 * Sources (mlxcel GitHub issues):
 *   #1616 "perf(moe): batched decode scales 1.55x against 3.25x on dense"
 *     Current Behavior - the decode MoE block (SwitchGLU + moe_weighted_sum),
 *       the B=1-only fused kernel and the 4-bit group-64 expert format;
 *     Leading hypothesis - per-slot expert traffic, no de-duplication;
 *     Proposed Solution - a token dimension for the fused kernel and
 *       de-duplicated expert planes;
 *     Implementation Notes - n_tokens as a runtime extent, f32 partials with
 *       a single final rounding, decline unsupported shapes instead of
 *       failing, validate shapes before dispatch.
 *   #1859 "perf(moe): attribute the MoE decode gap at the M = 1 expert
 *     gather", Problem / Background - one expert row per (token, k) slot.
 *
 * Conventions
 *   - Every pointer passed to moe_decode_forward is a DEVICE pointer owned by
 *     the caller, except where a comment says host. The library never frees
 *     or retains caller memory beyond the call.
 *   - The plan owns its workspace (device memory sized at plan creation for
 *     max_tokens). moe_decode_forward allocates nothing.
 *   - Calls are asynchronous on the given CUDA stream (NULL = legacy default
 *     stream) unless documented otherwise. Calls on one plan must not overlap
 *     on the device (they share the workspace): issue them on one stream, or
 *     order the streams.
 *   - Errors are returned as moe_status, never thrown or trapped. Argument
 *     checks happen on the host before any launch; on a non-OK return from
 *     a check, nothing was launched.
 *
 * Data formats (MLX-style affine 4-bit quantisation, group 64)
 *   plane q : uint32 [E, rows, cols/8]; nibble j (bits 4j..4j+3) of word i
 *             is the code (0..15) of input column 8*i + j
 *   6-bit down planes (cfg.down_bits = 6): bytes [E, D, 3*Dff/4]; the codes
 *             (0..63) of a row form one little-endian bit stream, code j in
 *             bits 6j..6j+5 (four codes in three bytes)
 *   scale s : bf16 [E, rows, cols/64]; bias b : bf16 [E, rows, cols/64]
 *   weight  : w = s * q + b, groups of 64 consecutive input columns
 *   gate, up: rows = Dff, cols = D;  down: rows = D, cols = Dff
 *   All planes row-major, expert-major, densely packed; 16-byte aligned.
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad n_tokens / top_k / dims */
    MOE_ERR_UNSUPPORTED = 2,  /* a shape or format this library declines */
    MOE_ERR_CUDA = 3,         /* a CUDA call or launch failed */
    MOE_ERR_OOM = 4,          /* workspace allocation failed */
    MOE_ERR_TIMEOUT = 5,      /* a device-side wait gave up (bounded spin) */
    MOE_ERR_RANGE = 6         /* an intermediate of the single-launch kernel left
                                 the range of its f16 operand (|h| > 65504): that
                                 step's output is invalid (reported like a
                                 timeout; MOE_FLAG_F32_DEBUG computes such
                                 layers in f32) */
} moe_status;

/* element types of x, router weights and out */
enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };

/* plan flags */
enum {
    /* CUDA-core f32 path for every expert: weights dequantised exactly to f32,
     * f32 accumulation throughout. Slower; used to check numerics. */
    MOE_FLAG_F32_DEBUG = 1u << 0,
    /* print the chosen path of each forward call to stderr */
    MOE_FLAG_TRACE = 1u << 1,
    /* record per-CTA timestamps of the fused kernel's phases (see
     * moe_get_phase_times); costs a few global stores per CTA */
    MOE_FLAG_PHASE_TIMES = 1u << 2,
    /* cohorts of 9..16 tokens take the grouped multi-kernel path (every
     * selected expert streamed once per step, tensor-core GEMMs for experts
     * with at least mma_min_tokens tokens) instead of chunks of the
     * single-launch kernel; see moe_decode_forward */
    MOE_FLAG_GROUPED_COHORTS = 1u << 3,
    /* TEST ONLY: in the plan's first forward call on the fused path, CTA 0
     * reaches the first grid barrier only after another CTA's bounded wait has
     * run out (about 1 s), so that step ends with a recorded timeout and
     * garbage output; later calls of the plan run normally. */
    MOE_FLAG_TEST_STALL = 1u << 8
};

/* expert activation h = act(g, u), g = Wg x, u = Wu x. The pages name the
 * variants without formulas (#1616 Implementation Notes: the GeGLU variant of
 * the fused kernel; #1859 Problem / Background: deepseek_v4's clamp stage);
 * the readings below are the plainest ones. */
enum {
    MOE_ACT_SWIGLU = 0,          /* silu(g) * u, silu(z) = z / (1 + exp(-z)) */
    MOE_ACT_GEGLU = 1,           /* gelu(g) * u, gelu(z) = z/2 (1 + erf(z / sqrt 2)) */
    MOE_ACT_GEGLU_TANH = 2,      /* gelu in its tanh form:
                                    z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) */
    MOE_ACT_SWIGLU_CLAMPED = 3   /* silu(min(g, L)) * min(max(u, -L), L),
                                    L = act_limit */
};

typedef struct {
    int E;              /* experts, 1..1024 */
    int top_k;          /* experts per token, 1..min(E, 16) */
    int D;              /* hidden size; multiple of 64, <= 16384 */
    int Dff;            /* expert intermediate size; multiple of 64, <= 8192 */
    int bits;           /* must be 4 */
    int group_size;     /* must be 64 */
    int max_tokens;     /* largest cohort a forward call may pass, 1..8192;
                           above 64 the plan also holds the prefill path's
                           workspace (h and y for max_tokens * top_k slots) */
    int x_dtype;        /* MOE_DTYPE_* of x */
    int router_dtype;   /* MOE_DTYPE_* of the router weights */
    int out_dtype;      /* MOE_DTYPE_* of out */
    unsigned flags;     /* MOE_FLAG_* */
    int mma_min_tokens; /* per-expert token count from which an expert of the
                           grouped and prefill paths takes the tcgen05 GEMMs
                           (the rest take the f32 GEMV; shapes whose D or Dff is
                           not a multiple of 128 keep every expert on the GEMV);
                           0 = library default, 1 */
    /* ABI version 2 */
    int activation;     /* MOE_ACT_* */
    float act_limit;    /* the clamp bound L of MOE_ACT_SWIGLU_CLAMPED (finite,
                           > 0); ignored by the other activations */
    int down_bits;      /* bits of the down codes: 0 or 4 (uint32 words), 6
                           (the byte stream above; Dff must be a multiple of 64) */
    int expert_begin;   /* the experts this plan owns, [expert_begin, expert_end):
                           routing still ranks all E experts, but only owned */
    int expert_end;     /* experts are streamed and summed (expert-parallel
                           shard); both 0 = all E experts */
} moe_config;

typedef struct {
    const uint32_t *gate_q; /* [E, Dff, D/8]  */
    const uint16_t *gate_s; /* [E, Dff, D/64] bf16 */
    const uint16_t *gate_b; /* [E, Dff, D/64] bf16 */
    const uint32_t *up_q;   /* [E, Dff, D/8]  */
    const uint16_t *up_s;   /* [E, Dff, D/64] bf16 */
    const uint16_t *up_b;   /* [E, Dff, D/64] bf16 */
    const uint32_t *down_q; /* [E, D, Dff/8]; bytes [E, D, 3*Dff/4] when
                               cfg.down_bits = 6 (16-byte aligned) */
    const uint16_t *down_s; /* [E, D, Dff/64] bf16 */
    const uint16_t *down_b; /* [E, D, Dff/64] bf16 */
} moe_expert_planes;

typedef struct moe_plan moe_plan;

/* Library ABI version (MOE_ABI_VERSION of the build). No counterpart on the
 * pages (a library utility). */
int moe_abi_version(void);

/* Human-readable name of a status code (static string). Source: #1616
 * Implementation Notes (errors are returned so the caller can fall back). */
const char *moe_status_str(moe_status s);

/* Device bytes a plan for cfg would allocate. Host-only; no CUDA call.
 * Returns INVALID_ARG / UNSUPPORTED exactly as moe_plan_create would.
 * Source: #1616 Implementation Notes (validate shapes before dispatch). */
moe_status moe_plan_workspace_bytes(const moe_config *cfg, size_t *bytes);

/* Validate cfg and allocate the plan's workspace on the current device.
 * Source: #1616 Implementation Notes -- templating on k / Din / Dff / bits /
 * group size with n_tokens a runtime extent, a decline for configurations the
 * kernels do not cover, validation before any dispatch.
 * The plan is bound to that device. Decline (UNSUPPORTED): bits != 4,
 * group_size != 64, D or Dff not a multiple of 64, D > 16384, Dff > 8192,
 * E > 1024, top_k > 16, activation not a MOE_ACT_*, down_bits not 0, 4 or 6.
 * INVALID_ARG: null pointers, non-positive sizes, top_k > E, max_tokens
 * outside 1..8192, unknown dtypes, negative mma_min_tokens, unknown flags, a
 * clamp bound that is not finite and positive (MOE_ACT_SWIGLU_CLAMPED), an
 * expert range other than 0 <= expert_begin < expert_end <= E (or 0, 0).
 * A plan with 6-bit down planes runs every cohort on the grouped path.
 * Source of the expert range: #1616 Proposed Solution (one read of each
 * expert plane per step, which an expert-parallel split keeps per GPU).
 * OOM / CUDA: the
 * allocation failed (nothing leaks). On success *out owns the workspace
 * until moe_plan_free. */
moe_status moe_plan_create(const moe_config *cfg, moe_plan **out);

/* One decode step. Source: #1616 Current Behavior (the routed decode block:
 * router, SwitchGLU experts, moe_weighted_sum) and Proposed Solution (a token
 * dimension and one read of each selected expert plane per step); #1859
 * Problem / Background (the per-(token, k) gather this replaces).
 *   x           [n_tokens, D] of cfg.x_dtype (device)
 *   router_w    [E, D] of cfg.router_dtype (device)
 *   router_bias [E] f32 added to the logits, or NULL (device)
 *   planes      expert planes (struct in host memory, pointers to device)
 *   n_tokens    cohort size, 1..cfg.max_tokens (runtime extent: no
 *               re-specialisation per n)
 *   top_k       must equal cfg.top_k (checked, INVALID_ARG otherwise)
 *   out         [n_tokens, D] of cfg.out_dtype (device); must not alias x
 *   stream      cudaStream_t, or NULL for the legacy default stream
 * Paths, chosen on the host from n_tokens and the plan:
 *   n_tokens 1..8    one launch of the single-launch kernel;
 *   n_tokens 9..16   balanced chunks of at most 8 tokens, each one launch of
 *                    the single-launch kernel (an expert picked in several
 *                    chunks is streamed once per chunk), then one grouping
 *                    kernel that writes the whole cohort's routing tables;
 *   n_tokens 17..64, or any n_tokens > 8 with MOE_FLAG_GROUPED_COHORTS:
 *                    the grouped multi-kernel path (router, top-k and
 *                    grouping, per-expert tcgen05 GEMMs (D and Dff multiples
 *                    of 128) or f32 GEMV kernels, combine);
 *   MOE_FLAG_F32_DEBUG, or a shape the single-launch kernel declines:
 *                    the grouped multi-kernel path with f32 GEMV kernels;
 *   n_tokens 65..max_tokens: the prefill path (#1616 Current Behavior and #1859
 *                    Problem / Background: the sorted matrix path, qmm, of
 *                    prompt processing): routing per token, grouping through
 *                    per-expert token bitmaps, then per expert a grouped GEMM
 *                    (tcgen05 over its tokens in blocks of 64, each weight
 *                    tile read once per block) or
 *                    the f32 GEMV for experts under mma_min_tokens, and the
 *                    combine.
 * Expert range. A plan that owns the experts [expert_begin, expert_end)
 * writes out[t] = sum over the ranks j whose expert it owns of w[t,j] *
 * y[t,j] (0 where it owns none): the plans of a partition of the experts
 * produce partial outputs that sum to the whole step (use out_dtype f32 for
 * partials that are summed afterwards). Routing (top-k and weights over all
 * E experts) is the same in every shard.
 * Asynchronous. Returns INVALID_ARG before any launch on a bad argument,
 * CUDA if a launch fails.
 * Device-side errors. Every wait inside a step is bounded (about 1 s); a wait
 * that gives up records MOE_ERR_TIMEOUT in the plan and the step's output is
 * garbage. Once that step has finished on the device, the next call on the
 * plan (this one, moe_decode_forward_host, or moe_plan_check) returns
 * MOE_ERR_TIMEOUT (MOE_ERR_RANGE for a saturated f16 intermediate, MOE_ERR_CUDA
 * for an internal error) and clears it; a
 * forward call that reports it launches nothing and only enqueues two small
 * memsets that reset the plan's error state on `stream`. A step that was
 * still running at the time is reported by a later call. The steps after a
 * timed-out one run normally: the grid-barrier counters stay consistent. */
moe_status moe_decode_forward(moe_plan *plan, const void *x, const void *router_w,
                              const float *router_bias, const moe_expert_planes *planes,
                              int n_tokens, int top_k, void *out, void *stream);

/* One layer's arguments of moe_decode_forward_layers (device pointers, as for
 * moe_decode_forward). */
typedef struct {
    const void *x;              /* [n_tokens, D] of cfg.x_dtype */
    const void *router_w;       /* [E, D] of cfg.router_dtype */
    const float *router_bias;   /* [E] f32 or NULL */
    moe_expert_planes planes;   /* this layer's expert planes */
    void *out;                  /* [n_tokens, D] of cfg.out_dtype; must not alias
                                   this layer's x (it may be the next layer's x) */
} moe_layer_io;

/* Decode steps of n_layers consecutive MoE layers of the plan's shape, in
 * order, on one stream: layer l is exactly moe_decode_forward on layers[l].
 * Source: #1616 Current Behavior (the routed decode block runs on all 48
 * layers every tick). On the single-launch path the launches form a chain with
 * programmatic dependent launch, and layer l's launch prefetches layer l+1's
 * router rows (and bias) into L2 while it streams its own experts, so the next
 * router GEMV reads L2 instead of HBM. A layer's x may be the previous layer's
 * out (a residual-free stack). Every layer's arguments are checked on the host
 * before the first launch (INVALID_ARG: nothing launched; n_layers must be at
 * least 1). Errors and ordering as for moe_decode_forward; moe_get_routing
 * then reports the last layer. */
moe_status moe_decode_forward_layers(moe_plan *plan, const moe_layer_io *layers, int n_layers,
                                     int n_tokens, int top_k, void *stream);

/* The same step with x and out in HOST memory (#1616 Current Behavior: the
 * decode tick of a serving loop hands activations in and out): copies x to the plan's device
 * staging buffer, runs moe_decode_forward, copies out back and synchronises
 * the stream before returning. Pinned host memory gives asynchronous copies;
 * pageable memory works but is slower. */
moe_status moe_decode_forward_host(moe_plan *plan, const void *x_host, const void *router_w,
                                   const float *router_bias, const moe_expert_planes *planes,
                                   int n_tokens, int top_k, void *out_host, void *stream);

/* The decode step without a plan and without any device allocation.
 *
 * For callers that cannot allocate device memory: for example code running
 * while a CUDA graph is being captured, runtimes that forbid cudaMalloc, or
 * processes whose device memory pool belongs to another framework. The pages
 * this library follows have no counterpart of this call; it exists only for
 * such callers.
 *
 * Runs the same single-launch kernel as moe_decode_forward, so it accepts what
 * that kernel accepts: n_tokens 1..8 and the shapes the kernel supports
 * (otherwise MOE_ERR_UNSUPPORTED). cfg gives the layer shape and dtypes.
 * MOE_FLAG_F32_DEBUG in cfg.flags is declined (MOE_ERR_UNSUPPORTED); every
 * other flag, and max_tokens, is ignored (no phase timing, no trace, no test
 * hook, no routing copy-out). All other arguments are as for
 * moe_decode_forward; the caller still owns x, router_w, router_bias, the
 * planes and out.
 *
 * Scratch: one statically sized device array of 4 MiB inside the library,
 * which every GPU that loads the library holds until the process exits. A call
 * whose scratch would exceed it returns MOE_ERR_UNSUPPORTED before any launch.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine); it issues one cudaMemsetAsync that clears the array's status word
 * and barrier counter, then the kernel, both on `stream`.
 *
 * The first call on a device looks up the array's device address on the
 * current device (a one-time set-up); make that first call before any stream
 * capture. The address is kept per device ordinal for the life of the
 * process: after cudaDeviceReset, or with a context other than the device's
 * primary context current, it is stale and this call must not be used. Every call on a device shares the one array: calls that overlap on
 * the GPU (different streams without ordering) race and give wrong results.
 * Asynchronous; device-side timeouts are not reported by this call. */
moe_status moe_decode_forward_noalloc(const moe_config *cfg, const void *x, const void *router_w,
                                      const float *router_bias, const moe_expert_planes *planes,
                                      int n_tokens, int top_k, void *out, void *stream);

/* Synchronise the plan's last stream and report a device-side timeout or
 * internal error recorded by earlier calls (then clear it). Source: #1616
 * Implementation Notes (errors are returned, never a terminate). */
moe_status moe_plan_check(moe_plan *plan);

/* Copy the routing and grouping of the plan's last forward call to HOST
 * arrays (any pointer may be NULL to skip it). Synchronises the last stream.
 * Source: #1616 Leading hypothesis (slots sorted by expert id) and Proposed
 * Solution (de-duplicated expert ids across the cohort).
 *   topk_idx [n,k] int32, topk_w [n,k] f32   (rank order: descending logit,
 *                                             ties to the lower expert id)
 *   counts [E], offsets [E+1]                (exclusive scan of counts)
 *   slot_token [n*k], slot_k [n*k]           (slots grouped by expert
 *                                             ascending, token ascending)
 *   unique [E] (first *U entries valid), U   (experts with count > 0)
 * With an expert range, topk_idx / topk_w cover every expert and the grouping
 * arrays cover the owned experts only (counts of the others are 0; the first
 * offsets[E] entries of slot_token / slot_k are valid). */
moe_status moe_get_routing(moe_plan *plan, int32_t *topk_idx, float *topk_w,
                           int32_t *counts, int32_t *offsets, int32_t *slot_token,
                           int32_t *slot_k, int32_t *unique, int32_t *U);

/* Phase timestamps (ns, %globaltimer) of the last fused step of a plan created
 * with MOE_FLAG_PHASE_TIMES. Source: #1859 Proposed Solution step 2 (split the
 * step into router, expert gather and combine and attribute the time): for
 * each CTA c, times[c*16 + i] with
 *   i = 0 start, 1 router done, 2 after grid barrier 1, 3 routing and work
 *   lists done, 4 gate/up done, 5 after grid barrier 2, 6 down done, 7 end;
 *   8/9 gate/up ns spent waiting for data / computing (consumer warp 0),
 *   10/11 the same for the down projection, 12 reserved (0), 13 gate/up
 *   chunks, 14 down tiles of the CTA.
 * Copies min(max_entries, ctas*16) entries to HOST memory, sets *ctas to the
 * kernel's CTA count, and synchronises the plan's last stream. */
moe_status moe_get_phase_times(moe_plan *plan, uint64_t *times, int max_entries, int *ctas);

/* Number of CUDA kernels this plan has enqueued since creation (host
 * counter; forward calls captured into a CUDA graph count once, at capture).
 * Source: #1859 Proposed Solution step 2 (attribute time per kernel). */
moe_status moe_plan_launch_count(const moe_plan *plan, uint64_t *count);

/* Free the plan's workspace (synchronises its last stream). NULL is a no-op.
 * No counterpart on the pages (a library utility). */
moe_status moe_plan_free(moe_plan *plan);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
