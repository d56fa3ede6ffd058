// decode_step.cu -- the decode step for cohorts of up to 8 tokens as one
// persistent kernel (one CTA per SM, cooperative launch, 20 warps: warps 0..15
// consume, warp 16 produces, warps 17 and 18 reduce, warp 19 copies routing
// tables out; after routing a setmaxnreg split gives the consumers 112 registers).
//
// Phases inside one launch:
//   R  router GEMV: logits[t, e] = x[t] . Wr[e] (+ bias). Each CTA owns at most
//      two experts (e = cta, cta + G) and publishes their logits as 64-bit words
//      (launch tag << 32 | value). Every CTA also stages x in shared memory as
//      f16 in the B-operand order of the tensor-core MMA, with per-group sums.
//   T  every CTA polls the tagged logits until all carry this launch's tag (the
//      exchange needs no grid barrier), then computes top-k, renormalised
//      weights and the grouping by expert itself (the same deterministic result
//      in every CTA, so there is no second exchange); one warp builds the
//      grouping, the slot table and the CTA's gate/up tile list.
//   A  gate/up: the U * Dff (gate row, up row) pairs of the selected experts are
//      split evenly over the CTAs; each CTA cuts its share into 16-row tiles.
//      The producer warp streams each tile (gate and up codes over all inputs,
//      and the tile's scales and biases) with 3-D TMA copies (128-byte swizzle)
//      into a shared-memory ring. All 16 consumer warps work on every stage,
//      each on its own pair of input groups, running m16n8k16 MMAs on the raw
//      4-bit codes; each warp writes its partial sums to one of two buffers and
//      a reducer warp sums the 16 partials in warp order and writes
//      h = w * act(g, u) as f16, one row per (token, expert) slot. -> barrier 2
//   B  down + combine: each CTA owns a slice of the D output rows for every
//      selected expert. The down codes stream into the same ring (issued as soon
//      as ring stages free up, before barrier 2); because the routing weight is
//      folded into h, every warp accumulates its share of sum_e Wd[e] h_e and one
//      fixed-order sum over warps gives the output with one final rounding.
//
// Sources (mlxcel GitHub issues):
//   #1616 "perf(moe): batched decode scales 1.55x against 3.25x on dense":
//     Proposed Solution - a token dimension for the fused decode kernel and one
//     read of each selected expert plane per step (de-duplication across the
//     cohort); Implementation Notes - f32 partials with a single final rounding,
//     n_tokens as a runtime extent.
//   #1859 "perf(moe): attribute the MoE decode gap at the M = 1 expert gather",
//     Problem / Background - the per-(token, k) gather this replaces.
//
// Numerics. Codes enter the MMA as exact integers through magic-exponent bit
// tricks, two codes per logic op; products and sums are f32.
//   gate/up (f16): OR-ing 1024 onto a code nibble gives 1024 + q (low nibble) or
//     1024 + 16 q (high nibble) with no shift; x is staged with the inputs of the
//     high nibbles divided by 16, so per group sum((1024 + m q) x / m) =
//     1024 sum(x / m) + sum(q x), and the row's contribution is
//     s * (acc - 1024 sum(x / m)) + b * sum(x).
//   down (f16): every nibble shifted down and OR-ed onto 1024.0 gives 1024 + q;
//     the row contribution is s * acc + (b - 1024 s) * sum(h); tile row 15 is
//     fed zero codes, so its MMA row returns 1024 * sum(h) for free.
// x and h enter the MMA as f16 (10 mantissa bits): x is scaled per token by a
// power of two when its magnitudes leave f16's comfortable range (phase R), and
// an |h| beyond f16's range is saturated and reported (MOE_ERR_RANGE). This path
// is held to the bf16 tolerance; the f32 check path keeps every product in f32.
// Every reduction has a fixed order: results are bitwise reproducible.
//
// MMA row mapping. Lane (g, c) of a warp holds MMA rows g and g + 8; they map to
// tile rows 2g and 2g + 1, so the eight rows a warp reads at once sit in eight
// different 16-byte columns of the 128-byte swizzle and the reads are free of
// bank conflicts.
//
// Every wait is bounded (globaltimer, 1 s). A timeout sets a status bit and an
// abort flag; the CTA then skips the remaining waits, still passes every barrier
// it shares with its own threads, lets its copies in flight land and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "activation.cuh"
#include "device_status.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {

namespace {

constexpr int kCW = 16;                      // consumer warps (the MMA work)
constexpr int kWarps = 20;                   // + one warpgroup: a producer warp and two reducer warps
constexpr int kThreads = kWarps * 32;
constexpr int kConsThreads = kCW * 32;
constexpr int kProducer = kCW;               // streams every stage into the ring
constexpr int kReducer0 = kCW + 1;           // warps kReducer0 + b reduce gate/up partial buffer b
constexpr int kRegsConsumer = 112;           // register split after the routing phase:
constexpr int kRegsProducer = 32;            // 512 * 112 + 128 * 32 = 640 * 96, the launch's registers
constexpr int kNFast = 8;                    // cohort sizes 1..8 (one n8 MMA tile)
constexpr int kMaxSlotsF = kNFast * kMaxTopK;
constexpr int kMaxRing = 8;
constexpr int kStageSlices = 8;              // K-slices (256 inputs each) per gate/up stage
constexpr int kMaxTilesF = 160;
constexpr int kStampsPerCta = 16;
constexpr int kMaxDI = 2;                    // down items (unit, group pair) per warp per stage
constexpr int kPartStride = 264;             // floats per warp partial (256 + 8: banks of the
                                             // four warps a reducing lane sums do not collide)
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s bound on any wait

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// bf16 value `which` (0: low half, 1: high half) of a packed pair, widened to f32
__device__ __forceinline__ float bf_half(uint32_t w, int which) {
    return __uint_as_float(which ? (w & 0xFFFF0000u) : (w << 16));
}

__device__ __forceinline__ uint16_t f2bf(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// f16 bits of f (round to nearest even); a magnitude beyond the largest f16
// saturates to +-65504 and sets *over
__device__ __forceinline__ uint16_t f2h_sat(float f, bool &over) {
    if (!(fabsf(f) <= 65504.0f)) {
        over = true;
        f = f != f ? 0.0f : copysignf(65504.0f, f);
    }
    return __half_as_ushort(__float2half_rn(f));
}

// codes of inputs p and p+4 of a packed word, as f16x2 values 1024 + q
__device__ __forceinline__ uint32_t code_pair(uint32_t word, int p) {
    return ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
}

// two k16 MMA steps over one packed word per MMA row (rows g and g+8) and the
// matching activation word (4 bf16x2 pairs: (v0,v4) (v1,v5) (v2,v6) (v3,v7))
__device__ __forceinline__ void mma_word(float (&acc)[4], uint32_t wg, uint32_t wg8, uint4 v) {
    uint32_t a0[4] = {code_pair(wg, 0), code_pair(wg8, 0), code_pair(wg, 1), code_pair(wg8, 1)};
    ptx::mma_f16_16816(acc, a0, v.x, v.y);
    uint32_t a1[4] = {code_pair(wg, 2), code_pair(wg8, 2), code_pair(wg, 3), code_pair(wg8, 3)};
    ptx::mma_f16_16816(acc, a1, v.z, v.w);
}

// f16 variant: f16 carries 10 mantissa bits, so both nibbles of a byte are
// codes as they sit: OR-ing 0x6400 (1024.0) onto bits 0..3 gives 1024 + q and
// onto bits 4..7 gives 1024 + 16 q. One shift by 8 brings the odd bytes down.
// The activations of the 16 q positions (inputs 8i+1, 3, 5, 7) are staged
// divided by 16, so every product is (1024 m + q) x / m with m = 1 or 16, and
// per group sum((1024 + m q) x / m) = 1024 * sum(x / m) + sum(q x).
__device__ __forceinline__ uint32_t code_lo(uint32_t w) { return (w & 0x000F000Fu) | 0x64006400u; }
__device__ __forceinline__ uint32_t code_hi(uint32_t w) { return (w & 0x00F000F0u) | 0x64006400u; }

__device__ __forceinline__ void mma_word_f16(float (&acc)[4], uint32_t wg, uint32_t wg8, uint4 v) {
    uint32_t a0[4] = {code_lo(wg), code_lo(wg8), code_hi(wg), code_hi(wg8)};
    ptx::mma_f16_16816(acc, a0, v.x, v.y);
    const uint32_t s8 = wg >> 8, t8 = wg8 >> 8;
    uint32_t a1[4] = {code_lo(s8), code_lo(t8), code_hi(s8), code_hi(t8)};
    ptx::mma_f16_16816(acc, a1, v.z, v.w);
}

__device__ __forceinline__ void load8f(const void *p, size_t i, int dtype, float (&v)[8]) {
    if (dtype == MOE_DTYPE_F32) {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        const float4 a = __ldg(q), b = __ldg(q + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + i));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

// byte offset of a swizzled shared-memory box element: TMA's 128/64/32-byte
// swizzle XORs the 16-byte column (address bits 4..6) with bits 7..9 of the
// offset from the 1024-byte aligned box base (mask 7, 3 or 1)
__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t mask) {
    return off ^ (((off >> 7) & mask) << 4);
}

// position of input f (within one expert's Dff) in the stored h row: each block
// of 16 is stored as the pairs (0,4) (1,5) (2,6) (3,7) (8,12) ... of the MMA
// B-operand order
__device__ __forceinline__ int h_pos(int f) {
    const int i = f & 15, lo = i & 7;
    return (f & ~15) | (i & 8) | (2 * (lo & 3) + (lo >> 2));
}

struct Smem {
    uint64_t *full, *empty;  // ring slots: data landed / consumed by every consumer warp
    uint64_t *pfull, *pempty;  // gate/up partial buffers: all partials written / reduced
    int *misc;             // [0] abort [1] barrier ok [2] U [3] tiles [4] b0 [5] b1
                           // [6] stages issued [7] x needs per-token scaling
                           // [8..9] partials written [10..11] shares reduced
                           // [16..23] stage release counts [24..39] grouping scans
                           // [40..47] per-token scale of x as f32 (2^e, 1 unless scaled)
                           // [48..55] per-token scale of h as f32 (2^2e or 1)
    unsigned long long *s_mask;
    int *s_idx, *s_st, *s_sk, *s_of, *s_counts, *s_off, *s_unique;
    float *s_w, *slot_w;
    int4 *uroute;          // per selected expert u: (expert, token mask, first slot, 0)
    int4 *tiles;           // per tile: (u, f0 of the box within the expert, valid lo, valid hi),
                           // then (expert, token mask, first slot, 0)
    unsigned char *xs;
    float *xsum;
    float *red;            // gate/up partials [2][kCW][32][8]; router / final scratch
    unsigned char *ring;
};

__device__ __forceinline__ Smem carve_smem(unsigned char *base, const DecodeLayout &L, int E) {
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(base + L.off_bar);
    s.empty = s.full + kMaxRing;
    s.pfull = s.full + 2 * kMaxRing;
    s.pempty = s.pfull + 2;
    s.misc = reinterpret_cast<int *>(base + L.off_misc);
    unsigned char *r = base + L.off_route;
    s.s_mask = reinterpret_cast<unsigned long long *>(r);
    int *ip = reinterpret_cast<int *>(r + 8 * (size_t)E);
    s.s_idx = ip; ip += kMaxSlotsF;
    s.s_w = reinterpret_cast<float *>(ip); ip += kMaxSlotsF;
    s.s_st = ip; ip += kMaxSlotsF;
    s.s_sk = ip; ip += kMaxSlotsF;
    s.s_of = ip; ip += kMaxSlotsF;
    s.slot_w = reinterpret_cast<float *>(ip); ip += kMaxSlotsF;
    s.s_counts = ip; ip += E;
    s.s_off = ip; ip += E + 1;
    s.s_unique = ip;
    s.tiles = reinterpret_cast<int4 *>(base + L.off_tiles);
    s.uroute = s.tiles + 2 * kMaxTilesF;
    s.xs = base + L.off_x;
    s.xsum = reinterpret_cast<float *>(base + L.off_xsum);
    s.red = reinterpret_cast<float *>(base + L.off_red);
    s.ring = base + L.off_ring;
    return s;
}

__device__ __forceinline__ void set_timeout(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    report_error(status, kDevErrTimeout);
}

// Bounded wait on an mbarrier phase; false on timeout or abort. The waiting
// thread suspends inside try_wait (a suspend-time hint) instead of polling: a
// polling warp takes issue slots from the warps doing the MMA work (measured on
// GB300: four polling warps slow sixteen MMA warps by ~40 %, suspended ones by
// nothing).
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool wait_phase_loop(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                unsigned *status) {
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_hint(bar, parity, kSuspendNs)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitNs) {
            set_timeout(abort_flag, status);
            return false;
        }
    }
}
// Consumer warps: the slow path stays out of line, so the hot loops that wait
// keep a short body.
__device__ __noinline__ bool wait_phase_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                             unsigned *status) {
    return wait_phase_loop(bar, parity, abort_flag, status);
}
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, status);
}
// Producer and reducer warps (32 registers after the split) wait inline: a
// function call made from that region leads ptxas to drop the setmaxnreg split
// altogether (every warp then keeps 96 registers).
__device__ __forceinline__ bool wait_phase_inl(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned *status) {
    return wait_phase_loop(bar, parity, abort_flag, status);
}

// Grid-wide barrier of all threads. The arrival counter only grows, by G per
// barrier and 2G per launch; `target` is its value once every CTA has arrived
// (the launch's base value plus G or 2G).
__device__ __forceinline__ void cta_sync(bool consumers_only) {
    if (consumers_only) ptx::named_bar(1, kConsThreads); else __syncthreads();
}

__device__ __forceinline__ bool grid_barrier(unsigned long long *cnt, unsigned long long target,
                                             volatile int *flag_ok, volatile int *abort_flag,
                                             unsigned *status, bool consumers_only = false) {
    cta_sync(consumers_only);
    if (threadIdx.x == 0) {
        int ok = 1;
        // the release add orders every write of this CTA before it (the CTA
        // barrier above, then release cumulativity); no separate fence
        ptx::red_release_gpu_u64(cnt, 1ull);
        if (ptx::ld_acquire_gpu_u64(cnt) < target) {
            const unsigned long long t0 = globaltimer();
            while (ptx::ld_acquire_gpu_u64(cnt) < target) {
                if (*abort_flag || globaltimer() - t0 > kWaitNs) {
                    ok = 0;
                    set_timeout(abort_flag, status);
                    break;
                }
            }
        }
        *flag_ok = ok;
    }
    cta_sync(consumers_only);
    return *flag_ok != 0;
}

__device__ __forceinline__ void stamp(unsigned long long *times, bool on, int i) {
    if (on && threadIdx.x == 0) times[blockIdx.x * kStampsPerCta + i] = globaltimer();
}

struct DecodeArgs {
    TMaps tm;  // first: 64-byte aligned members
    StepArgs a;
    Workspace ws;
    DecodeLayout L;
};

// routing facts a tile's reduction needs: expert, token mask, first slot
__device__ __forceinline__ int4 tile_route(const Smem &S, int u) {
    const int e = S.s_unique[u];
    return make_int4(e, (int)(unsigned)S.s_mask[e], S.s_off[e], 0);
}

// D-tile `dt` of a CTA's D rows [b0, b0 + 2 pp) (pp row pairs, ndt tiles):
// first row and height (both even)
__device__ __forceinline__ void d_tile(int b0, int pp, int ndt, int dt, int &start, int &h) {
    const int s0 = pp * dt / ndt, s1 = pp * (dt + 1) / ndt;
    start = b0 + 2 * s0;
    h = 2 * (s1 - s0);
}

__device__ __forceinline__ uint32_t lds32(const unsigned char *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// order-preserving map of f32 to u32 (larger float -> larger key; NaN lowest)
__device__ __forceinline__ uint32_t f2key(float f) {
    const uint32_t u = __float_as_uint(f);
    if (f != f) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Top-k of one token's logits (warp-wide; lane l holds experts l + 32 i, i < NPL,
// E <= 32 NPL): the k largest in descending order, ties to the lower expert id,
// and their renormalised softmax weights. The softmax denominator over all
// experts cancels in the renormalisation, so only the k selected logits are
// exponentiated.
// The logits come from the CTAs that own each expert, as 64-bit words (launch
// tag << 32 | f32 bits): the warp polls each word until it carries this
// launch's tag, so the exchange needs no grid barrier (bounded wait; on a
// timeout the flag is set and the result is garbage).
// Each lane then sorts its NPL (key, i) pairs (descending key, ascending i);
// every round takes the warp maximum of the lanes' heads, the lowest expert id
// among the lanes holding it, and the winning lane drops its head.
template <int NPL>
__device__ __forceinline__ void warp_topk_tagged(const unsigned long long *lt, uint32_t tag, int E, int k,
                                                 int lane, int *idx_out, float *w_out,
                                                 volatile int *abort_flag, unsigned *status) {
    uint32_t key[NPL], ix[NPL];
    unsigned need = 0;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        key[i] = 0u;
        ix[i] = (uint32_t)i;
        if (lane + 32 * i < E) need |= 1u << i;
    }
    const unsigned long long t0 = globaltimer();
    for (;;) {
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            if ((need >> i) & 1u) {
                const unsigned long long v = ptx::ld_relaxed_gpu_u64(lt + lane + 32 * i);
                if ((uint32_t)(v >> 32) == tag) {
                    key[i] = f2key(__uint_as_float((uint32_t)v));
                    need &= ~(1u << i);
                }
            }
        }
        if (__all_sync(0xffffffffu, need == 0u)) break;
        if (*abort_flag || globaltimer() - t0 > kWaitNs) {
            if (lane == 0) set_timeout(abort_flag, status);
            break;
        }
        // back off: every CTA's token warps poll at once, and a tight loop of
        // L2 loads slows the CTAs still writing their logits
        __nanosleep(200);
    }
    auto cx = [&](int a, int b) {
        const bool sw = key[b] > key[a] || (key[b] == key[a] && ix[b] < ix[a]);
        const uint32_t ka = key[a], ia = ix[a];
        key[a] = sw ? key[b] : ka;
        ix[a] = sw ? ix[b] : ia;
        key[b] = sw ? ka : key[b];
        ix[b] = sw ? ia : ix[b];
    };
    if (NPL == 8) {
        // Batcher's odd-even merge sort of 8 elements (19 compare-exchanges)
        cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
        cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
        cx(1, 2); cx(5, 6);
        cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
        cx(2, 4); cx(3, 5);
        cx(1, 2); cx(3, 4); cx(5, 6);
    } else {
        // 4 elements (5 compare-exchanges)
        cx(0, 1); cx(2, 3);
        cx(0, 2); cx(1, 3);
        cx(1, 2);
    }
    float lsel = 0.f, lmax = 0.f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        const uint32_t wk = __reduce_max_sync(0xffffffffu, key[0]);
        // a popped-out slot has i = NPL: its id lane + 32 NPL loses every tie
        const uint32_t ce = key[0] == wk ? (uint32_t)lane + 32u * ix[0] : 0xFFFFFFFFu;
        const uint32_t e = __reduce_min_sync(0xffffffffu, ce);
        if ((int)(e & 31u) == lane) {
#pragma unroll
            for (int i = 0; i < NPL - 1; ++i) {
                key[i] = key[i + 1];
                ix[i] = ix[i + 1];
            }
            key[NPL - 1] = 0u;
            ix[NPL - 1] = (uint32_t)NPL;
        }
        const float l = key2f(wk);
        if (j == 0) lmax = l;
        if (lane == j) {
            lsel = l;
            idx_out[j] = (int)e;
        }
    }
    const float ev = lane < k ? expf(lsel - lmax) : 0.f;
    const float z = warp_sum(ev);
    if (lane < k) w_out[lane] = ev / z;
}

// NKC: gate/up K chunks per tile (1 for D <= 2048, 2 for D <= 4096)
template <int NKC>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ DecodeArgs P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned start, as an offset into smem_raw (accesses stay shared-memory accesses)
    unsigned char *sbase = smem_raw + ((1024u - (ptx::smem_addr(smem_raw) & 1023u)) & 1023u);
    const DecodeLayout &L = P.L;
    const StepArgs &A = P.a;
    const Workspace &W = P.ws;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = A.s.E, K = A.s.k, D = A.s.D, F = A.s.F, n = A.s.n;
    const int GD = D / kGroup, GF = F / kGroup;
    const unsigned G = gridDim.x;
    const int cta = blockIdx.x;
    Smem S = carve_smem(sbase, L, E);
    volatile int *abort_flag = S.misc + 0;
    volatile int *bar_ok = S.misc + 1;
    const bool timing = (A.s.flags & MOE_FLAG_PHASE_TIMES) != 0;
    unsigned long long *gsync = reinterpret_cast<unsigned long long *>(W.sync);
    uint16_t *Hg = reinterpret_cast<uint16_t *>(W.h);  // [slots][F] f16, h_pos order

    // Prologue on shared memory and kernel parameters only: it may overlap the
    // tail of the previous kernel in the stream (programmatic dependent launch).
    unsigned long long epoch = 0;
    if (tid == 0) {
        for (int s = 0; s < L.NS; ++s) {
            ptx::mbar_init(&S.full[s], 1);
            ptx::mbar_init(&S.empty[s], kCW);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&S.pfull[b], kCW);
            ptx::mbar_init(&S.pempty[b], 1);
        }
        for (int i = 0; i < 32; ++i) S.misc[i] = 0;
        for (int t = 0; t < 2 * kNFast; ++t) reinterpret_cast<float *>(S.misc + 40)[t] = 1.0f;
        ptx::mbar_fence_init();
    }
    if (tid == 32) {
        const CUtensorMap *maps[] = {&P.tm.gq, &P.tm.uq, &P.tm.gs, &P.tm.gb, &P.tm.us, &P.tm.ub,
                                     &P.tm.dq[0], &P.tm.dq[1]};
        for (const CUtensorMap *m : maps) ptx::prefetch_tensormap(m);
    }
    // zero the expert token masks (grouping below)
#pragma unroll 1
    for (int e = tid; e < E; e += kThreads) S.s_mask[e] = 0ull;
    // the next kernel may start its own prologue as this grid's CTAs exit; every
    // global memory access below waits for the previous kernel to complete
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    stamp(W.phase_ns, timing, 0);
    // barrier epoch (thread 0 only): the counter grows by G per launch and no
    // CTA of this launch can pass barrier 2 before this CTA arrives there. The
    // launch tag of the logit exchange is the previous launch's plus one; CTA 0
    // stores it back only once every CTA has arrived at barrier 2, after all
    // of them have read it here.
    // Both loads are issued here and consumed later (the tag just before phase
    // R's CTA barrier, the epoch at barrier 2), so their latency overlaps the
    // router loads; the previous launch's writes are visible after
    // griddepcontrol.wait.
    unsigned prev_tag = 0;
    if (tid == 0) {
        epoch = *reinterpret_cast<volatile unsigned long long *>(gsync);
        prev_tag = *reinterpret_cast<volatile unsigned *>(W.sync + 32);
    }
    __syncthreads();

    // ---- phase R: router logits of this CTA's experts, x staging ----------------
    // Thread (token group tg, chunk ch) handles the 8-input chunk ch of tokens
    // tg, tg + TG, ... : it stages x in shared memory (f16, B-operand order) with
    // the chunk's sums, and dots the chunk with this CTA's router rows. A warp's
    // 32 threads share the token, so the per-token sums over chunks are warp
    // sums, combined over the chunk-warps in a fixed order.
    // f16 range: a chunk whose largest |x| is at least 2^15, or non-zero below
    // 2^-4, marks the step; the tokens are then staged again scaled by 2^-e
    // (e = ilogb(max |x_t|) - 2, exact: max |x_t| 2^-e in [4, 8)). The reducers
    // multiply the token's gate and up sums by 2^e. A token scaled up (e < 0)
    // has h shrinking as x^2 for the unclamped activations: its h is stored
    // times 2^-2e and its output multiplied by 2^2e, so h keeps f16's
    // precision. An h beyond f16's range saturates and is reported. N(0,1)-like
    // activations never take that path (a chunk of 8 all below 2^-4 has
    // probability below 1e-10).
    {
        const int nE = (cta < E ? 1 : 0) + (cta + (int)G < E ? 1 : 0);
        const int chunks = D >> 3;                  // a multiple of 32, at most kThreads
        const int NW = chunks >> 5;                 // chunk-warps per token
        const int TG = min(kThreads / chunks, kNFast);
        float *rs = S.red;                          // [token][router row][chunk-warp]
        float *xscale = reinterpret_cast<float *>(S.misc + 40);
        float *hscale = reinterpret_cast<float *>(S.misc + 48);
        // x -> f16 in B-operand order (pairs (0,4) (1,5) (2,6) (3,7)), odd inputs
        // divided by 16 (see mma_word_f16), times `inv`; the group's sums of x
        // and of x / m as the MMA sees them. Called by whole warps (one token).
        auto stage_chunk = [&](int t, int ch, const float (&xv)[8], float inv) {
            uint16_t b[8];
            float sm = 0.f, smd = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const __half hv = __float2half_rn((j & 1) ? xv[j] * inv * 0.0625f : xv[j] * inv);
                b[j] = __half_as_ushort(hv);
                const float f = __half2float(hv);
                smd += f;
                sm += (j & 1) ? f * 16.f : f;
            }
            uint4 o;
            o.x = (uint32_t)b[0] | ((uint32_t)b[4] << 16);
            o.y = (uint32_t)b[1] | ((uint32_t)b[5] << 16);
            o.z = (uint32_t)b[2] | ((uint32_t)b[6] << 16);
            o.w = (uint32_t)b[3] | ((uint32_t)b[7] << 16);
            *reinterpret_cast<uint4 *>(S.xs + (size_t)t * L.x_stride + (size_t)ch * 16) = o;
            // group sums: the 8 chunks of a group are 8 consecutive threads
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                sm += __shfl_xor_sync(0xffffffffu, sm, off);
                smd += __shfl_xor_sync(0xffffffffu, smd, off);
            }
            if ((lane & 7) == 0) *reinterpret_cast<float2 *>(S.xsum + ((ch >> 3) * kNFast + t) * 2) = make_float2(sm, smd);
        };
        if (tid < TG * chunks) {
            const int tg = tid / chunks, ch = tid - tg * chunks;
            float w0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, w1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (nE > 0) load8f(A.router_w, (size_t)cta * D + (size_t)ch * 8, A.s.w_dtype, w0);
            if (nE > 1) load8f(A.router_w, (size_t)(cta + (int)G) * D + (size_t)ch * 8, A.s.w_dtype, w1);
#pragma unroll 1
            for (int t = tg; t < n; t += TG) {
                float xv[8];
                load8f(A.x, (size_t)t * D + (size_t)ch * 8, A.s.x_dtype, xv);
                float d0 = 0.f, d1 = 0.f, am = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    d0 = fmaf(xv[j], w0[j], d0);
                    d1 = fmaf(xv[j], w1[j], d1);
                    am = fmaxf(am, fabsf(xv[j]));
                }
                if (am >= 32768.0f || (am > 0.0f && am < 0.0625f)) S.misc[7] = 1;
                stage_chunk(t, ch, xv, 1.0f);
                if (nE > 0) {
                    d0 = warp_sum(d0);
                    d1 = warp_sum(d1);
                    if (lane == 0) {
                        rs[(t * 2 + 0) * NW + (ch >> 5)] = d0;
                        rs[(t * 2 + 1) * NW + (ch >> 5)] = d1;
                    }
                }
            }
        }
        // rows of tokens n..7 are zero (the MMA reads all eight token columns)
#pragma unroll 1
        for (int i = tid; i < (kNFast - n) * chunks; i += kThreads) {
            const int t = n + i / chunks, ch = i - (t - n) * chunks;
            *reinterpret_cast<uint4 *>(S.xs + (size_t)t * L.x_stride + (size_t)ch * 16) = make_uint4(0, 0, 0, 0);
            if ((ch & 7) == 0) *reinterpret_cast<float2 *>(S.xsum + ((ch >> 3) * kNFast + t) * 2) = make_float2(0.f, 0.f);
        }
        if (tid == 0) S.misc[56] = (int)(prev_tag + 1u);  // this launch's tag
        __syncthreads();
        if (S.misc[7]) {
            // per-token scales: warp t finds max |x_t|
            if (warp < n) {
                float am = 0.f;
#pragma unroll 1
                for (int ch = lane; ch < chunks; ch += 32) {
                    float xv[8];
                    load8f(A.x, (size_t)warp * D + (size_t)ch * 8, A.s.x_dtype, xv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(xv[j]));
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
                if (lane == 0) {
                    const int e = (am > 0.0f && am <= 3.0e38f) ? min(max(ilogbf(am) - 2, -60), 60) : 0;
                    xscale[warp] = ldexpf(1.0f, e);
                    // h of a token scaled up shrinks as x^2 (the clamp bounds h
                    // from above only, which a small token never reaches)
                    hscale[warp] = e < 0 ? ldexpf(1.0f, 2 * e) : 1.0f;
                }
            }
            __syncthreads();
            if (tid < TG * chunks) {
                const int tg = tid / chunks, ch = tid - tg * chunks;
#pragma unroll 1
                for (int t = tg; t < n; t += TG) {
                    float xv[8];
                    load8f(A.x, (size_t)t * D + (size_t)ch * 8, A.s.x_dtype, xv);
                    stage_chunk(t, ch, xv, 1.0f / xscale[t]);
                }
            }
            __syncthreads();
        }
        if ((A.s.flags & MOE_FLAG_TEST_STALL) && cta == 0) {
            // test hook: CTA 0 publishes its logits late, only once another CTA's
            // bounded wait for them has given up (or after 2 s), so the others
            // time out while every CTA still arrives at barrier 2
            if (tid == 0) {
                const unsigned long long t0 = globaltimer();
                while (!(*reinterpret_cast<volatile unsigned *>(W.status) & kDevErrTimeout) &&
                       globaltimer() - t0 < 2 * kWaitNs) {
                }
            }
            __syncthreads();
        }
        const uint32_t tag = (uint32_t)S.misc[56];
        if (tid < nE * n) {
            const int ei = tid / n, t = tid - ei * n;
            float l = 0.f;
#pragma unroll 1
            for (int w = 0; w < NW; ++w) l += rs[(t * 2 + ei) * NW + w];
            const int e = cta + ei * (int)G;
            if (A.router_bias) l += A.router_bias[e];
            W.logits[(size_t)t * E + e] = l;  // for the grouping kernel of chunked cohorts
            ptx::st_relaxed_gpu_u64(W.tlog + (size_t)t * kTagSlots + e,
                                    ((unsigned long long)tag << 32) | __float_as_uint(l));
        }
    }

    const uint32_t tag = (uint32_t)S.misc[56];
    // ---- no grid barrier: phase T polls the tagged logits ------------------------
    stamp(W.phase_ns, timing, 1);
    if (tid == 0) epoch = epoch / G * G;
    stamp(W.phase_ns, timing, 2);

    // ---- phase T: routing and grouping, redundantly in every CTA ---------------
    // Warp 0 first waits for token 0's row: one polling warp per CTA keeps the
    // L2 traffic on these few lines low while the slowest CTAs still write. The
    // rows of the other tokens come from the same CTAs at the same time, so
    // their warps then usually read them once (and poll only on a mismatch).
    if (n > 1) {
        if (warp == 0) {
            const unsigned long long *lt = W.tlog;
            const unsigned long long t0 = globaltimer();
            unsigned need = 0;
#pragma unroll 1
            for (int e = lane; e < E; e += 32) need |= 1u << (e >> 5);
            while (!__all_sync(0xffffffffu, need == 0u)) {
#pragma unroll 1
                for (int i = 0; i < 8; ++i)
                    if (((need >> i) & 1u) && (uint32_t)(ptx::ld_relaxed_gpu_u64(lt + lane + 32 * i) >> 32) == tag)
                        need &= ~(1u << i);
                if (__all_sync(0xffffffffu, need == 0u) || *abort_flag || globaltimer() - t0 > kWaitNs) break;
                __nanosleep(200);
            }
            // gave up: report it now, so the token warps below stop at once
            // instead of spending a second bound of their own
            if (!__all_sync(0xffffffffu, need == 0u) && lane == 0 && !*abort_flag) set_timeout(abort_flag, W.status);
        }
        __syncthreads();
    }
    if (warp < n) {
        const unsigned long long *lt = W.tlog + (size_t)warp * kTagSlots;
        if (E <= 128)
            warp_topk_tagged<4>(lt, tag, E, K, lane, S.s_idx + warp * K, S.s_w + warp * K, abort_flag, W.status);
        else
            warp_topk_tagged<8>(lt, tag, E, K, lane, S.s_idx + warp * K, S.s_w + warp * K, abort_flag, W.status);
    }
    __syncthreads();
    const int Sl = n * K;
    // Grouping, slot table and tile list by warp 0 alone (no CTA barrier in
    // between; __syncwarp orders the warp's shared-memory accesses).
    // only the experts this plan owns ([e_lo, e_hi), all by default) are
    // grouped, streamed and summed
    const int e_lo = A.s.e_lo, e_hi = A.s.e_hi;
    if (warp == 0) {
#pragma unroll 1
        for (int i = lane; i < Sl; i += 32) {
            const int e = S.s_idx[i];
            if (e >= e_lo && e < e_hi) ptx::red_or_shared(S.s_mask + e, 1u << (i / K));
        }
        __syncwarp();
        // counts and exclusive scans over the experts; lane l owns experts
        // [8 l, 8 l + 8) (E <= 256), so the scans run in expert order
        int cnt8[8], csum = 0, usum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            cnt8[j] = e < E ? __popc((unsigned)S.s_mask[e]) : 0;
            csum += cnt8[j];
            usum += cnt8[j] > 0 ? 1 : 0;
        }
        int cinc = csum, uinc = usum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, cinc, o);
            const int w = __shfl_up_sync(0xffffffffu, uinc, o);
            if (lane >= o) {
                cinc += v;
                uinc += w;
            }
        }
        int cb = cinc - csum, ubs = uinc - usum;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            if (e < E) {
                S.s_off[e] = cb;
                S.s_counts[e] = cnt8[j];
                if (cnt8[j] > 0) S.s_unique[ubs++] = e;
                cb += cnt8[j];
            }
        }
        const int U0 = __shfl_sync(0xffffffffu, uinc, 31);
        if (lane == 31) {
            S.s_off[E] = cinc;
            S.misc[2] = uinc;
        }
        __syncwarp();
#pragma unroll 1
        for (int u = lane; u < U0; u += 32) S.uroute[u] = tile_route(S, u);
#pragma unroll 1
        for (int i = lane; i < Sl; i += 32) {
            const int t = i / K, e = S.s_idx[i];
            if (e < e_lo || e >= e_hi) continue;
            const unsigned m = (unsigned)S.s_mask[e];
            S.slot_w[S.s_off[e] + __popc(m & ((1u << t) - 1u))] = S.s_w[i];
        }
        __syncwarp();
    }
    // gate/up tile list: the U*F rows of the selected experts in 16-row blocks
    // (Dff is a multiple of 16, so no block straddles two experts), split evenly
    // over the CTAs by whole blocks: every tile is a full 16 rows, and no CTA
    // takes more than one block above the mean
    if (warp == 0) {
        const int U0 = S.misc[2];  // written by lane 31 before the __syncwarp above
        const unsigned NB = (unsigned)U0 * (unsigned)(F / 16);
        const int B0 = (int)(NB * (unsigned)cta / G), B1 = (int)(NB * (unsigned)(cta + 1) / G);
        int tb = B1 - B0;
#pragma unroll 1
        for (int b = lane; b < min(tb, L.max_tiles); b += 32) {
            const int r = 16 * (B0 + b), u = r / F;
            S.tiles[2 * b] = make_int4(u, r - u * F, 0, 16);
            S.tiles[2 * b + 1] = S.uroute[u];
        }
        if (lane == 0) {
            if (tb > L.max_tiles) {
                report_error(W.status, kDevErrInternal);  // the host bounds the count
                tb = L.max_tiles;
            }
            S.misc[3] = tb;
            // D rows of this CTA, in row pairs (even bounds)
            S.misc[4] = 2 * (int)((unsigned)(D / 2) * (unsigned)cta / G);
            S.misc[5] = 2 * (int)((unsigned)(D / 2) * (unsigned)(cta + 1) / G);
        }
    }
    __syncthreads();
    stamp(W.phase_ns, timing, 3);

    const int U = S.misc[2];
    const int nTiles = S.misc[3];
    const int b0 = S.misc[4], rowsB = S.misc[5] - S.misc[4];
    const int pp = rowsB / 2;                    // row pairs
    const int ndt = (pp + 6) / 7;                // D-tiles of at most 14 rows (0, 1 or 2)
    const int dsh = ndt > 1 ? 1 : 0;             // unit -> (expert index, D-tile) shift
    int ds0 = b0, h0 = 0, ds1 = b0, h1 = 0;
    if (ndt > 0) d_tile(b0, pp, ndt, 0, ds0, h0);
    if (ndt > 1) d_tile(b0, pp, ndt, 1, ds1, h1);
    const int nU = U * ndt;                      // down units of this CTA
    const int tsh = NKC > 1 ? 1 : 0;             // gate/up stage -> (tile, K chunk) shift
    const int nA = nTiles * NKC;                 // gate/up stages
    const int nB = (nU + L.P - 1) / L.P;         // down stages
    const int total = nA + nB;

    // ---- ring stages: issuing and release ----------------------------------------
    // Stage st (gate/up tiles first, then down units) goes to ring slot st % NS.
    // The first NS stages are issued here; after that the last warp to release a
    // stage issues the stage NS further on into the freed slot. Called by a whole warp.
    const uint64_t pol = ptx::policy_evict_first();
    auto issue_stage = [&](int st) {
        const int slot = st % L.NS;
        unsigned char *buf = S.ring + (size_t)slot * L.stage_bytes;
        uint64_t *bar = &S.full[slot];
        if (st < nA) {
            if (lane == 0) {
                const int4 tl = S.tiles[2 * (st >> tsh)];
                const int kc = st & tsh;
                const int row0 = S.s_unique[tl.x] * F + tl.y;  // first row of the box (even)
                ptx::mbar_arrive_expect_tx(bar, 2u * L.KS * 16u * 128u + 4u * 16u * L.sc_w);
                ptx::tma_load_3d(buf, &P.tm.gq, 0, row0, kc * L.KS, bar, pol);
                ptx::tma_load_3d(buf + L.off_up, &P.tm.uq, 0, row0, kc * L.KS, bar, pol);
                const int gx = kc * L.GDc, py = row0 >> 1;
                ptx::tma_load_3d(buf + L.off_sc, &P.tm.gs, gx, py, 0, bar, pol);
                ptx::tma_load_3d(buf + L.off_sc + 1024, &P.tm.gb, gx, py, 0, bar, pol);
                ptx::tma_load_3d(buf + L.off_sc + 2048, &P.tm.us, gx, py, 0, bar, pol);
                ptx::tma_load_3d(buf + L.off_sc + 3072, &P.tm.ub, gx, py, 0, bar, pol);
            }
        } else {
            const int jb = (st - nA) * L.P;
            const int nu = min(L.P, nU - jb);
            if (lane == 0) {
                uint32_t bytes = 0;
#pragma unroll 1
                for (int j = 0; j < nu; ++j)
                    bytes += (uint32_t)(((jb + j) & dsh) ? h1 : h0) *
                             (uint32_t)(L.sl_d * L.kw_d * 4 + 2 * L.rb_d);
                ptx::mbar_arrive_expect_tx(bar, bytes);
            }
            __syncwarp();
            if (lane < nu) {
                const int unit = jb + lane;
                const int e = S.s_unique[unit >> dsh];
                const int dt = unit & dsh;
                const int ds = dt ? ds1 : ds0, h = dt ? h1 : h0;
                const int hi = h == L.Hd[0] ? 0 : 1;
                unsigned char *ub = buf + (size_t)lane * L.unit_bytes;
                const int row = e * D + ds;  // even
                ptx::tma_load_3d(ub, &P.tm.dq[hi], 0, row, 0, bar, pol);
                if (L.dmode) {
                    ptx::tma_load_3d(ub + L.unit_sc, &P.tm.ds[hi], 0, row >> 1, 0, bar, pol);
                    ptx::tma_load_3d(ub + L.unit_sc + L.unit_sc_stride, &P.tm.db[hi], 0, row >> 1, 0, bar, pol);
                } else {
                    const size_t off = (size_t)row * L.rb_d;  // 16-byte aligned: even row, rb_d = 8 mod 16
                    const uint32_t nb = (uint32_t)h * L.rb_d;
                    ptx::bulk_g2s(ub + L.unit_sc, reinterpret_cast<const unsigned char *>(A.planes.down_s) + off,
                                  nb, bar, pol);
                    ptx::bulk_g2s(ub + L.unit_sc + L.unit_sc_stride,
                                  reinterpret_cast<const unsigned char *>(A.planes.down_b) + off, nb, bar, pol);
                }
            }
        }
    };
    if (warp >= kCW) {
        // the fifth warpgroup hands most of its registers to the consumers; its
        // first warp streams every stage into the ring as slots are released, the
        // next two reduce the consumers' gate/up partials
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
        if (warp >= kReducer0 + 2) {
            if (warp == kReducer0 + 2 && lane == 0 && A.next_router_w) {
                // the next layer of a chain routes right after this step: bring
                // the router rows its CTA c will read (experts c and c + G) and
                // the bias into L2 while this step streams its experts
                const size_t rb = (size_t)D * (A.s.w_dtype == MOE_DTYPE_F32 ? 4 : 2);
                const unsigned char *nr = static_cast<const unsigned char *>(A.next_router_w);
                if (cta < E) ptx::prefetch_l2_bulk(nr + (size_t)cta * rb, (uint32_t)rb);
                if (cta + (int)G < E) ptx::prefetch_l2_bulk(nr + (size_t)(cta + (int)G) * rb, (uint32_t)rb);
                if (cta == 0 && A.next_router_bias && ((uintptr_t)A.next_router_bias & 15u) == 0 && (E & 3) == 0)
                    ptx::prefetch_l2_bulk(A.next_router_bias, (uint32_t)(E * 4));
            }
            if (warp == kReducer0 + 2 && cta == 0) {
                // the routing tables the host may read back (CTA 0's copy)
#pragma unroll 1
                for (int i = lane; i < n * K; i += 32) {
                    const int t = i / K, e = S.s_idx[i];
                    W.topk_idx[i] = e;
                    W.topk_w[i] = S.s_w[i];
                    if (e < A.s.e_lo || e >= A.s.e_hi) {
                        W.slot_of[i] = -1;  // an expert this plan does not own
                        continue;
                    }
                    const unsigned m = (unsigned)S.s_mask[e];
                    const int p = S.s_off[e] + __popc(m & ((1u << t) - 1u));
                    W.slot_token[p] = t;
                    W.slot_k[p] = i - t * K;
                    W.slot_of[i] = p;
                }
#pragma unroll 1
                for (int e = lane; e < E; e += 32) {
                    W.counts[e] = S.s_counts[e];
                    W.offsets[e] = S.s_off[e];
                    W.unique[e] = e < U ? S.s_unique[e] : -1;
                }
                if (lane == 0) {
                    W.offsets[E] = S.s_off[E];
                    *W.U = U;
                }
            }
            return;
        }
        if (warp != kProducer) {
            // Reducer of partial buffer b = warp - kReducer0, i.e. of tiles b, b + 2, ...
            // Lane l sums fragment lane l's four (row, token) values of the 16
            // consumer warps in warp order, frees the buffer, then writes
            // h = w * act(g, u) as f16 for the valid (row, token) pairs.
            const int b = warp - kReducer0;
            for (int t = b, r = 0; t < nTiles; t += 2, ++r) {
                if (!__shfl_sync(0xffffffffu, (int)wait_phase_inl(&S.pfull[b], (uint32_t)(r & 1), abort_flag, W.status), 0))
                    break;
                const float *q = S.red + (size_t)b * kCW * kPartStride + lane * 4;
                float4 gs = *reinterpret_cast<const float4 *>(q);
                float4 us = *reinterpret_cast<const float4 *>(q + 128);
#pragma unroll
                for (int w = 1; w < kCW; ++w) {
                    const float4 a = *reinterpret_cast<const float4 *>(q + (size_t)w * kPartStride);
                    const float4 u = *reinterpret_cast<const float4 *>(q + (size_t)w * kPartStride + 128);
                    gs.x += a.x; gs.y += a.y; gs.z += a.z; gs.w += a.w;
                    us.x += u.x; us.y += u.y; us.z += u.z; us.w += u.w;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&S.pempty[b], 1);
                const int4 tl = S.tiles[2 * t], tr = S.tiles[2 * t + 1];
                const unsigned m = (unsigned)tr.y;
                bool over = false;
                const float gv[4] = {gs.x, gs.y, gs.z, gs.w}, uv[4] = {us.x, us.y, us.z, us.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = 2 * (lane >> 2) + (i >> 1), tok = 2 * (lane & 3) + (i & 1);
                    if (row >= tl.z && row < tl.w && ((m >> tok) & 1u)) {
                        const int pslot = tr.z + __popc(m & ((1u << tok) - 1u));
                        const float xsc = reinterpret_cast<const float *>(S.misc + 40)[tok];
                        const float hinv = 1.0f / reinterpret_cast<const float *>(S.misc + 48)[tok];
                        Hg[(size_t)pslot * F + h_pos(tl.y + row)] =
                            f2h_sat(S.slot_w[pslot] * glu_act<false>(A.s.act, A.s.act_limit, gv[i] * xsc, uv[i] * xsc) * hinv,
                                    over);
                    }
                }
                if (over) report_error(W.status, kDevErrRange);
            }
            // every h row of this CTA written: the consumers pass grid barrier 2 after this
            ptx::named_bar(2, kConsThreads + 64);
            return;
        }
        int issued = 0;
        for (int st = 0; st < total; ++st) {
            const int slot = st % L.NS, use = st / L.NS;
            int ok = 1;
            if (lane == 0 && use > 0) {
                ok = wait_phase_inl(&S.empty[slot], (use - 1) & 1, abort_flag, W.status);
                ptx::fence_proxy_async_shared();  // the consumers' reads before the refill's async writes
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            issue_stage(st);
            issued = st + 1;
        }
        if (lane == 0) {
            // drain: every issued copy must land before the CTA may exit
#pragma unroll 1
            for (int st = max(0, issued - L.NS); st < issued; ++st) {
                const unsigned long long t0 = globaltimer();
                while (!ptx::mbar_try_wait(&S.full[st % L.NS], (st / L.NS) & 1))
                    if (globaltimer() - t0 > kWaitNs) break;
            }
        }
        __syncwarp();
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsConsumer));
    // a consumer warp is done with a ring stage
    auto release_stage = [&](int slot) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.empty[slot], 1);
    };

    const int g = lane >> 2, c = lane & 3;
    const int r0 = 2 * g, r1 = 2 * g + 1;  // tile rows of MMA rows g and g + 8
    unsigned long long ta_wait = 0, ta_comp = 0, tb_wait = 0, tb_comp = 0;
    int slot = 0, par = 0;                 // ring position of the current stage

    // ---- phase A: gate/up ---------------------------------------------------------
    // A warp owns at most one pair of input groups per K chunk, the same pair in
    // every tile, so its x fragments and group sums stay in registers.
    const uint32_t X0 = (uint32_t)((c >> 1) ^ (r0 & 7)), X1 = (uint32_t)((c >> 1) ^ (r1 & 7));
    const uint32_t rb0 = (uint32_t)(r0 * 128 + (c & 1) * 8), rb1 = (uint32_t)(r1 * 128 + (c & 1) * 8);
    const uint32_t sco0 = (uint32_t)(g * L.sc_w), sco1 = (uint32_t)((8 + g) * L.sc_w);
    int pw[NKC];
    uint4 xf[NKC][2][2];
    float4 xsm[NKC][2];
#pragma unroll
    for (int kc = 0; kc < NKC; ++kc) {
        const int nP = min(L.GDc, GD - kc * L.GDc) >> 1;  // group pairs in K chunk kc
        const int pA = warp * nP / kCW, pB = (warp + 1) * nP / kCW;
        pw[kc] = pB > pA ? pA : -1;
        const int p0 = pB > pA ? pA : 0;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int gg = kc * L.GDc + 2 * p0 + h2;
            const unsigned char *xr = S.xs + (size_t)g * L.x_stride + (size_t)gg * 128 + c * 32;
            xf[kc][h2][0] = *reinterpret_cast<const uint4 *>(xr);
            xf[kc][h2][1] = *reinterpret_cast<const uint4 *>(xr + 16);
            const float2 s0 = *reinterpret_cast<const float2 *>(S.xsum + (gg * kNFast + 2 * c) * 2);
            const float2 s1 = *reinterpret_cast<const float2 *>(S.xsum + (gg * kNFast + 2 * c + 1) * 2);
            xsm[kc][h2] = make_float4(s0.x, s1.x, s0.y, s1.y);
        }
    }
    float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t_idx = 0; t_idx < nTiles; ++t_idx) {
#pragma unroll
        for (int kc = 0; kc < NKC; ++kc) {
            const unsigned long long tw0 = timing ? globaltimer() : 0ull;
            const bool ok = __shfl_sync(0xffffffffu, (int)wait_phase(&S.full[slot], par, abort_flag, W.status), 0) != 0;
            const unsigned long long tw1 = timing ? globaltimer() : 0ull;
            if (ok) {
                if (pw[kc] >= 0) {
                    const int p = pw[kc];
                    const unsigned char *gb = S.ring + (size_t)slot * L.stage_bytes;
                    const unsigned char *ubx = gb + L.off_up;
                    const unsigned char *sc = gb + L.off_sc;
                    uint32_t sw[8];  // (gate s, gate b, up s, up b) of rows 2g, 2g + 1 for the pair
                    {
                        const uint32_t a0 = swz(sco0 + 4u * p, (uint32_t)L.sc_m);
                        const uint32_t a1 = swz(sco1 + 4u * p, (uint32_t)L.sc_m);
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                            sw[a] = lds32(sc + a * 1024 + a0);
                            sw[4 + a] = lds32(sc + a * 1024 + a1);
                        }
                    }
                    const uint32_t kb = (uint32_t)(p >> 1) * 2048u;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const uint32_t gi2 = (uint32_t)(((p & 1) * 2 + h2) * 2);
                        const uint32_t o0 = kb + rb0 + ((gi2 ^ X0) << 4);
                        const uint32_t o1 = kb + rb1 + ((gi2 ^ X1) << 4);
                        const uint2 wg0 = *reinterpret_cast<const uint2 *>(gb + o0);
                        const uint2 wg1 = *reinterpret_cast<const uint2 *>(gb + o1);
                        const uint2 wu0 = *reinterpret_cast<const uint2 *>(ubx + o0);
                        const uint2 wu1 = *reinterpret_cast<const uint2 *>(ubx + o1);
                        float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_word_f16(cg, wg0.x, wg1.x, xf[kc][h2][0]);
                        mma_word_f16(cu, wu0.x, wu1.x, xf[kc][h2][0]);
                        mma_word_f16(cg, wg0.y, wg1.y, xf[kc][h2][1]);
                        mma_word_f16(cu, wu0.y, wu1.y, xf[kc][h2][1]);
                        const float4 xs4 = xsm[kc][h2];  // sum x, sum x/m of tokens 2c, 2c+1
                        const float gs0 = bf_half(sw[0], h2), gb0 = bf_half(sw[1], h2);
                        const float us0 = bf_half(sw[2], h2), ub0 = bf_half(sw[3], h2);
                        const float gs1 = bf_half(sw[4], h2), gb1 = bf_half(sw[5], h2);
                        const float us1 = bf_half(sw[6], h2), ub1 = bf_half(sw[7], h2);
                        // row contribution: s * (acc - 1024 * sum(x/m)) + b * sum(x)
                        const float ng0 = -1024.f * gs0, ng1 = -1024.f * gs1;
                        const float nu0 = -1024.f * us0, nu1 = -1024.f * us1;
                        tg[0] = fmaf(gs0, cg[0], fmaf(gb0, xs4.x, fmaf(ng0, xs4.z, tg[0])));
                        tg[1] = fmaf(gs0, cg[1], fmaf(gb0, xs4.y, fmaf(ng0, xs4.w, tg[1])));
                        tg[2] = fmaf(gs1, cg[2], fmaf(gb1, xs4.x, fmaf(ng1, xs4.z, tg[2])));
                        tg[3] = fmaf(gs1, cg[3], fmaf(gb1, xs4.y, fmaf(ng1, xs4.w, tg[3])));
                        tu[0] = fmaf(us0, cu[0], fmaf(ub0, xs4.x, fmaf(nu0, xs4.z, tu[0])));
                        tu[1] = fmaf(us0, cu[1], fmaf(ub0, xs4.y, fmaf(nu0, xs4.w, tu[1])));
                        tu[2] = fmaf(us1, cu[2], fmaf(ub1, xs4.x, fmaf(nu1, xs4.z, tu[2])));
                        tu[3] = fmaf(us1, cu[3], fmaf(ub1, xs4.y, fmaf(nu1, xs4.w, tu[3])));
                    }
                }
                // release the stage (after an abort the stage may still be in flight: keep it)
                release_stage(slot);
            }
            if (++slot == L.NS) {
                slot = 0;
                par ^= 1;
            }
            if (timing) {
                ta_wait += tw1 - tw0;
                ta_comp += globaltimer() - tw1;
            }
        }
        // tile done: this warp's partial [gate | up][lane][4] into buffer t & 1,
        // once its reducer has read tile t - 2 out of it
        {
            const int b = t_idx & 1, r = t_idx >> 1;
            if (r >= 1)
                __shfl_sync(0xffffffffu, (int)wait_phase(&S.pempty[b], (uint32_t)((r - 1) & 1), abort_flag, W.status), 0);
            float *pp4 = S.red + (size_t)(b * kCW + warp) * kPartStride + lane * 4;
            *reinterpret_cast<float4 *>(pp4) = make_float4(tg[0], tg[1], tg[2], tg[3]);
            *reinterpret_cast<float4 *>(pp4 + 128) = make_float4(tu[0], tu[1], tu[2], tu[3]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&S.pfull[b], 1);
#pragma unroll
            for (int i = 0; i < 4; ++i) tg[i] = tu[i] = 0.f;
        }
    }

    // ---- grid barrier 2: every h row written ----------------------------------
    stamp(W.phase_ns, timing, 4);
    ptx::named_bar(2, kConsThreads + 64);  // the reducers have written every h row of this CTA
    grid_barrier(gsync, epoch + G, bar_ok, abort_flag, W.status, true);
    // every CTA has read the launch tag (it arrived here): publish it for the
    // next launch (also after a timeout, so a later launch never reuses it)
    if (cta == 0 && tid == 0) W.sync[32] = tag;
    stamp(W.phase_ns, timing, 5);

    // ---- phase B: down, all experts summed per warp ----------------------------
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    // this warp's items of a down stage: item warp + 16 q is (unit j, group pair gp)
    const int GP = GF >> 1;
    int itj[kMaxDI], itg[kMaxDI];
#pragma unroll
    for (int q = 0; q < kMaxDI; ++q) {
        const int it = warp + q * kCW;
        itj[q] = it / GP;
        itg[q] = it - itj[q] * GP;
    }
    const int nItems = L.P * GP;
    // h of item q of down stage st (written by other CTAs before barrier 2), or 0:
    // token g's 32 bytes of each group of the pair
    auto load_h = [&](int st, int q, uint4 (&hv)[4]) {
        hv[0] = hv[1] = hv[2] = hv[3] = make_uint4(0, 0, 0, 0);
        if (st >= total) return;
        const int jb = (st - nA) * L.P;
        if (warp + q * kCW < nItems && itj[q] < nU - jb) {
            const int4 ur = S.uroute[(jb + itj[q]) >> dsh];
            const unsigned m = (unsigned)ur.y;
            if ((m >> g) & 1u) {
                const int ps = ur.z + __popc(m & ((1u << g) - 1u));
                const unsigned char *hp = reinterpret_cast<const unsigned char *>(Hg + (size_t)ps * F) +
                                          (size_t)itg[q] * 256 + c * 32;
                hv[0] = ptx::ld_cg_v4(hp);
                hv[1] = ptx::ld_cg_v4(hp + 16);
                hv[2] = ptx::ld_cg_v4(hp + 128);
                hv[3] = ptx::ld_cg_v4(hp + 144);
            }
        }
    };
    // scale/bias byte offsets of rows 2g and 2g + 1: [row parity][row pair][bytes]
    const uint32_t rs2 = L.dmode ? (uint32_t)L.rb_d : (uint32_t)(2 * L.rb_d);
    // shared-memory offsets of an item inside a unit of height h: codes of rows
    // 2g and 2g + 1 for the pair's two groups (16-byte chunks ch0 and ch0 + 2 of
    // the pair's 256-input slice), then the scale words of the two rows
    auto item_offsets = [&](int gp, int h, uint32_t (&o)[6]) {
        const int rowA = (gp >> 1) * h + r0, rowB = rowA + 1;
        const uint32_t ch0 = (uint32_t)(4 * (gp & 1) + (c >> 1));
        const uint32_t la = (uint32_t)(rowA * 128 + (c & 1) * 8), lb = (uint32_t)(rowB * 128 + (c & 1) * 8);
        const uint32_t xa = (uint32_t)(rowA & 7), xb = (uint32_t)(rowB & 7);
        o[0] = la + ((ch0 ^ xa) << 4);
        o[1] = la + (((ch0 + 2) ^ xa) << 4);
        o[2] = lb + ((ch0 ^ xb) << 4);
        o[3] = lb + (((ch0 + 2) ^ xb) << 4);
        const uint32_t ps = L.dmode ? (uint32_t)(h / 2 * L.rb_d) : (uint32_t)L.rb_d;
        const uint32_t cbo = (uint32_t)(gp * 4);
        o[4] = swz(g * rs2 + cbo, (uint32_t)L.sc_md);
        o[5] = swz(ps + g * rs2 + cbo, (uint32_t)L.sc_md);
    };
    // the same for every stage when the unit is D-tile 0 (the only one for D <= 2048)
    uint32_t io0[kMaxDI][6];
#pragma unroll
    for (int q = 0; q < kMaxDI; ++q) item_offsets(itg[q], h0, io0[q]);
    // h fragments of this warp's items, loaded one stage ahead
    uint4 hq[kMaxDI][4];
#pragma unroll
    for (int q = 0; q < kMaxDI; ++q) load_h(nA, q, hq[q]);
    for (int st = nA; st < total; ++st) {
        const int jb = (st - nA) * L.P;
        const int nu = min(L.P, nU - jb);
        const unsigned long long tw0 = timing ? globaltimer() : 0ull;
        const bool ok = __shfl_sync(0xffffffffu, (int)wait_phase(&S.full[slot], par, abort_flag, W.status), 0) != 0;
        const unsigned long long tw1 = timing ? globaltimer() : 0ull;
        const unsigned char *buf = S.ring + (size_t)slot * L.stage_bytes;
        if (ok) {
#pragma unroll
            for (int q = 0; q < kMaxDI; ++q) {
                if (warp + q * kCW < nItems && itj[q] < nu) {
                    const int j = itj[q];
                    const int dt = (jb + j) & dsh;
                    uint32_t o[6];
                    if (dt == 0) {
#pragma unroll
                        for (int i = 0; i < 6; ++i) o[i] = io0[q][i];
                    } else {
                        item_offsets(itg[q], h1, o);
                    }
                    const unsigned char *ubase = buf + (size_t)j * L.unit_bytes;
                    const uint2 wa0 = *reinterpret_cast<const uint2 *>(ubase + o[0]);
                    const uint2 wa1 = *reinterpret_cast<const uint2 *>(ubase + o[1]);
                    uint2 wb0 = *reinterpret_cast<const uint2 *>(ubase + o[2]);
                    uint2 wb1 = *reinterpret_cast<const uint2 *>(ubase + o[3]);
                    if (g == 7) wb0 = wb1 = make_uint2(0u, 0u);  // tile row 15: zero codes -> 1024 * sum(h)
                    float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_word(ca, wa0.x, wb0.x, hq[q][0]);
                    mma_word(cb, wa1.x, wb1.x, hq[q][2]);
                    mma_word(ca, wa0.y, wb0.y, hq[q][1]);
                    mma_word(cb, wa1.y, wb1.y, hq[q][3]);
                    const float ha0 = __shfl_sync(0xffffffffu, ca[2], 28 + c);
                    const float ha1 = __shfl_sync(0xffffffffu, ca[3], 28 + c);
                    const float hb0 = __shfl_sync(0xffffffffu, cb[2], 28 + c);
                    const float hb1 = __shfl_sync(0xffffffffu, cb[3], 28 + c);
                    // one 32-bit word holds the pair's two bf16 scales (or biases)
                    const uint32_t sa = o[4], sb = o[5];
                    const unsigned char *scs = ubase + L.unit_sc, *scb = scs + L.unit_sc_stride;
                    const uint32_t s0w = lds32(scs + sa), s1w = lds32(scs + sb);
                    const uint32_t b0w = lds32(scb + sa), b1w = lds32(scb + sb);
                    float v[4];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float *cd = hh ? cb : ca;
                        const float hs0 = hh ? hb0 : ha0, hs1 = hh ? hb1 : ha1;
                        const float s0 = bf_half(s0w, hh), s1 = bf_half(s1w, hh);
                        const float o0 = fmaf(-1024.f, s0, bf_half(b0w, hh)) * 0.0009765625f;
                        const float o1 = fmaf(-1024.f, s1, bf_half(b1w, hh)) * 0.0009765625f;
                        if (hh == 0) {
                            v[0] = fmaf(s0, cd[0], o0 * hs0);
                            v[1] = fmaf(s0, cd[1], o0 * hs1);
                            v[2] = fmaf(s1, cd[2], o1 * hs0);
                            v[3] = fmaf(s1, cd[3], o1 * hs1);
                        } else {
                            v[0] += fmaf(s0, cd[0], o0 * hs0);
                            v[1] += fmaf(s0, cd[1], o0 * hs1);
                            v[2] += fmaf(s1, cd[2], o1 * hs0);
                            v[3] += fmaf(s1, cd[3], o1 * hs1);
                        }
                    }
                    if (dt == 0) {
                        acc0[0] += v[0]; acc0[1] += v[1]; acc0[2] += v[2]; acc0[3] += v[3];
                    } else {
                        acc1[0] += v[0]; acc1[1] += v[1]; acc1[2] += v[2]; acc1[3] += v[3];
                    }
                }
                load_h(st + 1, q, hq[q]);
            }
            release_stage(slot);
        }
        if (++slot == L.NS) {
            slot = 0;
            par ^= 1;
        }
        if (timing) {
            tb_wait += tw1 - tw0;
            tb_comp += globaltimer() - tw1;
        }
    }
    if (timing && tid == 0) {
        unsigned long long *tt = W.phase_ns + cta * kStampsPerCta;
        tt[8] = ta_wait;
        tt[9] = ta_comp;
        tt[10] = tb_wait;
        tt[11] = tb_comp;
        tt[13] = (unsigned long long)nA;
        tt[14] = (unsigned long long)(total - nA);
    }

    // ---- final: fixed-order sum over warps of their partial outputs -------------
    {
        float *red = S.red + ((size_t)warp * 32 + lane) * 8;
        *reinterpret_cast<float4 *>(red) = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
        *reinterpret_cast<float4 *>(red + 4) = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
    }
    cta_sync(true);
    stamp(W.phase_ns, timing, 6);
#pragma unroll 1
    for (int o = tid; o < n * rowsB; o += kConsThreads) {
        const int t = o / rowsB, r = o - t * rowsB;
        const int dt = (ndt > 1 && b0 + r >= ds1) ? 1 : 0;
        const int rt = b0 + r - (dt ? ds1 : ds0);
        const int ln = (rt >> 1) * 4 + (t >> 1), idx = dt * 4 + (rt & 1) * 2 + (t & 1);
        float v = 0.f;
        for (int w = 0; w < kCW; ++w) v += S.red[((size_t)w * 32 + ln) * 8 + idx];
        v *= reinterpret_cast<const float *>(S.misc + 48)[t];  // 1 unless token t was scaled
        const size_t at = (size_t)t * D + b0 + r;
        if (A.s.out_dtype == MOE_DTYPE_F32)
            static_cast<float *>(A.out)[at] = v;
        else
            static_cast<uint16_t *>(A.out)[at] = f2bf(v);
    }
    if (timing) {
        cta_sync(true);
        stamp(W.phase_ns, timing, 7);
    }
}

}  // namespace

// ---- host side -----------------------------------------------------------------

static int round_up(int v, int m) { return (v + m - 1) / m * m; }

bool fused_layout(const moe_config &c, int num_sms, int max_smem, DecodeLayout *out) {
    DecodeLayout L{};
    const int D = c.D, F = c.Dff, E = c.E, k = c.top_k, G = num_sms;
    if (k * kNFast > kMaxSlotsF) return false;
    // gate/up: K-slices of 256 inputs; scale row pairs with 16-byte aligned strides
    if (D % 512 != 0) return false;
    if (F % 256 != 0) return false;  // down K-slices of 256 inputs
    if (E > 2 * G) return false;     // at most two router rows per CTA
    if (E > 256) return false;       // top-k holds 8 logits per lane
    if (D > 4096) return false;      // at most two K chunks per gate/up tile
    L.G = G;
    // gate/up stages
    L.KS = D / 256 < kStageSlices ? D / 256 : kStageSlices;
    L.NKC = (D / 256 + L.KS - 1) / L.KS;
    L.GDc = 4 * L.KS;
    L.off_up = L.KS * 16 * 128;
    L.off_sc = 2 * L.off_up;
    L.sc_w = 2 * L.GDc;  // 16, 32 or 64 bytes
    L.sc_m = L.sc_w == 64 ? 3 : L.sc_w == 32 ? 1 : 0;
    const int stage_a = L.off_sc + 4 * 1024;
    // down units: D-tile heights of every CTA (even, at most 14; two distinct values)
    int nh = 0;
    L.Hd[0] = L.Hd[1] = 0;
    for (int cta = 0; cta < G; ++cta) {
        const int p0 = (int)((long long)(D / 2) * cta / G), p1 = (int)((long long)(D / 2) * (cta + 1) / G);
        const int pairs = p1 - p0;
        if (pairs == 0) continue;
        const int ndt = (pairs + 6) / 7;
        if (ndt > 2) return false;
        for (int dt = 0; dt < ndt; ++dt) {
            const int h = 2 * (pairs * (dt + 1) / ndt - pairs * dt / ndt);
            if (h == L.Hd[0] || (nh > 1 && h == L.Hd[1])) continue;
            if (nh == 2) return false;
            L.Hd[nh++] = h;
        }
    }
    if (nh == 0) return false;
    if (nh == 1) L.Hd[1] = L.Hd[0];
    const int Hmax = L.Hd[0] > L.Hd[1] ? L.Hd[0] : L.Hd[1];
    L.kw_d = 32;
    L.sl_d = F / 256;
    L.swz_d = 7;
    // down scales: rows of rb_d bytes; rb_d = 8 mod 16 keeps the rows of a bulk
    // copy on distinct banks, 32/64/128 use row-pair boxes with swizzle
    L.rb_d = F / 32;
    if (L.rb_d % 16 == 8) {
        L.dmode = 0;
        L.sc_md = 0;
        L.unit_sc_stride = round_up(Hmax * L.rb_d, 16);
    } else if (L.rb_d == 32 || L.rb_d == 64 || L.rb_d == 128) {
        L.dmode = 1;
        L.sc_md = L.rb_d == 128 ? 7 : L.rb_d == 64 ? 3 : 1;
        L.unit_sc_stride = round_up(Hmax * L.rb_d, 1024);
    } else {
        return false;
    }
    L.unit_w = round_up(L.sl_d * Hmax * L.kw_d * 4, 1024);
    L.unit_sc = L.unit_w;
    L.unit_bytes = round_up(L.unit_w + 2 * L.unit_sc_stride, 1024);
    const int GF = F / kGroup;
    L.P = stage_a / L.unit_bytes;
    if (L.P < 1) L.P = 1;
    // items (unit, group pair) of a stage: at most kMaxDI per warp
    if (GF / 2 > kMaxDI * kCW) return false;
    while (L.P > 1 && L.P * (GF / 2) > kMaxDI * kCW) --L.P;
    if (L.P * (GF / 2) > kMaxDI * kCW) return false;
    L.stage_bytes = round_up(stage_a > L.P * L.unit_bytes ? stage_a : L.P * L.unit_bytes, 1024);
    // gate/up tiles per CTA: rows ceil(U*F/G) (+2 for even bounds) with U <= min(E, 8k)
    const int Umax = E < kNFast * k ? E : kNFast * k;
    const long long rows_cta = ((long long)Umax * F + G - 1) / G + 2;
    const long long tiles = 2 * ((rows_cta + 15) / 16);
    if (tiles > kMaxTilesF) return false;
    L.max_tiles = kMaxTilesF;
    L.x_stride = 2 * D + 16;
    int off = 0;
    L.off_bar = off;
    off += 256;
    L.off_misc = off;
    off += 256;
    L.off_route = off;
    off += round_up(8 * E + 4 * (6 * kMaxSlotsF + E + (E + 1) + E), 128);
    L.off_tiles = off;
    off += round_up(32 * kMaxTilesF + 16 * kMaxSlotsF, 128);
    L.off_x = off;
    off += round_up(kNFast * L.x_stride, 128);
    L.off_xsum = off;
    off += round_up(8 * kNFast * (D / kGroup), 128);
    L.off_red = off;
    off += 2 * kCW * kPartStride * 4;
    off = round_up(off, 1024);
    L.off_ring = off;
    const int tail = 2048 + 1024;  // over-read pad of the last stage + base alignment slack
    const int room = max_smem - off - tail;
    int ns = room / L.stage_bytes;
    if (ns > kMaxRing) ns = kMaxRing;
    if (ns < 2) return false;
    L.NS = ns;
    L.smem_bytes = off + ns * L.stage_bytes + tail;
    *out = L;
    return true;
}

static const void *kernel_for(const DecodeLayout &L) {
    return L.NKC == 1 ? (const void *)decode_step_kernel<1> : (const void *)decode_step_kernel<2>;
}

cudaError_t fused_prepare(const DecodeLayout &L, int *blocks_per_sm) {
    const void *k = kernel_for(L);
    // the register split inside the kernel hands exactly the launch's registers
    // (640 threads x 96) from the fifth warpgroup to the consumers; any other
    // per-thread count at launch would make the split wait forever, so such a
    // build is declined here
    cudaFuncAttributes fa{};
    cudaError_t err = cudaFuncGetAttributes(&fa, k);
    if (err != cudaSuccess) return err;
    if (fa.numRegs * kThreads != kRegsConsumer * kConsThreads + kRegsProducer * (kThreads - kConsThreads)) {
        *blocks_per_sm = 0;
        return cudaSuccess;
    }
    err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem_bytes);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kThreads, (size_t)L.smem_bytes);
}

int fused_max_tokens() { return kNFast; }

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    }
    return fn;
}

CUtensorMapSwizzle swizzle_for(int inner_bytes) {
    return inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : inner_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
         : inner_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
}

// 3-D view of a code plane [rows][words] as {inner words, rows, K-slices}: a box
// of {inner, box_rows, box_slices} lands in shared memory as
// [slice][row][inner * 4 bytes], swizzled
bool encode_codes(CUtensorMap *m, const void *base, int words_per_row, long long rows, int inner,
                  int box_rows, int box_slices) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)(words_per_row / inner)};
    cuuint64_t strides[2] = {(cuuint64_t)words_per_row * 4u, (cuuint64_t)inner * 4u};
    cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)box_rows, (cuuint32_t)box_slices};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(inner * 4), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a bf16 scale (or bias) array [rows][groups] as {groups, row pairs,
// parity}: a box of {box_groups, box_pairs, 2} lands in shared memory as
// [parity][row pair][box_groups * 2 bytes], swizzled, so rows 2i and 2i + 1 sit
// in separate halves
bool encode_scales(CUtensorMap *m, const void *base, int groups, long long rows, int box_groups,
                   int box_pairs) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)groups, (cuuint64_t)(rows / 2), 2};
    cuuint64_t strides[2] = {(cuuint64_t)groups * 4u, (cuuint64_t)groups * 2u};
    cuuint32_t box[3] = {(cuuint32_t)box_groups, (cuuint32_t)box_pairs, 2};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_groups * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fused_encode_tmaps(const moe_config &c, const DecodeLayout &L, const moe_expert_planes &planes,
                        TMaps *out) {
    const long long E = c.E, D = c.D, F = c.Dff;
    const int GD = (int)(D / kGroup), GF = (int)(F / kGroup);
    bool ok = encode_codes(&out->gq, planes.gate_q, (int)(D / 8), E * F, 32, 16, L.KS) &&
              encode_codes(&out->uq, planes.up_q, (int)(D / 8), E * F, 32, 16, L.KS) &&
              encode_scales(&out->gs, planes.gate_s, GD, E * F, L.GDc, 8) &&
              encode_scales(&out->gb, planes.gate_b, GD, E * F, L.GDc, 8) &&
              encode_scales(&out->us, planes.up_s, GD, E * F, L.GDc, 8) &&
              encode_scales(&out->ub, planes.up_b, GD, E * F, L.GDc, 8);
    for (int i = 0; i < 2 && ok; ++i) {
        ok = encode_codes(&out->dq[i], planes.down_q, (int)(F / 8), E * D, L.kw_d, L.Hd[i], L.sl_d);
        if (ok && L.dmode)
            ok = encode_scales(&out->ds[i], planes.down_s, GF, E * D, GF, L.Hd[i] / 2) &&
                 encode_scales(&out->db[i], planes.down_b, GF, E * D, GF, L.Hd[i] / 2);
    }
    return ok;
}

cudaError_t launch_fused(const StepArgs &a, const Workspace &ws, const DecodeLayout &L,
                         const TMaps &tm, cudaStream_t st, int &launched) {
    DecodeArgs P;
    P.tm = tm;
    P.a = a;
    P.ws = ws;
    P.L = L;
    void *args[] = {&P};
    // cooperative (every CTA resident at once, which the grid barriers need),
    // and with programmatic stream serialization: the launch may begin while
    // the previous kernel of the stream finishes; the kernel's prologue touches
    // shared memory only and then waits for that kernel (griddepcontrol.wait).
    // A driver that declines the combination gets the plain cooperative launch.
    static bool pdl_ok = true;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)L.smem_bytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_ok ? 2 : 1;
    cudaError_t err = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kernel_for(L)), args);
    if (err != cudaSuccess && pdl_ok) {
        cudaGetLastError();
        pdl_ok = false;
        cfg.numAttrs = 1;
        err = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(kernel_for(L)), args);
    }
    if (err == cudaSuccess) launched += 1;
    return err;
}

}  // namespace moe
