// fused_step.cu -- the decode step as one persistent kernel (one CTA per SM).
//
// Phases inside one launch (cooperative: every CTA is resident):
//   0  router GEMV: logits[t, e] = x[t] . Wr[e] (+ bias), experts spread over
//      CTAs, D split over the consumer warps; x is staged in shared memory as
//      bf16 in the layout of the tensor-core B operand.      -> grid barrier
//   1  every CTA reads the logits and computes softmax, top-k, renormalised
//      weights and the grouping by expert in its own shared memory (the same
//      deterministic result in every CTA; no second exchange).
//   A  gate/up: the U * Dff rows of the selected experts are split evenly over
//      the CTAs into 16-row tiles, each cut into K-slices of 512 inputs. A
//      producer warp streams every slice (one bulk async copy per row) into a
//      shared-memory ring; each slice is owned by one of 15 consumer warps,
//      which runs m16n8k16 tensor-core MMAs on the raw 4-bit codes and applies
//      the groups' scales and biases in f32. The warp finishing a tile's last
//      slice sums the slices' partials in slice order and writes
//      w * silu(g) * u (bf16) for every token routed to the tile's expert.
//                                                            -> grid barrier
//   B  down + combine: each CTA owns a slice of the D output rows for every
//      selected expert; since the routing weight is already folded into h,
//      every warp accumulates its share of sum_e Wd[e] h_e for all tokens and
//      one fixed-order reduction over warps gives the layer output with a
//      single final rounding. The down weights stream into the ring during
//      phase A; the h blocks follow once the grid barrier has passed.
//
// Sources (mlxcel GitHub issues):
//   #1616 "perf(moe): batched decode scales 1.55x against 3.25x on dense":
//     Proposed Solution - a token dimension for the fused decode kernel and
//     one read of each expert plane per step (de-duplication across the
//     cohort); Implementation Notes - f32 partials, single final rounding,
//     n_tokens as a runtime extent.
//   #1859 "perf(moe): attribute the MoE decode gap at the M = 1 expert
//     gather", Problem / Background - the per-(token, k) gather this replaces.
//
// Numerics: codes enter the MMA as exact bf16 integers (128 + q, from a
// magic-exponent bit trick); products and sums are f32. Per group of 64
// inputs, acc = sum (128 + q) v and the row's contribution is
// s * acc + (b - 128 s) * sum(v). Activations enter as bf16 (x, and w * h for
// the down projection), so this path is held to the bf16 tolerance; the f32
// check path keeps every product in f32. All reductions have a fixed order, so
// results are bitwise reproducible run to run.
//
// Every wait is bounded (globaltimer, 1 s); a timeout sets a status bit and
// the CTA skips the remaining waits, still passes every barrier it shares
// with its own threads, drains its in-flight copies and exits.
#include <cuda_bf16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {

namespace {

// 16 warps per CTA: registers are allocated to warps in groups of four, so a
// 17th warp would cost the register budget of 20
constexpr int kCW = 15;                      // consumer warps
constexpr int kThreads = (kCW + 1) * 32;     // + one producer warp
constexpr int kProducer = kCW;
constexpr int kNFast = 8;                    // cohort sizes 1..8 (one n8 MMA tile)
constexpr int kMaxSlotsF = kNFast * kMaxTopK;
constexpr int kMaxATiles = 192;
constexpr int kGA = 8;                       // groups per gate/up K-slice
constexpr int kGB = 4;                       // groups per down K-slice
constexpr int kRT = 4;                       // gate/up partial-sum buffers
constexpr int kMaxRing = 32;
constexpr int kSbuf = 1024;                  // per-warp scale buffer (bytes)
constexpr int kHBlock = 512;                 // bytes of one token's h in a down K-slice
constexpr int kStampsPerCta = 16;
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s bound on any wait

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// codes of inputs p and p+4 of a packed word, as bf16x2 values 128 + q
__device__ __forceinline__ uint32_t code_pair(uint32_t word, int p) {
    return ((word >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}

// two k16 MMA steps over one packed word per row (rows g and g+8) and the
// matching activation word (4 bf16x2 pairs: (v0,v4) (v1,v5) (v2,v6) (v3,v7))
__device__ __forceinline__ void mma_word(float (&acc)[4], uint32_t wg, uint32_t wg8, uint4 v) {
    uint32_t a0[4] = {code_pair(wg, 0), code_pair(wg8, 0), code_pair(wg, 1), code_pair(wg8, 1)};
    ptx::mma_bf16_16816(acc, a0, v.x, v.y);
    uint32_t a1[4] = {code_pair(wg, 2), code_pair(wg8, 2), code_pair(wg, 3), code_pair(wg8, 3)};
    ptx::mma_bf16_16816(acc, a1, v.z, v.w);
}

__device__ __forceinline__ float sum_bf16x8(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) s += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xFFFF0000u);
    return s;
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

// byte offset of (down K-slice ks, grouped slot p) in the h area: blocks of
// 32 words x 16 bytes (pair-permuted bf16, as the B operand wants), each
// word position XOR-ed with the token index so that the 8 tokens' fragment
// loads fall on distinct shared-memory banks once copied
__device__ __forceinline__ size_t h_block(int ks, int p, int S) {
    return ((size_t)ks * S + p) * kHBlock;
}

struct Smem {
    uint64_t *full, *empty;
    unsigned long long *s_mask;
    int *s_idx, *s_st, *s_sk, *s_of, *s_counts, *s_off, *s_unique;
    float *s_w, *slot_w;  // slot_w[p]: routing weight of grouped slot p
    int *s_misc;          // [0] abort [1] barrier ok [2] U [3] tiles [4] b0 [5] b1 [6] h ready
    int *seq;             // [kMaxRing] chunk index last stamped into each ring slot
    int *arrivals;        // [kRT] K-slices of the buffer's current tile done
    int *bufround;        // [kRT] tiles completed on each buffer
    int4 *tiles;
    unsigned char *xs;
    float *xsum;
    float *part;          // [kRT][nksA][32 lanes][8]; later the final [kCW][32][8]
    unsigned char *sbuf;  // [kCW][2][kSbuf] per-warp scale double buffer
    unsigned char *ring;
};

__device__ __forceinline__ Smem carve_smem(unsigned char *base, const FusedLayout &L, int E) {
    Smem s;
    s.full = reinterpret_cast<uint64_t *>(base + L.off_bar);
    s.empty = s.full + kMaxRing;
    unsigned char *r = base + L.off_route;  // 128-byte aligned
    s.s_mask = reinterpret_cast<unsigned long long *>(r);
    int *ip = reinterpret_cast<int *>(r + 8 * (size_t)E);
    s.s_idx = ip; ip += kMaxSlotsF;
    s.s_w = reinterpret_cast<float *>(ip); ip += kMaxSlotsF;
    s.s_st = ip; ip += kMaxSlotsF;
    s.s_sk = ip; ip += kMaxSlotsF;
    s.s_of = ip; ip += kMaxSlotsF;
    s.slot_w = reinterpret_cast<float *>(ip); ip += kMaxSlotsF;
    s.s_misc = ip; ip += 16;
    s.seq = ip; ip += kMaxRing;
    s.arrivals = ip; ip += kRT;
    s.bufround = ip; ip += kRT;
    s.s_counts = ip; ip += E;
    s.s_off = ip; ip += E + 1;
    s.s_unique = ip;
    s.tiles = reinterpret_cast<int4 *>(base + L.off_tiles);
    s.xs = base + L.off_x;
    s.xsum = reinterpret_cast<float *>(base + L.off_xsum);
    s.part = reinterpret_cast<float *>(base + L.off_part);
    s.sbuf = base + L.off_sbuf;
    s.ring = base + L.off_ring;
    return s;
}

__device__ __forceinline__ void set_timeout(volatile int *abort_flag, unsigned *status) {
    *abort_flag = 1;
    atomicOr(status, kDevErrTimeout);
}

// bounded wait on an mbarrier phase; false on timeout or abort
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           unsigned *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (unsigned it = 0;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 63) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) {
                set_timeout(abort_flag, status);
                return false;
            }
        }
    }
}

// bounded spin until *flag == want (shared memory, written by another warp)
__device__ __forceinline__ bool wait_value(volatile int *flag, int want, volatile int *abort_flag,
                                           unsigned *status) {
    if (*flag == want) return true;
    const unsigned long long t0 = globaltimer();
    while (*flag != want) {
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitNs) {
            set_timeout(abort_flag, status);
            return false;
        }
    }
    return true;
}

// wait for ring chunk `ci`: first until the producer has stamped the slot with
// this chunk (a consumer may be several uses of a slot ahead of the data it
// holds, which a parity test alone cannot tell apart), then for the data
__device__ __forceinline__ bool wait_chunk(uint64_t *full, volatile int *seq, int ci, int NS,
                                           volatile int *abort_flag, unsigned *status) {
    const int slot = ci % NS;
    if (!wait_value(seq + slot, ci, abort_flag, status)) return false;
    return wait_phase(&full[slot], (ci / NS) & 1, abort_flag, status);
}

// grid-wide barrier among all CTAs. The arrival counter only grows: a CTA that
// arrives as number `prev` waits until the counter reaches the next multiple of
// G. `cons_only` syncs the consumer warps with a named barrier (the producer
// warp does not take part), otherwise all threads with __syncthreads.
__device__ __forceinline__ bool grid_barrier(unsigned long long *cnt, unsigned G,
                                             volatile int *flag_ok, volatile int *abort_flag,
                                             unsigned *status, bool cons_only) {
    if (cons_only) ptx::named_bar(1, kCW * 32); else __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        const unsigned long long prev = ptx::atom_add_release_gpu_u64(cnt, 1ull);
        const unsigned long long target = (prev / G + 1) * G;
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
    if (cons_only) ptx::named_bar(1, kCW * 32); else __syncthreads();
    return *flag_ok != 0;
}

__device__ __forceinline__ void stamp(unsigned long long *times, bool on, int i) {
    if (on && threadIdx.x == 0) times[blockIdx.x * kStampsPerCta + i] = globaltimer();
}

struct FusedArgs {
    StepArgs a;
    Workspace ws;
    FusedLayout L;
};

// decoded down chunk: expert index u, 16-row tile rt, K-slice ks
struct BChunk {
    int u, rt, ks;
};

__device__ __forceinline__ BChunk decode_b(int bi, int nrt, int nksB) {
    BChunk b;
    b.u = bi / (nrt * nksB);
    const int rem = bi - b.u * nrt * nksB;
    b.rt = rem / nksB;
    b.ks = rem - b.rt * nksB;
    return b;
}

__global__ void __launch_bounds__(kThreads, 1) fused_step_kernel(const __grid_constant__ FusedArgs P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const FusedLayout &L = P.L;
    const StepArgs &A = P.a;
    const Workspace &W = P.ws;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = A.s.E, K = A.s.k, D = A.s.D, F = A.s.F, n = A.s.n;
    const int GD = D / kGroup, GF = F / kGroup;
    const unsigned G = gridDim.x;
    const int cta = blockIdx.x;
    Smem S = carve_smem(smem_raw, L, E);
    volatile int *abort_flag = S.s_misc + 0;
    volatile int *bar_ok = S.s_misc + 1;
    volatile int *h_ready = S.s_misc + 6;
    volatile int *seq = S.seq;
    volatile int *arrivals = S.arrivals;
    volatile int *bufround = S.bufround;
    unsigned char *Hb = reinterpret_cast<unsigned char *>(W.h);  // h blocks, see h_block
    const int Sl = n * K;                                         // grouped slots
    const bool timing = (A.s.flags & MOE_FLAG_PHASE_TIMES) != 0;
    unsigned long long *gsync = reinterpret_cast<unsigned long long *>(W.sync);

    stamp(W.phase_ns, timing, 0);
    if (tid == 0) {
        for (int s = 0; s < L.NS; ++s) {
            ptx::mbar_init(&S.full[s], 1);
            ptx::mbar_init(&S.empty[s], 1);
            S.seq[s] = -1;
        }
        for (int b = 0; b < kRT; ++b) {
            S.arrivals[b] = 0;
            S.bufround[b] = 0;
        }
        S.s_misc[0] = 0;
        S.s_misc[6] = 0;
        ptx::mbar_fence_init();
    }
    __syncthreads();

    // ---- phase 0a: router logits (consumer warps split D) -----------------------
    if (warp < kCW) {
        for (int e = cta; e < E; e += G) {
            float acc[kNFast];
#pragma unroll
            for (int t = 0; t < kNFast; ++t) acc[t] = 0.f;
            for (int i = (warp * 32 + lane) * 8; i < D; i += kCW * 256) {
                float wv[8];
                load8f(A.router_w, (size_t)e * D + i, A.s.w_dtype, wv);
#pragma unroll
                for (int t = 0; t < kNFast; ++t) {
                    if (t < n) {
                        float xv[8];
                        load8f(A.x, (size_t)t * D + i, A.s.x_dtype, xv);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[t] = fmaf(xv[j], wv[j], acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kNFast; ++t) {
                const float v = warp_sum(acc[t]);
                if (lane == 0) S.part[warp * kNFast + t] = v;
            }
            ptx::named_bar(1, kCW * 32);
            if (tid < n) {
                float l = 0.f;
                for (int w = 0; w < kCW; ++w) l += S.part[w * kNFast + tid];
                if (A.router_bias) l += A.router_bias[e];
                W.logits[(size_t)tid * E + e] = l;
            }
            ptx::named_bar(1, kCW * 32);
        }
    }

    // ---- phase 0b: x -> bf16, pair-permuted per 8-word, plus group sums ----------
    {
        const int words = D / 8;
        for (int i = tid; i < n * words; i += kThreads) {
            const int t = i / words, wd = i - t * words;
            float v[8];
            load8f(A.x, (size_t)t * D + (size_t)wd * 8, A.s.x_dtype, v);
            uint16_t b[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = f2bf(v[j]);
            uint4 o;
            o.x = (uint32_t)b[0] | ((uint32_t)b[4] << 16);
            o.y = (uint32_t)b[1] | ((uint32_t)b[5] << 16);
            o.z = (uint32_t)b[2] | ((uint32_t)b[6] << 16);
            o.w = (uint32_t)b[3] | ((uint32_t)b[7] << 16);
            *reinterpret_cast<uint4 *>(S.xs + (size_t)t * L.x_stride + (size_t)wd * 16) = o;
        }
    }
    __syncthreads();
    for (int i = tid; i < GD * n; i += kThreads) {
        const int gg = i / n, t = i - gg * n;
        const unsigned char *row = S.xs + (size_t)t * L.x_stride + (size_t)gg * 128;
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += sum_bf16x8(*reinterpret_cast<const uint4 *>(row + w * 16));
        S.xsum[gg * kNFast + t] = s;
    }

    // ---- grid barrier 1: all logits written -------------------------------------
    stamp(W.phase_ns, timing, 1);
    if ((A.s.flags & MOE_FLAG_TEST_STALL) && cta == 0)
        __syncthreads();  // test hook: CTA 0 never arrives; the others time out
    else
        grid_barrier(gsync, G, bar_ok, abort_flag, W.status, false);
    stamp(W.phase_ns, timing, 2);

    // ---- phase 1: routing and grouping, redundantly in every CTA ---------------
    block_topk(W.logits, n, E, K, S.s_idx, S.s_w);
    __syncthreads();
    stamp(W.phase_ns, timing, 15);
    int *s_Uptr = S.s_misc + 2;
    block_group(S.s_idx, n, E, K, S.s_mask, S.s_counts, S.s_off, S.s_st, S.s_sk, S.s_of,
                S.s_unique, s_Uptr);
    for (int s = tid; s < Sl; s += kThreads) S.slot_w[S.s_of[s]] = S.s_w[s];
    if (cta == 0) {
        for (int s = tid; s < Sl; s += kThreads) {
            W.topk_idx[s] = S.s_idx[s];
            W.topk_w[s] = S.s_w[s];
            W.slot_token[s] = S.s_st[s];
            W.slot_k[s] = S.s_sk[s];
            W.slot_of[s] = S.s_of[s];
        }
        const int U = *s_Uptr;
        for (int e = tid; e < E; e += kThreads) {
            W.counts[e] = S.s_counts[e];
            W.offsets[e] = S.s_off[e];
            W.unique[e] = e < U ? S.s_unique[e] : -1;
        }
        if (tid == 0) {
            W.offsets[E] = S.s_off[E];
            *W.U = U;
        }
    }
    // work lists: gate/up row tiles of this CTA, and its down rows
    if (tid == 0) {
        const unsigned U = (unsigned)*s_Uptr;
        const unsigned RA = U * (unsigned)F;
        const unsigned a0 = RA * (unsigned)cta / G, a1 = RA * (unsigned)(cta + 1) / G;
        unsigned pos = a0;
        int nt = 0;
        while (pos < a1 && nt < kMaxATiles) {
            const unsigned u = pos / (unsigned)F, f = pos - u * (unsigned)F;
            const unsigned seg_end = min(a1, (u + 1) * (unsigned)F);
            const unsigned rows = min(16u, seg_end - pos);
            S.tiles[nt++] = make_int4((int)u, (int)f, (int)rows, 0);
            pos += rows;
        }
        if (pos < a1) atomicOr(W.status, kDevErrInternal);  // the host bounds the count
        S.s_misc[3] = nt;
        S.s_misc[4] = (int)((unsigned)D * (unsigned)cta / G);
        S.s_misc[5] = (int)((unsigned)D * (unsigned)(cta + 1) / G);
    }
    __syncthreads();
    stamp(W.phase_ns, timing, 3);

    const int U = S.s_misc[2];
    const int nTiles = S.s_misc[3];
    const int b0 = S.s_misc[4], rowsB = S.s_misc[5] - S.s_misc[4];
    const int nrt = (rowsB + 15) >> 4;
    const int nA = nTiles * L.nksA;
    const int nB = rowsB > 0 ? U * nrt * L.nksB : 0;
    const int total = nA + nB;

    if (warp == kProducer) {
        // ================= producer: stream the selected planes =================
        const uint64_t pol = ptx::policy_evict_first();
        const unsigned char *gq = reinterpret_cast<const unsigned char *>(A.planes.gate_q);
        const unsigned char *uq = reinterpret_cast<const unsigned char *>(A.planes.up_q);
        const unsigned char *dq = reinterpret_cast<const unsigned char *>(A.planes.down_q);
        int pend_lo = nA, pend_hi = nA;  // down chunks whose h block is not issued yet
        bool fenced = false;
        unsigned long long t_wait = 0;
        int issued = 0;
        // lane 0 only: issue the deferred h blocks once h is complete
        auto flush = [&]() {
            if (!fenced) {
                __threadfence_block();
                ptx::fence_proxy_async_global();
                fenced = true;
            }
            for (int pi = pend_lo; pi < pend_hi; ++pi) {
                const BChunk bc = decode_b(pi - nA, nrt, L.nksB);
                const int e = S.s_unique[bc.u];
                ptx::bulk_g2s(S.ring + (size_t)(pi % L.NS) * L.slot_bytes + L.hoff,
                              Hb + h_block(bc.ks, S.s_off[e], Sl), (uint32_t)S.s_counts[e] * kHBlock,
                              &S.full[pi % L.NS], pol);
            }
            pend_lo = pend_hi;
        };
        for (int ci = 0; ci < total; ++ci) {
            const int slot = ci % L.NS, use = ci / L.NS;
            int ok = 1;
            if (lane == 0) {
                const unsigned long long tw0 = timing ? globaltimer() : 0ull;
                if (use > 0) {
                    const unsigned long long t0 = globaltimer();
                    for (unsigned it = 0;; ++it) {
                        if (ptx::mbar_try_wait(&S.empty[slot], (use - 1) & 1)) break;
                        if (pend_lo < pend_hi && *h_ready) flush();
                        if ((it & 63) == 63 && (*abort_flag || globaltimer() - t0 > kWaitNs)) {
                            if (!*abort_flag) set_timeout(abort_flag, W.status);
                            ok = 0;
                            break;
                        }
                    }
                }
                if (timing) t_wait += globaltimer() - tw0;
                if (ok) seq[slot] = ci;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            unsigned char *dst = S.ring + (size_t)slot * L.slot_bytes;
            if (ci < nA) {
                const int4 tl = S.tiles[ci / L.nksA];
                const int ks = ci % L.nksA;
                const int e = S.s_unique[tl.x], rows = tl.z;
                const int kb = min(256, D / 2 - 256 * ks);
                const size_t row0 = (size_t)e * F + tl.y;
                if (lane == 0) ptx::mbar_arrive_expect_tx(&S.full[slot], 2u * rows * kb);
                __syncwarp();
                if (lane < rows)
                    ptx::bulk_g2s(dst + lane * L.SA, gq + (row0 + lane) * (D / 2) + 256 * ks, kb,
                                  &S.full[slot], pol);
                else if (lane >= 16 && lane - 16 < rows)
                    ptx::bulk_g2s(dst + 16 * L.SA + (lane - 16) * L.SA,
                                  uq + (row0 + lane - 16) * (D / 2) + 256 * ks, kb, &S.full[slot], pol);
            } else {
                const BChunk bc = decode_b(ci - nA, nrt, L.nksB);
                const int e = S.s_unique[bc.u];
                const int rowsT = min(16, rowsB - 16 * bc.rt);
                const int kb = min(128, F / 2 - 128 * bc.ks);
                const uint32_t hbytes = (uint32_t)S.s_counts[e] * kHBlock;
                if (lane == 0) ptx::mbar_arrive_expect_tx(&S.full[slot], (uint32_t)rowsT * kb + hbytes);
                __syncwarp();
                if (lane < rowsT)
                    ptx::bulk_g2s(dst + lane * L.SB,
                                  dq + ((size_t)e * D + b0 + 16 * bc.rt + lane) * (F / 2) + 128 * bc.ks, kb,
                                  &S.full[slot], pol);
                if (lane == 0) {
                    if (pend_lo == pend_hi) pend_lo = ci;
                    pend_hi = ci + 1;
                    if (*h_ready) flush();
                }
            }
            issued = ci + 1;
        }
        if (lane == 0) {
            // every down chunk needs its h blocks: wait for h, then issue the rest
            if (pend_lo < pend_hi && wait_value(h_ready, 1, abort_flag, W.status)) flush();
            if (timing) W.phase_ns[cta * kStampsPerCta + 12] = t_wait;
            // drain: every issued copy must land before the CTA may exit
            for (int ci = max(0, issued - L.NS); ci < issued; ++ci) {
                const int slot = ci % L.NS, use = ci / L.NS;
                if (ci >= nA && ci >= pend_lo && ci < pend_hi) continue;  // h never issued
                const unsigned long long t0 = globaltimer();
                while (!ptx::mbar_try_wait(&S.full[slot], use & 1)) {
                    if (globaltimer() - t0 > kWaitNs) {
                        atomicOr(W.status, kDevErrTimeout);
                        break;
                    }
                }
            }
        }
        __syncwarp();
        return;
    }

    // ===================== consumers (warps 0..kCW-1) ===========================
    const int g = lane >> 2, c = lane & 3;
    const bool tok_live = g < n;  // this lane's B-operand column is a real token
    unsigned char *my_sbuf = S.sbuf + (size_t)warp * 2 * kSbuf;
    // scale/bias arrays selected by value (no indexed pointer arrays, which would
    // live in local memory)
    auto scA = [&](int a) -> const uint16_t * {
        return a == 0 ? A.planes.gate_s : a == 1 ? A.planes.gate_b : a == 2 ? A.planes.up_s : A.planes.up_b;
    };
    auto scB = [&](int a) -> const uint16_t * { return a == 0 ? A.planes.down_s : A.planes.down_b; };

    // prefetch the scales and biases chunk ci needs into scale buffer buf
    auto prefetch_scales = [&](int ci, unsigned char *buf) {
        if (ci >= total) {
            ptx::cp_async_commit();
            return;
        }
        if (ci < nA) {
            const int4 tl = S.tiles[ci / L.nksA];
            const int ks = ci % L.nksA;
            const size_t row0 = (size_t)S.s_unique[tl.x] * F + tl.y;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = lane + 32 * j;
                const int a = i >> 6, r = (i >> 2) & 15, p = i & 3, grp = kGA * ks + 2 * p;
                if (r < tl.z && grp < GD)
                    ptx::cp_async4(buf + (a * 16 + r) * 16 + p * 4, scA(a) + (row0 + r) * GD + grp);
            }
        } else {
            const BChunk bc = decode_b(ci - nA, nrt, L.nksB);
            const int rowsT = min(16, rowsB - 16 * bc.rt);
            const size_t row0 = (size_t)S.s_unique[bc.u] * D + b0 + 16 * bc.rt;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j;
                const int a = i >> 5, r = (i >> 1) & 15, p = i & 1, grp = kGB * bc.ks + 2 * p;
                if (r < rowsT && grp < GF)
                    ptx::cp_async4(buf + (a * 16 + r) * 8 + p * 4, scB(a) + (row0 + r) * GF + grp);
            }
        }
        ptx::cp_async_commit();
    };

    unsigned long long ta_wait = 0, ta_comp = 0, tb_wait = 0, tb_comp = 0;
    int jj = 0;  // index of this warp's current chunk in its own sequence
    prefetch_scales(warp, my_sbuf);

    // ---- phase A: gate/up K-slices ------------------------------------------------
    for (int ci = warp; ci < nA; ci += kCW, ++jj) {
        const int slot = ci % L.NS;
        unsigned char *sb = my_sbuf + (jj & 1) * kSbuf;
        prefetch_scales(ci + kCW, my_sbuf + ((jj + 1) & 1) * kSbuf);
        const unsigned long long tw0 = timing ? globaltimer() : 0ull;
        const bool ok = wait_chunk(S.full, seq, ci, L.NS, abort_flag, W.status);
        ptx::cp_async_wait<1>();
        __syncwarp();
        const unsigned long long tw1 = timing ? globaltimer() : 0ull;
        const int t_idx = ci / L.nksA, ks = ci % L.nksA;
        const int4 tl = S.tiles[t_idx];
        const int e = S.s_unique[tl.x], f0 = tl.y, rows = tl.z;
        const unsigned char *gqs = S.ring + (size_t)slot * L.slot_bytes;
        const unsigned char *uqs = gqs + 16 * L.SA;
        const uint16_t *scs = reinterpret_cast<const uint16_t *>(sb);  // [4][16][8]
        float tg[4] = {0.f, 0.f, 0.f, 0.f}, tu[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll 1
            for (int G0 = 0; G0 < kGA; G0 += 4) {
                uint2 wg0[4], wg1[4], wu0[4], wu1[4];
                uint4 xb0[4], xb1[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int Gl = G0 + i;
                    const int gg = min(kGA * ks + Gl, GD - 1);
                    wg0[i] = *reinterpret_cast<const uint2 *>(gqs + g * L.SA + Gl * 32 + c * 8);
                    wg1[i] = *reinterpret_cast<const uint2 *>(gqs + (g + 8) * L.SA + Gl * 32 + c * 8);
                    wu0[i] = *reinterpret_cast<const uint2 *>(uqs + g * L.SA + Gl * 32 + c * 8);
                    wu1[i] = *reinterpret_cast<const uint2 *>(uqs + (g + 8) * L.SA + Gl * 32 + c * 8);
                    xb0[i] = make_uint4(0, 0, 0, 0);
                    xb1[i] = make_uint4(0, 0, 0, 0);
                    if (tok_live) {
                        const unsigned char *xr = S.xs + (size_t)g * L.x_stride + (size_t)(8 * gg + 2 * c) * 16;
                        xb0[i] = *reinterpret_cast<const uint4 *>(xr);
                        xb1[i] = *reinterpret_cast<const uint4 *>(xr + 16);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int Gl = G0 + i;
                    const int gg = kGA * ks + Gl;
                    if (gg < GD) {
                        float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_word(cg, wg0[i].x, wg1[i].x, xb0[i]);
                        mma_word(cu, wu0[i].x, wu1[i].x, xb0[i]);
                        mma_word(cg, wg0[i].y, wg1[i].y, xb1[i]);
                        mma_word(cu, wu0[i].y, wu1[i].y, xb1[i]);
                        const float2 xsm = *reinterpret_cast<const float2 *>(S.xsum + gg * kNFast + 2 * c);
                        const float sg0 = bf2f(scs[(0 * 16 + g) * 8 + Gl]), bg0 = bf2f(scs[(1 * 16 + g) * 8 + Gl]);
                        const float sg1 = bf2f(scs[(0 * 16 + g + 8) * 8 + Gl]), bg1 = bf2f(scs[(1 * 16 + g + 8) * 8 + Gl]);
                        const float su0 = bf2f(scs[(2 * 16 + g) * 8 + Gl]), bu0 = bf2f(scs[(3 * 16 + g) * 8 + Gl]);
                        const float su1 = bf2f(scs[(2 * 16 + g + 8) * 8 + Gl]), bu1 = bf2f(scs[(3 * 16 + g + 8) * 8 + Gl]);
                        const float og0 = fmaf(-128.f, sg0, bg0), og1 = fmaf(-128.f, sg1, bg1);
                        const float ou0 = fmaf(-128.f, su0, bu0), ou1 = fmaf(-128.f, su1, bu1);
                        tg[0] = fmaf(sg0, cg[0], fmaf(og0, xsm.x, tg[0]));
                        tg[1] = fmaf(sg0, cg[1], fmaf(og0, xsm.y, tg[1]));
                        tg[2] = fmaf(sg1, cg[2], fmaf(og1, xsm.x, tg[2]));
                        tg[3] = fmaf(sg1, cg[3], fmaf(og1, xsm.y, tg[3]));
                        tu[0] = fmaf(su0, cu[0], fmaf(ou0, xsm.x, tu[0]));
                        tu[1] = fmaf(su0, cu[1], fmaf(ou0, xsm.y, tu[1]));
                        tu[2] = fmaf(su1, cu[2], fmaf(ou1, xsm.x, tu[2]));
                        tu[3] = fmaf(su1, cu[3], fmaf(ou1, xsm.y, tu[3]));
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.empty[slot], 1);

        // partial of this K-slice -> the tile's buffer; the last slice reduces
        const int b = t_idx % kRT, round = t_idx / kRT;
        if (lane == 0) wait_value(bufround + b, round, abort_flag, W.status);
        __syncwarp();
        float *pp = S.part + ((size_t)(b * L.nksA + ks) * 32 + lane) * 8;
        *reinterpret_cast<float4 *>(pp) = make_float4(tg[0], tg[1], tg[2], tg[3]);
        *reinterpret_cast<float4 *>(pp + 4) = make_float4(tu[0], tu[1], tu[2], tu[3]);
        __syncwarp();
        int prev = 0;
        if (lane == 0) {
            __threadfence_block();
            prev = atomicAdd(const_cast<int *>(arrivals + b), 1);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == L.nksA - 1) {
            __threadfence_block();
            const unsigned long long m = S.s_mask[e];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int o = lane + 32 * i;
                const int r = o >> 3, t = o & 7;
                const int gl = (r & 7) * 4 + (t >> 1), idx = ((r >> 3) << 1) | (t & 1);
                float gs = 0.f, us = 0.f;
                for (int k2 = 0; k2 < L.nksA; ++k2) {
                    const float *q = S.part + ((size_t)(b * L.nksA + k2) * 32 + gl) * 8;
                    gs += q[idx];
                    us += q[4 + idx];
                }
                if (r < rows && t < n && ((m >> t) & 1ull)) {
                    const int p = S.s_off[e] + __popcll(m & ((1ull << t) - 1ull));
                    const float h = S.slot_w[p] * (gs / (1.0f + expf(-gs)) * us);
                    const int f = f0 + r;
                    const int w = f >> 3, j = f & 7;
                    const int ksb = w >> 5, wl = (w & 31) ^ t;
                    const size_t at = h_block(ksb, p, Sl) + (size_t)wl * 16 + (2 * (j & 3) + (j >> 2)) * 2;
                    *reinterpret_cast<uint16_t *>(Hb + at) = f2bf(h);
                }
            }
            __syncwarp();
            if (lane == 0) {
                arrivals[b] = 0;
                __threadfence_block();
                bufround[b] = round + 1;
            }
        }
        if (timing) {
            ta_wait += tw1 - tw0;
            ta_comp += globaltimer() - tw1;
        }
    }

    // ---- grid barrier 2: every h block written ---------------------------------
    stamp(W.phase_ns, timing, 4);
    grid_barrier(gsync, G, bar_ok, abort_flag, W.status, true);
    if (tid == 0) {
        __threadfence_block();
        *h_ready = 1;
    }
    stamp(W.phase_ns, timing, 5);

    // ---- phase B: down K-slices, all experts summed per warp --------------------
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    const int key = g & 7;
    for (int ci = nA + ((warp - nA % kCW + kCW) % kCW); ci < total; ci += kCW, ++jj) {
        const int slot = ci % L.NS;
        unsigned char *sb = my_sbuf + (jj & 1) * kSbuf;
        prefetch_scales(ci + kCW, my_sbuf + ((jj + 1) & 1) * kSbuf);
        const unsigned long long tw0 = timing ? globaltimer() : 0ull;
        const bool ok = wait_chunk(S.full, seq, ci, L.NS, abort_flag, W.status);
        ptx::cp_async_wait<1>();
        __syncwarp();
        const unsigned long long tw1 = timing ? globaltimer() : 0ull;
        const BChunk bc = decode_b(ci - nA, nrt, L.nksB);
        const int e = S.s_unique[bc.u];
        const unsigned long long m = S.s_mask[e];
        const bool routed = tok_live && ((m >> g) & 1ull);
        const int rank = routed ? __popcll(m & ((1ull << g) - 1ull)) : 0;
        const unsigned char *tb = S.ring + (size_t)slot * L.slot_bytes;
        const unsigned char *hs_base = tb + L.hoff + rank * kHBlock;
        const uint16_t *scs = reinterpret_cast<const uint16_t *>(sb);  // [2][16][4]
        float cacc[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll
            for (int Gl = 0; Gl < kGB; ++Gl) {
                const int Gg = kGB * bc.ks + Gl;
                if (Gg < GF) {
                    const uint2 w0 = *reinterpret_cast<const uint2 *>(tb + g * L.SB + Gl * 32 + c * 8);
                    const uint2 w1 = *reinterpret_cast<const uint2 *>(tb + (g + 8) * L.SB + Gl * 32 + c * 8);
                    uint4 hb0 = make_uint4(0, 0, 0, 0), hb1 = make_uint4(0, 0, 0, 0);
                    if (routed) {
                        hb0 = *reinterpret_cast<const uint4 *>(hs_base + (((8 * Gl + 2 * c) ^ key) * 16));
                        hb1 = *reinterpret_cast<const uint4 *>(hs_base + (((8 * Gl + 2 * c + 1) ^ key) * 16));
                    }
                    float hs = sum_bf16x8(hb0) + sum_bf16x8(hb1);
                    hs += __shfl_xor_sync(0xffffffffu, hs, 1);
                    hs += __shfl_xor_sync(0xffffffffu, hs, 2);
                    const float hs0 = __shfl_sync(0xffffffffu, hs, 8 * c);
                    const float hs1 = __shfl_sync(0xffffffffu, hs, 8 * c + 4);
                    float cd[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_word(cd, w0.x, w1.x, hb0);
                    mma_word(cd, w0.y, w1.y, hb1);
                    const float s0 = bf2f(scs[(0 * 16 + g) * 4 + Gl]), o0 = fmaf(-128.f, s0, bf2f(scs[(1 * 16 + g) * 4 + Gl]));
                    const float s1 = bf2f(scs[(0 * 16 + g + 8) * 4 + Gl]), o1 = fmaf(-128.f, s1, bf2f(scs[(1 * 16 + g + 8) * 4 + Gl]));
                    cacc[0] = fmaf(s0, cd[0], fmaf(o0, hs0, cacc[0]));
                    cacc[1] = fmaf(s0, cd[1], fmaf(o0, hs1, cacc[1]));
                    cacc[2] = fmaf(s1, cd[2], fmaf(o1, hs0, cacc[2]));
                    cacc[3] = fmaf(s1, cd[3], fmaf(o1, hs1, cacc[3]));
                }
            }
        }
        if (bc.rt == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) acc0[i] += cacc[i];
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) acc1[i] += cacc[i];
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.empty[slot], 1);
        if (timing) {
            tb_wait += tw1 - tw0;
            tb_comp += globaltimer() - tw1;
        }
    }
    ptx::cp_async_wait<0>();
    if (timing && tid == 0) {
        unsigned long long *tt = W.phase_ns + cta * kStampsPerCta;
        tt[8] = ta_wait;
        tt[9] = ta_comp;
        tt[10] = tb_wait;
        tt[11] = tb_comp;
        tt[13] = (unsigned long long)nA;
        tt[14] = (unsigned long long)nB;
    }

    // ---- final: fixed-order sum over warps of their partial outputs -------------
    {
        float *red = S.part + ((size_t)warp * 32 + lane) * 8;
        *reinterpret_cast<float4 *>(red) = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
        *reinterpret_cast<float4 *>(red + 4) = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
    }
    ptx::named_bar(1, kCW * 32);
    stamp(W.phase_ns, timing, 6);
    for (int o = tid; o < n * rowsB; o += kCW * 32) {
        const int t = o / rowsB, r = o - t * rowsB;
        const int rr = r & 15;
        const int gl = (rr & 7) * 4 + (t >> 1), idx = (r >> 4) * 4 + ((rr >> 3) << 1) + (t & 1);
        float v = 0.f;
        for (int w = 0; w < kCW; ++w) v += S.part[((size_t)w * 32 + gl) * 8 + idx];
        const size_t at = (size_t)t * D + b0 + r;
        if (A.s.out_dtype == MOE_DTYPE_F32)
            static_cast<float *>(A.out)[at] = v;
        else
            static_cast<uint16_t *>(A.out)[at] = f2bf(v);
    }
    if (timing) {
        ptx::named_bar(1, kCW * 32);
        stamp(W.phase_ns, timing, 7);
    }
}

}  // namespace

// ---- host side -----------------------------------------------------------------

static int round_up(int v, int m) { return (v + m - 1) / m * m; }

// row stride in shared memory for rows of `bytes` bytes: keeps the 8 rows a
// fragment load touches on distinct bank groups (stride/4 == 8 mod 32)
static int padded_stride(int bytes) {
    const int words = bytes / 4;
    const int pad_words = ((8 - words) % 32 + 32) % 32;
    return bytes + pad_words * 4;
}

bool fused_layout(const moe_config &c, int num_sms, int max_smem, FusedLayout *out) {
    FusedLayout L{};
    const int D = c.D, F = c.Dff, E = c.E, k = c.top_k;
    if (k * kNFast > kMaxSlotsF) return false;
    if (D % 128 || F % 128) return false;  // even group counts: 4-byte scale copies
    L.G = num_sms;
    L.nksA = (D / kGroup + kGA - 1) / kGA;
    L.nksB = (F / kGroup + kGB - 1) / kGB;
    const int rowsBmax = (D + L.G - 1) / L.G;
    if (rowsBmax > 32) return false;
    L.SA = padded_stride(kGA * 32);
    L.SB = padded_stride(kGB * 32);
    L.hoff = round_up(16 * L.SB, 128);
    const int a_bytes = 32 * L.SA;
    const int b_bytes = L.hoff + kNFast * kHBlock;
    L.slot_bytes = round_up(a_bytes > b_bytes ? a_bytes : b_bytes, 128);
    // gate/up tiles per CTA: rows ceil(U*F/G) with U <= min(E, 8k), split at expert edges
    const int Umax = E < kNFast * k ? E : kNFast * k;
    const long long rows_cta = ((long long)Umax * F + L.G - 1) / L.G;
    const long long tiles = (rows_cta + 15) / 16 + rows_cta / F + 2;
    if (tiles > kMaxATiles) return false;
    L.x_tokens = c.max_tokens < kNFast ? c.max_tokens : kNFast;
    L.x_stride = 2 * D + 16;
    int off = 0;
    L.off_bar = off;
    off += round_up(2 * 8 * kMaxRing, 128);
    L.off_route = off;
    off += round_up(8 * E + 4 * (6 * kMaxSlotsF + 16 + kMaxRing + 2 * kRT + E + (E + 1) + E) + 64, 128);
    L.off_tiles = off;
    off += round_up(16 * kMaxATiles, 128);
    L.off_x = off;
    off += round_up(L.x_tokens * L.x_stride, 128);
    L.off_xsum = off;
    off += round_up(4 * kNFast * (D / kGroup), 128);
    L.part_bytes = 4 * 8 * 32 * (kRT * L.nksA > kCW ? kRT * L.nksA : kCW);
    L.off_part = off;
    off += round_up(L.part_bytes, 128);
    L.off_sbuf = off;
    off += kCW * 2 * kSbuf;
    off = round_up(off, 1024);
    L.off_ring = off;
    const int room = max_smem - off;
    int ns = room / L.slot_bytes;
    if (ns > kMaxRing) ns = kMaxRing;
    if (ns < 4) return false;
    L.NS = ns;
    L.smem_bytes = off + ns * L.slot_bytes;
    *out = L;
    return true;
}

cudaError_t fused_prepare(const FusedLayout &L, int *blocks_per_sm) {
    cudaError_t err = cudaFuncSetAttribute(fused_step_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem_bytes);
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fused_step_kernel, kThreads,
                                                         (size_t)L.smem_bytes);
}

int fused_max_tokens() { return kNFast; }

cudaError_t launch_fused(const StepArgs &a, const Workspace &ws, const FusedLayout &L,
                         cudaStream_t st, int &launched) {
    FusedArgs P;
    P.a = a;
    P.ws = ws;
    P.L = L;
    void *args[] = {&P};
    cudaError_t err = cudaLaunchCooperativeKernel((const void *)fused_step_kernel, dim3(L.G),
                                                  dim3(kThreads), args, (size_t)L.smem_bytes, st);
    if (err == cudaSuccess) launched += 1;
    return err;
}

}  // namespace moe
