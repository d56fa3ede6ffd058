// prefill_tc.cu -- the grouped (17..64 tokens) and prefill paths' tensor-core
// kernels on the 5th-generation tensor cores (tcgen05.mma, accumulators in
// tensor memory): the expert GEMMs (expert_tc_kernel, with x_to_f16_kernel for
// their B operand) and the prefill router (router_tc_kernel, near the end).
//
// A prefill cohort gives each selected expert tens to hundreds of tokens, so
// its MLP is a real matrix product (the sorted qmm path of prompt processing in
// mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against 3.25x on
// dense", Current Behavior, and issue #1859 "perf(moe): attribute the MoE decode
// gap at the M = 1 expert gather", Problem / Background).
//
// Operands. The tensor core reads f16 tiles in the K-major layout with the
// 128-byte swizzle: a chunk's 64 inputs of a row are one 128-byte row, whose
// 16-byte pieces (8 inputs each) are permuted by XOR with the row index mod 8,
// which spreads 8 consecutive rows over all shared-memory banks for both the
// tensor core's reads and the CUDA cores' stores. Inside every piece both
// operands keep the order 0 4 1 5 2 6 3 7: the 4-bit decode
// (nibbles p and p + 4 of a word into one f16 pair) produces it directly, and a
// dot product does not depend on the order of its terms.
//   - B (activations) is stored in that order once, as f16: x by x_to_f16_kernel
//     (into the workspace's y area, unused until the down projection writes
//     it), h by the gate/up epilogue (into the first half of each h row). The
//     GEMMs copy B rows straight into swizzled tiles with 16-byte cp.async.
//   - A (weights) is dequantised by the CUDA cores: w = s q + b, one f16
//     rounding, as the grouped path's tile variant.
//
// Per work item: one expert, 128 weight rows, 64 of the expert's tokens at a time,
// K (the reduction) in chunks of 128 inputs = two quantisation groups:
//   - a ring of S stages holds, per chunk, the B tile, the raw codes and the
//     scale/bias words of the CTA's rows, filled S - 1 chunks ahead;
//   - the CUDA cores dequantise chunk i into one of two A tiles while the
//     tensor core runs chunk i - 1 (one thread issues M = 128, N = 64, K = 16
//     MMAs and commits them to an mbarrier);
//   - token blocks alternate between two accumulators; one chunk after a
//     block's last one, tcgen05.ld brings its f32 accumulators to registers:
//     h = act(gate, up) (gate row r and up row r are both tensor-memory lane
//     r) or y for the down projection.
// An operand beyond f16's range saturates and is reported (MOE_ERR_RANGE);
// every mbarrier wait gives up after 1 s and reports a timeout.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "activation.cuh"
#include "device_status.cuh"
#include "moe_internal.h"
#include "prefill_tc.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kM = 128;          // weight rows per A tile
constexpr int kN = 64;           // tokens per block
constexpr int kK = 128;          // inputs per chunk: two quantisation groups
constexpr int kSbo = 1024;       // bytes between 8-row swizzle atoms (8 rows x 128 B)
constexpr int kSubB = kN * 64 * 2;    // 8 KB: 64 tokens x 64 inputs, one 128-byte swizzled sub-tile
constexpr int kTileB = 2 * kSubB;     // 16 KB: the chunk's activation tile
constexpr unsigned long long kWaitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// bounded wait on an mbarrier phase: false (and a reported timeout) after 1 s
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned *status) {
    uint32_t ok = 0;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(tc::smem_u32(bar)), "r"(parity), "r"(20000u)
            : "memory");
        if (ok) return true;
        if (globaltimer() - t0 > kWaitNs) {
            report_error(status, kDevErrTimeout);
            return false;
        }
    }
}

// f16 of an f32 value; beyond f16's range: saturate and report
__device__ __forceinline__ __half sat_h(float v, unsigned *status) {
    if (fabsf(v) > 65504.0f) {
        report_error(status, kDevErrRange);
        v = fminf(fmaxf(v, -65504.0f), 65504.0f);
    }
    return __float2half_rn(v);
}

__device__ __forceinline__ uint32_t h2u(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// position of input p (0..7) inside its group of 8 in the core order 0 4 1 5 2 6 3 7
__host__ __device__ __forceinline__ int core_pos(int p) { return p < 4 ? 2 * p : 2 * (p - 4) + 1; }

// one 8-input core of f16 weights from a packed 4-bit word (inputs 8i..8i+7,
// code j at bits 4j): the pairs (0,4) (1,5) (2,6) (3,7), each w = s q + b with
// one rounding. Codes 0 and 4 (2 and 6 after one shift) masked into an f16's
// mantissa give 1024 + q; codes 1 and 5 (3 and 7) masked in place give
// 1024 + 16 q, and (1024 + 16 q) / 16 - 64 = q exactly: five integer ops per
// eight codes
__device__ __forceinline__ uint4 deq_word(uint32_t w, __half2 s2, __half2 b2) {
    const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
    const __half2 k16th = __floats2half2_rn(0.0625f, 0.0625f), km64 = __floats2half2_rn(-64.f, -64.f);
    const uint32_t w8 = w >> 8;
    const uint32_t v[4] = {(w & 0x000F000Fu) | 0x64006400u, (w & 0x00F000F0u) | 0x64006400u,
                           (w8 & 0x000F000Fu) | 0x64006400u, (w8 & 0x00F000F0u) | 0x64006400u};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&v[p]);
        const __half2 q = (p & 1) ? __hfma2(h, k16th, km64) : __hsub2(h, k1024);  // q, exact
        const __half2 r = __hfma2(q, s2, b2);
        o[p] = *reinterpret_cast<const uint32_t *>(&r);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// the same for the 8 codes 8i..8i+7 of a 6-bit row chunk (code j at bits 6j)
__device__ __forceinline__ uint4 deq_6bit(const uint32_t (&v)[12], int i, __half2 s2, __half2 b2) {
    const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int bit = 6 * (8 * i + p + 4 * h), wi = bit >> 5, sh = bit & 31;
            q[h] = __funnelshift_r(v[wi], wi + 1 < 12 ? v[wi + 1] : 0u, sh) & 0x3Fu;
        }
        const uint32_t c = (q[0] | (q[1] << 16)) | 0x64006400u;
        const __half2 qq = __hsub2(*reinterpret_cast<const __half2 *>(&c), k1024);
        const __half2 r = __hfma2(qq, s2, b2);
        o[p] = *reinterpret_cast<const uint32_t *>(&r);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// byte offset of (row, 8-input piece j) in a K-major tile of 64-input rows with
// the 128-byte swizzle (piece j of row r at piece j ^ (r % 8) of its 128 bytes)
__device__ __forceinline__ uint32_t core_off(int row, int j) {
    return (uint32_t)((row >> 3) * kSbo + (row & 7) * 128 + ((j ^ (row & 7)) << 4));
}

// ---- x -> f16 in the core order ------------------------------------------------
// One thread per 8 inputs of a token; the f16 copy lives in the workspace's y
// area (n x D f16 fits in the n k x D f32 of y, which the down projection
// writes only after the gate/up GEMMs have read x).
template <int XD>
__global__ void x_to_f16_kernel(StepArgs a, Workspace ws) {
    const int D = a.s.D, per_tok = D / 8;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)a.s.n * per_tok) return;
    const size_t t = i / per_tok, g = i % per_tok;
    float v[8];
    if (XD == MOE_DTYPE_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.x) + t * D + 8 * g);
        const float4 f0 = src[0], f1 = src[1];
        v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
        v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
    } else {
        const uint4 w = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + t * D + 8 * g);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(ww[k] << 16);
            v[2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
        }
    }
    __half h[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) h[core_pos(p)] = sat_h(v[p], ws.status);
    *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(ws.y) + t * D + 8 * g) =
        make_uint4(h2u(h[0], h[1]), h2u(h[2], h[3]), h2u(h[4], h[5]), h2u(h[6], h[7]));
}

// ---- the GEMMs -------------------------------------------------------------------
// Warp roles (MATS = 2 for gate/up, 1 for down):
//   - MATS x 8 dequantisation warps: thread (lane quadrant q, matrix m, group
//     g of the chunk) owns weight row 32 q + lane of matrix m -- the
//     tensor-memory lane of that row -- and dequantises that row's 64 weights
//     of group g of every chunk. Once the chunk's codes (c_full) and scale words
//     (b_full) are in the ring and the MMAs of chunk - 2 are done (mma_done),
//     it dequantises into A buffer (chunk % 2), arrives on c_empty and a_full.
//     The same warps run a token block's epilogue, one chunk after the block's
//     last one.
//   - four producer warps, one per SM sub-partition (a single one held up the
//     dequantisation warps of its sub-partition behind its copies), copy the B
//     tiles (64 tokens x 128 inputs, f16) and the chunk's scale and bias words
//     into the ring, each lane arriving on b_full when its copies have landed;
//     lane 0 of the first also loads the chunk's codes (one TMA box of 128 rows
//     per matrix, completing on c_full). A stage is refilled once its MMAs
//     (b_empty) and its dequantisation (c_empty) are done.
//   - one MMA warp waits for a_full and b_full (and, at a block's first chunk,
//     for the epilogue of block - 2 to have read the accumulator, acc_empty),
//     and one elected lane issues the chunk's MMAs and commits them to mma_done
//     (A buffer free), b_empty (ring stage free) and, after a block's last
//     chunk, acc_full.
// Every wait gives up after 1 s: it reports a timeout and sets the CTA's abort
// flag, which every role checks once per chunk.
//
// Ring stage layout (bytes): [B tile: two 8 KB sub-tiles, inputs 0..63 and
// 64..127 of the chunk][codes: MATS x 128 rows x cbr bytes, cbr = 64 (4-bit,
// 64-byte TMA swizzle: 16-byte piece p of row r stored at p ^ ((r / 2) % 4),
// which spreads 8 consecutive rows reading the same piece over all banks) or
// 96 (6-bit, no swizzle)][scale words: MATS x 128 rows x 8 bytes, the bf16
// scales of the chunk's two groups, then their two biases].
__host__ __device__ constexpr int stage_bytes_of(int mats, int cbr) {
    return (kTileB + mats * kM * cbr + mats * kM * 8 + 1023) & ~1023;
}

__host__ __device__ constexpr int code_swz(int rr) { return (rr >> 1) & 3; }

__device__ __forceinline__ void bar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// arrive on the mbarrier once every earlier cp.async of this thread has landed
// (the barrier's count includes this arrival)
__device__ __forceinline__ void bar_arrive_cp_async(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// A work item: one expert, one block of 128 weight rows, token blocks z, z + ZB,
// ... of the expert's tokens. Only items with work are numbered: unique
// expert u (with at least thr tokens) owns items pref[u] .. pref[u + 1] - 1,
// RB x min(ZB, its token blocks) of them, row block fastest. CTA c of G takes
// items c, c + G, c + 2 G, ... (item costs differ by at most one token block).
struct TcItem {
    int e, off_e, cnt_e, r0, z, total;  // total: chunks (token blocks x chunks per row)
};

// the CTA's table of the unique experts, in shared memory: per unique expert u,
// {first item number pref[u], expert id, first slot, slot count}
struct TcGrid {
    int RB, ZB, U, nchunks, G, NI;
    const int4 *tab;  // [U]
};

// item k (or -1 past the last): a binary search over the table, shared memory only
__device__ __forceinline__ int tc_seek(const TcGrid &g, int k, TcItem &it) {
    if (k >= g.NI) return -1;
    int lo = 0, hi = g.U;                 // last u with pref[u] <= k
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.tab[mid].x <= k) lo = mid;
        else hi = mid;
    }
    const int4 t = g.tab[lo];
    const int local = k - t.x;
    it.e = t.y;
    it.off_e = t.z;
    it.cnt_e = t.w;
    it.r0 = (local % g.RB) * kM;
    it.z = local / g.RB;
    const int nblk = (it.cnt_e + kN - 1) / kN;
    it.total = ((nblk - it.z + g.ZB - 1) / g.ZB) * g.nchunks;
    return k;
}

// tm0, tm1: tensor maps of the code planes (gate and up, or down and unused),
// 2-D {row bytes, rows} with boxes of {cbr, 128}. The kernel is persistent: the
// ring, the A buffers and the two accumulators run on across item boundaries,
// so the next item's loads overlap this one's tail.
template <bool GATEUP, int S>
__global__ void __launch_bounds__(GATEUP ? 672 : 416, GATEUP ? 1 : 2)
    expert_tc_kernel(StepArgs a, Workspace ws, int thr, int ZB, int ucap, const __grid_constant__ CUtensorMap tm0,
                     const __grid_constant__ CUtensorMap tm1) {
    constexpr int MATS = GATEUP ? 2 : 1;
    constexpr int kDq = MATS * 256;            // dequantisation threads
    constexpr int kProdW = kDq / 32;           // first of the four producer warps
    constexpr int kMmaW = kProdW + 4;          // MMA warp
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned start of the dynamic area, as an offset into smem_raw
    // (so every access below stays a shared-memory access)
    unsigned char *base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // after a timeout anywhere in the launch, later CTAs do no work
    if (*reinterpret_cast<volatile unsigned *>(ws.status) & kDevErrTimeout) return;
    const int D = a.s.D, F = a.s.F;
    const int K = GATEUP ? D : F;            // reduction length
    const int rows_pe = GATEUP ? F : D;      // weight rows per expert
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const bool six = !GATEUP && a.s.down_bits == 6;
    const int cbr = six ? 96 : 64;           // code bytes per row and chunk
    const int stage_stride = stage_bytes_of(MATS, cbr);
    const int off_codes = kTileB;
    const int off_sc = kTileB + MATS * kM * cbr;
    const int groups = K / 64;               // scale/bias entries per row (even)

    unsigned char *ring = base;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + S * stage_stride);
    constexpr int NA = 2;                      // A buffers in tensor memory
    uint64_t *a_full = bars, *mma_done = bars + NA, *b_full = bars + 2 * NA, *b_empty = b_full + S;
    uint64_t *c_full = b_empty + S, *c_empty = c_full + S;
    uint64_t *acc_full = c_empty + S, *acc_empty = acc_full + 2;   // per accumulator
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
    int4 *tab = reinterpret_cast<int4 *>(tslot + 4);   // [ucap], 16-byte aligned

    // the item numbering: prefix over the unique experts of their items, with
    // each expert's id and slot range, into the table
    TcGrid g;
    g.RB = rows_pe / kM;
    g.ZB = ZB;
    g.U = *ws.U;
    g.nchunks = K / kK;
    g.G = (int)gridDim.x;
    g.tab = tab;
    if (g.U > ucap) {                        // more unique experts than selected slots: impossible
        if (tid == 0) report_error(ws.status, kDevErrInternal);
        return;
    }
    __shared__ int s_ni;
    if (warp == 0) {
        int run = 0;
        for (int u0 = 0; u0 < g.U; u0 += 32) {
            const int u = u0 + lane;
            int v = 0, e = 0, off = 0, cnt = 0;
            if (u < g.U) {
                e = ws.unique[u];
                off = ws.offsets[e];
                cnt = ws.offsets[e + 1] - off;
                v = cnt >= thr ? g.RB * min(ZB, (cnt + kN - 1) / kN) : 0;
            }
            int inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += t;
            }
            if (u < g.U) tab[u] = make_int4(run + inc - v, e, off, cnt);
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_ni = run;
    }
    __syncthreads();
    g.NI = s_ni;
    TcItem first;
    const int i0 = tc_seek(g, (int)blockIdx.x, first);
    if (i0 < 0) return;                      // no work for this CTA
    const int nchunks = g.nchunks;

    // tensor memory: two accumulators (gate and up, or y: 64 columns each per
    // matrix), token block b in accumulator b % 2, then the NA A buffers (MATS
    // tiles of 64 columns: 128 inputs, two f16 per column)
    constexpr uint32_t kCols = GATEUP ? 512 : 256;
    constexpr uint32_t kAccCols = MATS * kN;
    constexpr uint32_t kAcol = 2 * kAccCols;
    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NA; ++i) {
            bar_init(&a_full[i], kDq);
            bar_init(&mma_done[i], 1);
        }
        for (int i = 0; i < S; ++i) {
            bar_init(&b_full[i], 128);
            bar_init(&b_empty[i], 1);
            bar_init(&c_full[i], 1);
            bar_init(&c_empty[i], kDq);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(&acc_full[i], 1);
            bar_init(&acc_empty[i], kDq);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(tslot, kCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp >= kProdW && warp < kMmaW) {
        // ---- producers: codes (TMA), scales and B tiles -------------------------
        // B rows: x in f16 (y area, n x D) or h in f16 (first half of each h row)
        // producer warp pw, lane -> 16-byte piece j (of 16) of tokens 16 pw + tq + 2 i;
        // the tokens' row offsets (f16 elements, below 2^31 for every allowed
        // shape: n D <= 8192 x 16384, n k x 2 Dff <= 131072 x 16384) are looked
        // up once per token block
        const uint16_t *bsrc = reinterpret_cast<const uint16_t *>(GATEUP ? (const void *)ws.y : (const void *)ws.h);
        const int j = lane & 15, tq = 16 * (warp - kProdW) + (lane >> 4);
        // producer thread pt copies the scale and bias words of weight row pt of
        // each matrix: groups 2c and 2c + 1, 4 bytes each (through L1: the next
        // chunks read the same 32-byte sectors)
        const int pt = tid - kProdW * 32;
        const uint16_t *s_pl0 = GATEUP ? a.planes.gate_s : a.planes.down_s;
        const uint16_t *b_pl0 = GATEUP ? a.planes.gate_b : a.planes.down_b;
        uint32_t roff[kN / 8];
        size_t srow = 0;
        // chunk gidx of the CTA goes to ring stage sidx = gidx % S, in that
        // stage's use number gidx / S (parity sph)
        int gidx = 0, sidx = 0;
        uint32_t sph = 0;
        bool stop = false;
        TcItem it = first;
        for (int i = i0; i >= 0 && !stop; i = tc_seek(g, i + g.G, it)) {
            for (int li = 0, c = 0, blk = it.z; li < it.total; ++li) {
                if (c == 0) {
#pragma unroll
                    for (int q = 0; q < kN / 8; ++q) {
                        const int jj = blk * kN + tq + 2 * q;
                        // tokens past the expert's count are not copied: their
                        // accumulator columns are never read
                        roff[q] = jj >= it.cnt_e ? 0xFFFFFFFFu
                                  : GATEUP       ? (uint32_t)ws.slot_token[it.off_e + jj] * (uint32_t)D
                                                 : (uint32_t)(it.off_e + jj) * (uint32_t)(2 * F);
                    }
                    srow = ((size_t)it.e * rows_pe + it.r0 + pt) * groups;
                }
                if (gidx >= S) {
                    // the stage's previous use (parity sph ^ 1) has been consumed
                    if (!wait_bar(&b_empty[sidx], sph ^ 1u, ws.status) || !wait_bar(&c_empty[sidx], sph ^ 1u, ws.status))
                        *abort_flag = 1;
                }
                if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // warp-uniform
                    stop = true;
                    break;
                }
                unsigned char *st = ring + sidx * stage_stride;
                if (warp == kProdW && lane == 0) {
                    // the chunk's codes: one box of 128 rows x cbr bytes per matrix
                    tc::arrive_expect_tx(&c_full[sidx], (uint32_t)(MATS * kM * cbr));
                    const int y = it.e * rows_pe + it.r0;
                    tc::tma_load_2d(st + off_codes, &tm0, c * cbr, y, &c_full[sidx]);
                    if (GATEUP) tc::tma_load_2d(st + off_codes + kM * cbr, &tm1, c * cbr, y, &c_full[sidx]);
                }
                {
                    unsigned char *sd = st + off_sc + pt * 8;
                    tc::cp_async4(sd, s_pl0 + srow + 2 * c);
                    tc::cp_async4(sd + 4, b_pl0 + srow + 2 * c);
                    if (GATEUP) {
                        tc::cp_async4(sd + kM * 8, a.planes.up_s + srow + 2 * c);
                        tc::cp_async4(sd + kM * 8 + 4, a.planes.up_b + srow + 2 * c);
                    }
                }
                const uint16_t *src = bsrc + (size_t)c * kK + 8 * j;
                unsigned char *sub = st + (j >> 3) * kSubB;
#pragma unroll
                for (int q = 0; q < kN / 8; ++q)
                    if (roff[q] != 0xFFFFFFFFu) tc::cp_async16(sub + core_off(tq + 2 * q, j & 7), src + roff[q]);
                bar_arrive_cp_async(&b_full[sidx]);
                ++gidx;
                if (++sidx == S) {
                    sidx = 0;
                    sph ^= 1u;
                }
                if (++c == nchunks) {
                    c = 0;
                    blk += ZB;
                }
            }
        }
    } else if (warp == kMmaW) {
        // ---- MMA issue --------------------------------------------------------
        const uint32_t idesc = tc::idesc_f16_f32(kM, kN);
        // matrix descriptor of the first ring stage's B tile (a K step of 16
        // inputs adds 32 bytes, 2 in the start field)
        const uint64_t descB0 = tc::smem_desc_sw128(tc::smem_u32(ring), kSbo);
        // chunk gidx: ring stage sidx = gidx % S (use parity sph), A buffer
        // bsel = gidx % NA (use parity aph); token block gblk in accumulator
        // gblk % 2
        int issued = -1, gidx = 0, gblk = 0, sidx = 0, bsel = 0;
        uint32_t sph = 0, aph = 0;
        bool stop = false;
        TcItem it = first;
        for (int i = i0; i >= 0 && !stop; i = tc_seek(g, i + g.G, it)) {
            for (int li = 0, c = 0; li < it.total; ++li) {
                bool ok = wait_bar(&a_full[bsel], aph, ws.status);
                ok = ok && wait_bar(&b_full[sidx], sph, ws.status);
                // a block's first MMAs overwrite the accumulator of block gblk - 2,
                // whose epilogue (use (gblk / 2) - 1) must have read it
                if (ok && c == 0 && gblk >= 2)
                    ok = wait_bar(&acc_empty[gblk & 1], (((uint32_t)gblk >> 1) & 1u) ^ 1u, ws.status);
                if (!ok) *abort_flag = 1;
                if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // warp-uniform
                    stop = true;
                    break;
                }
                const uint64_t bd0 = descB0 + (uint64_t)((sidx * stage_stride) >> 4);
                const uint32_t a0 = tmem + kAcol + (uint32_t)(bsel * MATS * 64);
                const uint32_t d0 = tmem + (uint32_t)(gblk & 1) * kAccCols;
                __syncwarp();
                if (tc::elect_one()) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int ks = 0; ks < kK / 16; ++ks) {
                        // K step ks: sub-tile ks / 4 of B, 32 bytes per step inside it
                        const uint64_t bd = bd0 + (uint64_t)(((ks >> 2) * kSubB) >> 4) + 2 * (ks & 3);
#pragma unroll
                        for (int m = 0; m < MATS; ++m)
                            tc::mma_f16_ts(d0 + m * kN, a0 + (uint32_t)(m * 64 + ks * 8), bd, idesc,
                                           (c > 0 || ks > 0) ? 1u : 0u);
                    }
                    tc::commit(&mma_done[bsel]);
                    tc::commit(&b_empty[sidx]);
                    if (c == nchunks - 1) tc::commit(&acc_full[gblk & 1]);
                }
                __syncwarp();
                issued = gidx;
                ++gidx;
                if (++sidx == S) {
                    sidx = 0;
                    sph ^= 1u;
                }
                if (++bsel == NA) {
                    bsel = 0;
                    aph ^= 1u;
                }
                if (++c == nchunks) {
                    c = 0;
                    ++gblk;
                }
            }
        }
        // after an abort: wait (bounded) for the MMAs still in flight before
        // the tensor memory is freed
        if (*abort_flag && issued >= 0)
            wait_bar(&mma_done[issued % NA], (uint32_t)((issued / NA) & 1), ws.status);
    } else {
        // ---- dequantisation and epilogue ------------------------------------
        const int m = (warp >> 2) % MATS, gsel = warp / (4 * MATS);
        const int rr = 32 * (warp & 3) + lane;
        const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
        // The epilogue of token block pb runs one chunk late, after the next
        // chunk's dequantisation, so the block's last MMAs complete meanwhile
        // (the next block accumulates into the other accumulator). Its item
        // fields are kept: the next chunk may belong to the next item.
        bool pend = false;
        int p_b = 0, p_blk = 0, p_off = 0, p_cnt = 0, p_r0 = 0;
        auto epilogue = [&]() {
            if (!wait_bar(&acc_full[p_b & 1], ((uint32_t)p_b >> 1) & 1u, ws.status)) *abort_flag = 1;
            __syncwarp();
            tc::fence_after_sync();
            const uint32_t acc = tmem + tlane + (uint32_t)(p_b & 1) * kAccCols;
            constexpr int kTokW = kN / (kDq / 128);          // tokens per warp (16 or 32)
            const int t0 = kTokW * (warp >> 2);               // tokens [t0, t0 + kTokW) of the block
            const int r = p_r0 + rr;
#pragma unroll
            for (int hh = 0; hh < kTokW / 16; ++hh) {
                const int tc0 = t0 + 16 * hh;
                float gv[16];
                tc::ld_32x32b_x16(acc + tc0, gv);
                if (GATEUP) {
                    float uu[16];
                    tc::ld_32x32b_x16(acc + kN + tc0, uu);
                    // h row of the slot, f16 in the core order, in the first half of the f32 row
                    const int pos = (r & ~7) | core_pos(r & 7);
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int jj = p_blk * kN + tc0 + q;
                        if (jj < p_cnt)
                            reinterpret_cast<__half *>(ws.h + (size_t)(p_off + jj) * F)[pos] =
                                sat_h(glu_act<false>(a.s.act, a.s.act_limit, gv[q], uu[q]), ws.status);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int jj = p_blk * kN + tc0 + q;
                        if (jj < p_cnt) ws.y[(size_t)(p_off + jj) * D + r] = gv[q];
                    }
                }
            }
            tc::fence_before_sync();
            bar_arrive(&acc_empty[p_b & 1]);
        };
        // chunk gidx: ring stage sidx (use parity sph), A buffer bsel (use
        // parity aph), chunk c of the row pass over token block blk
        int gidx = 0, gblk = 0, sidx = 0, bsel = 0;
        uint32_t sph = 0, aph = 0;
        bool stop = false;
        TcItem it = first;
        for (int i = i0; i >= 0 && !stop; i = tc_seek(g, i + g.G, it)) {
            for (int li = 0, c = 0, blk = it.z; li < it.total; ++li) {
                const unsigned char *st = ring + sidx * stage_stride;
                // the chunk's codes (c_full) and its scale words (b_full: the
                // producers' copies of the stage)
                bool ok = wait_bar(&c_full[sidx], sph, ws.status) && wait_bar(&b_full[sidx], sph, ws.status);
                // A buffer bsel is free once the MMAs of chunk gidx - NA are done
                if (ok && gidx >= NA) ok = wait_bar(&mma_done[bsel], aph ^ 1u, ws.status);
                if (!ok) *abort_flag = 1;
                // warp-uniform: tcgen05.st and tcgen05.ld below are warp-collective
                if (__any_sync(0xffffffffu, *abort_flag != 0)) {
                    stop = true;
                    break;
                }
                {
                    // this row's scale and bias words of the chunk's two groups
                    const uint2 sbw = *reinterpret_cast<const uint2 *>(st + off_sc + (m * kM + rr) * 8);
                    float s = bf16f((uint16_t)(gsel ? sbw.x >> 16 : sbw.x & 0xFFFFu));
                    float b = bf16f((uint16_t)(gsel ? sbw.y >> 16 : sbw.y & 0xFFFFu));
                    if (fabsf(s) > 65504.0f || fabsf(b) > 65504.0f) {  // beyond f16: saturate, report
                        report_error(ws.status, kDevErrRange);
                        s = fminf(fmaxf(s, -65504.0f), 65504.0f);
                        b = fminf(fmaxf(b, -65504.0f), 65504.0f);
                    }
                    const __half2 s2 = __floats2half2_rn(s, s), b2 = __floats2half2_rn(b, b);
                    uint32_t o[32];
                    if (six) {
                        const unsigned char *cr = st + off_codes + (m * kM + rr) * 96 + 48 * gsel;
                        uint32_t v[12];
#pragma unroll
                        for (int q = 0; q < 3; ++q) {
                            const uint4 t4 = *reinterpret_cast<const uint4 *>(cr + 16 * q);
                            v[4 * q] = t4.x; v[4 * q + 1] = t4.y; v[4 * q + 2] = t4.z; v[4 * q + 3] = t4.w;
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint4 r4 = deq_6bit(v, q, s2, b2);
                            o[4 * q] = r4.x; o[4 * q + 1] = r4.y; o[4 * q + 2] = r4.z; o[4 * q + 3] = r4.w;
                        }
                    } else {
                        // 16-byte pieces 2 gsel and 2 gsel + 1 of the row's 64 bytes
                        const unsigned char *cr = st + off_codes + (m * kM + rr) * 64;
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(cr + 16 * ((2 * gsel) ^ code_swz(rr)));
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(cr + 16 * ((2 * gsel + 1) ^ code_swz(rr)));
                        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint4 r4 = deq_word(wv[q], s2, b2);
                            o[4 * q] = r4.x; o[4 * q + 1] = r4.y; o[4 * q + 2] = r4.z; o[4 * q + 3] = r4.w;
                        }
                    }
                    // two f16 per 32-bit column in the stored input order: columns
                    // 32 gsel .. 32 gsel + 31 of this matrix's A tile
                    const uint32_t ta = tmem + tlane + kAcol + (uint32_t)((bsel * MATS + m) * 64 + gsel * 32);
                    tc::st_32x32b_x16_async(ta, *reinterpret_cast<const uint32_t(*)[16]>(o));
                    tc::st_32x32b_x16_async(ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(o + 16));
                }
                // the codes and scale words of this stage have been read
                bar_arrive(&c_empty[sidx]);
                tc::wait_st();
                tc::fence_before_sync();
                bar_arrive(&a_full[bsel]);
                if (pend) {
                    epilogue();
                    pend = false;
                }
                if (c == nchunks - 1) {
                    pend = true;
                    p_b = gblk++;
                    p_blk = blk;
                    p_off = it.off_e;
                    p_cnt = it.cnt_e;
                    p_r0 = it.r0;
                }
                ++gidx;
                if (++sidx == S) {
                    sidx = 0;
                    sph ^= 1u;
                }
                if (++bsel == NA) {
                    bsel = 0;
                    aph ^= 1u;
                }
                if (++c == nchunks) {
                    c = 0;
                    blk += ZB;
                }
            }
        }
        // the last token block's epilogue (warp-uniform: it holds warp-collective loads)
        if (pend && !stop && !__any_sync(0xffffffffu, *abort_flag != 0)) epilogue();
    }
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---- router logits -----------------------------------------------------------------
// logits[t, e] = x[t] . Wr[e] (+ bias[e]) as a bf16 x bf16 -> f32 GEMM: per CTA
// 128 tokens (M) x 32 experts (N: more CTAs share the router matrix's read),
// K in chunks of 64 inputs (one 128-byte
// swizzled row per token or expert), both operands by TMA into a 4-stage ring,
// the accumulator in tensor memory. One thread issues the loads and the MMAs;
// the CTA's four warps read the accumulator back (lane = token) and add the
// bias. Products of bf16 are exact in f32; only the order of the f32 sum
// differs from the CUDA-core router, far inside the top-k margins.
constexpr int kRM = 128, kRN = 32, kRK = 64, kRS = 4;
constexpr int kRTileA = kRM * kRK * 2;    // 16 KB of x per stage
constexpr int kRTileB = kRN * kRK * 2;    // 4 KB of router rows per stage
constexpr int kRStage = kRTileA + kRTileB;

__global__ void __launch_bounds__(128, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                     const float *bias, float *logits, int n, int E, int D, unsigned *status) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + kRS * kRStage);
    uint64_t *empty = full + kRS, *acc = empty + kRS;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(acc + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRM, e0 = blockIdx.y * kRN, nk = D / kRK;
    if (tid == 0) {
        for (int i = 0; i < kRS; ++i) {
            bar_init(&full[i], 1);
            bar_init(&empty[i], 1);
        }
        bar_init(acc, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(tslot, kRN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    if (warp == 0) {
        if (tc::elect_one()) {
            const uint32_t idesc = tc::idesc_bf16_f32(kRM, kRN);
            auto load = [&](int kc) {
                unsigned char *st = base + (kc % kRS) * kRStage;
                tc::arrive_expect_tx(&full[kc % kRS], (uint32_t)kRStage);
                tc::tma_load_2d(st, &tmx, kc * kRK, t0, &full[kc % kRS]);
                tc::tma_load_2d(st + kRTileA, &tmw, kc * kRK, e0, &full[kc % kRS]);
            };
            int issued = 0, used = 0;
            bool ok = true;
            for (; issued < min(kRS - 1, nk); ++issued) load(issued);
            for (int kc = 0; kc < nk && ok; ++kc) {
                if (issued < nk) {
                    // the slot of chunk issued - kRS = kc - 1 is free once its MMAs are done
                    if (issued >= kRS)
                        ok = wait_bar(&empty[issued % kRS], (uint32_t)((issued / kRS - 1) & 1), status);
                    if (!ok) break;
                    load(issued++);
                }
                ok = wait_bar(&full[kc % kRS], (uint32_t)((kc / kRS) & 1), status);
                if (!ok) break;
                tc::fence_after_sync();
                const unsigned char *st = base + (kc % kRS) * kRStage;
                const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(st), kSbo);
                const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(st + kRTileA), kSbo);
#pragma unroll
                for (int ks = 0; ks < kRK / 16; ++ks)
                    tc::mma_f16(tmem, ad + 2 * ks, bd + 2 * ks, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
                tc::commit(&empty[kc % kRS]);
                used = kc + 1;
            }
            tc::commit(acc);  // arrives once every MMA issued above has completed
            // after a timeout: let the loads still in flight land before the CTA exits
            for (int i = used; i < issued; ++i) wait_bar(&full[i % kRS], (uint32_t)((i / kRS) & 1), status);
        }
        __syncwarp();
    }
    const bool done = wait_bar(acc, 0u, status);
    tc::fence_after_sync();
    const int t = t0 + 32 * warp + lane;   // this thread's TMEM lane = token
#pragma unroll 1
    for (int c = 0; c < kRN; c += 16) {
        float v[16];
        tc::ld_32x32b_x16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
        if (done && t < n) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = e0 + c + i;
                if (e < E) logits[(size_t)t * E + e] = v[i] + (bias ? bias[e] : 0.f);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kRN);
}

// ring stages per variant
constexpr int kStagesGateUp = 4;   // 4 x 34 KB (a fifth stage measured slower)
constexpr int kStagesDown = 3;     // 3 x 25 KB (6-bit 29 KB): two CTAs per SM

// alignment slack, ring, mbarriers (2 x 2 A-buffer, 4 x S ring, 2 x 2
// accumulator), tensor-memory slot and abort flag, then the table of at most
// ucap unique experts (16 bytes each)
size_t tc_smem_bytes(bool gateup, bool six, int ucap) {
    const int mats = gateup ? 2 : 1;
    const int S = gateup ? kStagesGateUp : kStagesDown;
    return 1024 + (size_t)S * stage_bytes_of(mats, six ? 96 : 64) + (4 + 4 * S + 4) * 8 + 16 + (size_t)ucap * 16;
}

// the driver's tensor-map encoder, resolved once (a function-local static is
// initialised once even when several host threads launch at the same time);
// null if the driver does not provide it
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        PFN_cuTensorMapEncodeTiled_v12000 r = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            r = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
        return r;
    }();
    return fn;
}

// a code plane [rows][row_bytes] as 2-D bytes with boxes of {cbr, 128 rows}
bool encode_code_plane(CUtensorMap *m, const void *base, long long row_bytes, long long rows, int cbr) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)cbr, (cuuint32_t)kM};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, cbr == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_variant_supported(const Shape &s) { return s.D % kM == 0 && s.F % kM == 0; }

cudaError_t launch_expert_tc(const StepArgs &a, const Workspace &ws, int thr, bool down, cudaStream_t st,
                             int &launched) {
    cudaError_t err;
    if (!down) {
        // x in f16, core order, into the y area
        const size_t items = (size_t)a.s.n * (a.s.D / 8);
        const int blocks = (int)((items + 255) / 256);
        if (a.s.x_dtype == MOE_DTYPE_F32)
            x_to_f16_kernel<MOE_DTYPE_F32><<<blocks, 256, 0, st>>>(a, ws);
        else
            x_to_f16_kernel<MOE_DTYPE_BF16><<<blocks, 256, 0, st>>>(a, ws);
        launched += 1;
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    const bool six = down && a.s.down_bits == 6;
    // unique experts: at most one per selected slot
    const int maxU = min(a.s.E, a.s.n * a.s.k);
    const size_t smem = tc_smem_bytes(!down, six, maxU);
    // tensor maps of the code planes (rows of D or Dff inputs)
    alignas(64) CUtensorMap tm0, tm1;
    const int K = down ? a.s.F : a.s.D;
    const long long rows = (long long)a.s.E * (down ? a.s.D : a.s.F);
    const int cbr = six ? 96 : 64;
    const long long row_bytes = six ? (long long)K * 3 / 4 : (long long)K / 2;
    if (!encode_code_plane(&tm0, down ? (const void *)a.planes.down_q : (const void *)a.planes.gate_q, row_bytes,
                           rows, cbr) ||
        !encode_code_plane(&tm1, down ? (const void *)a.planes.down_q : (const void *)a.planes.up_q, row_bytes,
                           rows, cbr))
        return cudaErrorInvalidValue;
    const void *k = down ? (const void *)expert_tc_kernel<false, kStagesDown>
                         : (const void *)expert_tc_kernel<true, kStagesGateUp>;
    if ((err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return err;
    // token-block slices: about 1.5x the mean tokens per selected expert, in
    // blocks of 64 (an item loops over its slice's blocks)
    const long mean = ((long)a.s.n * a.s.k + maxU - 1) / maxU;
    const int zb = (int)max(1L, min(8L, (3 * mean / 2 + kN - 1) / kN));
    // persistent: as many CTAs as fit at once (gate/up one per SM, down two),
    // at most one per item; SM counts cached per device (atomics: launches may
    // come from several host threads)
    static std::atomic<int> sm_count[64];
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) sms = sm_count[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) sm_count[dev].store(sms, std::memory_order_relaxed);
    }
    const long items = (long)((down ? a.s.D : a.s.F) / kM) * maxU * zb;
    const int grid = (int)min(items, (long)sms * (down ? 2 : 1));
    if (!down)
        expert_tc_kernel<true, kStagesGateUp><<<grid, 672, smem, st>>>(a, ws, thr, zb, maxU, tm0, tm1);
    else
        expert_tc_kernel<false, kStagesDown><<<grid, 416, smem, st>>>(a, ws, thr, zb, maxU, tm0, tm1);
    launched += 1;
    return cudaGetLastError();
}


bool router_tc_supported(const Shape &s) {
    return s.x_dtype == MOE_DTYPE_BF16 && s.w_dtype == MOE_DTYPE_BF16 && s.D % kRK == 0;
}

cudaError_t launch_router_tc(const StepArgs &a, const Workspace &ws, cudaStream_t st, int &launched) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cudaErrorInvalidValue;
    alignas(64) CUtensorMap tmx, tmw;
    // 2-D bf16 views {D, rows}, boxes of {64 inputs, 128 tokens or 32 experts},
    // 128-byte swizzle; rows past the end (tokens or experts) read as zeros
    auto enc = [&](CUtensorMap *m, const void *p, int rows, int box_rows) {
        cuuint64_t dims[2] = {(cuuint64_t)a.s.D, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)a.s.D * 2u};
        cuuint32_t box[2] = {(cuuint32_t)kRK, (cuuint32_t)box_rows};
        cuuint32_t es[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    // a map the driver declines: the CUDA-core router computes the same logits
    if (!enc(&tmx, a.x, a.s.n, kRM) || !enc(&tmw, a.router_w, a.s.E, kRN))
        return launch_router_logits(a, ws, st, launched);
    const int smem = 1024 + kRS * kRStage + 64;
    cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    dim3 grid((a.s.n + kRM - 1) / kRM, (a.s.E + kRN - 1) / kRN);
    router_tc_kernel<<<grid, 128, smem, st>>>(tmx, tmw, a.router_bias, ws.logits, a.s.n, a.s.E, a.s.D, ws.status);
    launched += 1;
    return cudaGetLastError();
}

}  // namespace moe
