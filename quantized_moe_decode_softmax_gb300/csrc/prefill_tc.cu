// prefill_tc.cu -- the prefill path's expert GEMMs on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory).
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
// Per CTA: one expert, 128 weight rows, 64 of the expert's tokens at a time,
// K (the reduction) in chunks of 64 inputs = one quantisation group:
//   - a ring of S stages holds, per chunk, the B tile, the raw codes and the
//     scale/bias words of the CTA's rows, filled S - 1 chunks ahead;
//   - the CUDA cores dequantise chunk i into one of two A tiles while the
//     tensor core runs chunk i - 1 (one thread issues M = 128, N = 64, K = 16
//     MMAs and commits them to an mbarrier);
//   - after the last chunk of a token block, tcgen05.ld brings the f32
//     accumulators to registers: h = act(gate, up) (gate row r and up row r
//     are both tensor-memory lane r) or y for the down projection.
// An operand beyond f16's range saturates and is reported (MOE_ERR_RANGE);
// every mbarrier wait gives up after 1 s and reports a timeout.
#include <cuda_fp16.h>

#include "activation.cuh"
#include "device_status.cuh"
#include "moe_internal.h"
#include "prefill_tc.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kM = 128;          // weight rows per A tile
constexpr int kN = 64;           // tokens per block
constexpr int kK = 64;           // inputs per chunk
constexpr int kSbo = 1024;       // bytes between 8-row swizzle atoms (8 rows x 128 B)
constexpr int kTileB = kN * kK * 2;   // 8 KB: one f16 activation tile
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
// code j at bits 4j): the pairs (0,4) (1,5) (2,6) (3,7), each w = s q + b
__device__ __forceinline__ uint4 deq_word(uint32_t w, __half2 s2, __half2 b2) {
    const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t v = ((w >> (4 * p)) & 0x000F000Fu) | 0x64006400u;  // 1024 + q, exact
        const __half2 q = __hsub2(*reinterpret_cast<const __half2 *>(&v), k1024);
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
// Ring stage layout (bytes): [B tile 8 KB][codes: MATS x 128 rows x cb][scale
// and bias words: MATS x 128 rows x 2 x 4 B]. Codes of 4-bit rows are two
// 16-byte halves, swapped on rows 4..7 of every 8 (no shared-memory bank
// conflicts when 8 consecutive rows read the same half).
__host__ __device__ constexpr int stage_bytes_of(int mats, int cb) {
    return (kTileB + mats * kM * cb + mats * kM * 8 + 1023) & ~1023;
}

__host__ __device__ constexpr int code_swz(int rr) { return (rr >> 2) & 1; }

// GATEUP: gate and up rows (two A tiles, two accumulators), x as B, epilogue
// h = act(g, u) written as f16; else the down projection: Wd rows, h as B,
// epilogue y (f32). S: ring stages. One dequantisation item (matrix, row, half
// of the row's 8 pieces) per thread: 512 threads for gate/up, 256 for down.
template <bool GATEUP, int S>
__global__ void __launch_bounds__(GATEUP ? 512 : 256, 1) expert_tc_kernel(StepArgs a, Workspace ws, int thr) {
    constexpr int MATS = GATEUP ? 2 : 1;
    constexpr int kThr = MATS * 256;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~static_cast<uintptr_t>(1023));
    const int u = blockIdx.y;
    if (u >= *ws.U) return;
    // after a timeout anywhere in the launch, later blocks do no work
    if (*reinterpret_cast<volatile unsigned *>(ws.status) & kDevErrTimeout) return;
    const int e = ws.unique[u];
    const int off_e = ws.offsets[e], cnt_e = ws.offsets[e + 1] - off_e;
    if (cnt_e < thr) return;
    const int nblk = (cnt_e + kN - 1) / kN;
    if ((int)blockIdx.z >= nblk) return;
    const int my_blocks = (nblk - (int)blockIdx.z + (int)gridDim.z - 1) / (int)gridDim.z;

    const int D = a.s.D, F = a.s.F;
    const int K = GATEUP ? D : F;            // reduction length
    const int nchunks = K / kK;
    const int r0 = blockIdx.x * kM;          // first weight row (gate/up: f; down: d)
    const int tid = threadIdx.x;
    const bool six = !GATEUP && a.s.down_bits == 6;
    const int cb = six ? 48 : 32;            // code bytes per row and chunk
    const int stage_stride = stage_bytes_of(MATS, cb);
    const int off_codes = kTileB, off_sc = kTileB + MATS * kM * cb;

    unsigned char *ring = base;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base + S * stage_stride);  // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

    if (tid == 0) {
        *abort_flag = 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc::smem_u32(&bar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc::smem_u32(&bar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // tensor memory: accumulators (gate, up or y: 64 columns each), then the
    // two A buffers (MATS tiles of 32 columns each)
    constexpr uint32_t kCols = GATEUP ? 256 : 128;
    constexpr uint32_t kAcol = MATS * kN;
    if ((tid >> 5) == 0) tc::tmem_alloc(tslot, kCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    const uint32_t *q0 = GATEUP ? a.planes.gate_q : a.planes.down_q;
    const uint16_t *s0 = GATEUP ? a.planes.gate_s : a.planes.down_s;
    const uint16_t *b0 = GATEUP ? a.planes.gate_b : a.planes.down_b;
    const size_t rows_per_e = GATEUP ? (size_t)F : (size_t)D;
    const size_t groups = (size_t)K / 64;    // scale/bias entries per row (even: K % 128 == 0)
    // B rows: x in f16 (y area, n x D) or h in f16 (first half of each h row)
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(ws.y);
    const uint16_t *hb = reinterpret_cast<const uint16_t *>(ws.h);

    const int total = my_blocks * nchunks;
    // fill ring stage idx % S with chunk idx (token block, chunk) -- or, past
    // the end, commit an empty group so the wait counts stay uniform
    auto issue = [&](int idx) {
        if (idx < total) {
            const int blk = (int)blockIdx.z + (idx / nchunks) * (int)gridDim.z, c = idx % nchunks;
            unsigned char *st = ring + (idx % S) * stage_stride;
            // B: 64 tokens x 8 cores of 16 bytes (tokens past the expert's count
            // are not copied: their accumulator columns are never read)
            for (int p = tid; p < kN * 8; p += kThr) {
                const int t = p >> 3, j = p & 7, jj = blk * kN + t;
                if (jj >= cnt_e) continue;
                const uint16_t *src = GATEUP ? xb + (size_t)ws.slot_token[off_e + jj] * D
                                             : hb + (size_t)(off_e + jj) * F * 2;
                tc::cp_async16(st + core_off(t, j), src + (size_t)c * kK + 8 * j);
            }
            // codes: MATS x 128 rows x cb bytes
            const int pr = cb / 16;
            for (int p = tid; p < MATS * kM * pr; p += kThr) {
                const int m = p / (kM * pr), rr = (p / pr) % kM, h = p % pr;
                const size_t row = (size_t)e * rows_per_e + r0 + rr;
                const unsigned char *src;
                if (six) {
                    src = reinterpret_cast<const unsigned char *>(a.planes.down_q) + row * ((size_t)K * 3 / 4) +
                          (size_t)c * 48 + h * 16;
                } else {
                    const uint32_t *qq = (GATEUP && m) ? a.planes.up_q : q0;
                    src = reinterpret_cast<const unsigned char *>(qq + row * ((size_t)K / 8) + (size_t)c * 8) + h * 16;
                }
                const int hd = six ? h : (h ^ code_swz(rr));
                tc::cp_async16(st + off_codes + (m * kM + rr) * cb + hd * 16, src);
            }
            // scale and bias: the 4-byte word holding entry (row, c) of each
            for (int p = tid; p < MATS * kM * 2; p += kThr) {
                const int m = p / (kM * 2), rr = (p >> 1) % kM, arr = p & 1;
                const size_t gi = ((size_t)e * rows_per_e + r0 + rr) * groups + c;
                const uint16_t *sp = (GATEUP && m) ? (arr ? a.planes.up_b : a.planes.up_s) : (arr ? b0 : s0);
                tc::cp_async4(st + off_sc + ((m * kM + rr) * 2 + arr) * 4, sp + (gi & ~(size_t)1));
            }
        }
        tc::cp_async_commit();
    };
    for (int i = 0; i < S - 1; ++i) issue(i);

    const uint32_t idesc = tc::idesc_f16_f32(kM, kN);
    // matrix descriptor of the first ring stage's B tile (a K step of 16 inputs
    // adds 32 bytes, 2 in the start field)
    const uint64_t descB0 = tc::smem_desc_sw128(tc::smem_u32(ring), kSbo);
    // dequantisation: warp -> (lane quadrant q, matrix m, half of the row's 8
    // pieces); lane -> row 32 q + lane, the tensor-memory lane of that row
    const int warp = tid >> 5, lane = tid & 31;
    const int dq_m = (warp >> 2) % MATS, dq_half = warp / (4 * MATS);
    const int dq_rr = 32 * (warp & 3) + lane;
    const uint32_t dq_lane = (uint32_t)(32 * (warp & 3)) << 16;
    int issued = -1;  // the last chunk whose MMAs were committed
    for (int idx = 0; idx < total; ++idx) {
        const int bsel = idx & 1, c = idx % nchunks, blk = (int)blockIdx.z + (idx / nchunks) * (int)gridDim.z;
        const unsigned char *st = ring + (idx % S) * stage_stride;
        tc::cp_async_wait<S - 2>();
        __syncthreads();
        // dequantise this thread's 32 inputs into its lane of A buffer bsel
        {
            const int m = dq_m, rr = dq_rr, half = dq_half;
            const uint32_t *scw = reinterpret_cast<const uint32_t *>(st + off_sc) + (m * kM + rr) * 2;
            const int sh = (c & 1) * 16;
            float s = bf16f((uint16_t)(scw[0] >> sh)), b = bf16f((uint16_t)(scw[1] >> sh));
            if (fabsf(s) > 65504.0f || fabsf(b) > 65504.0f) {  // beyond f16: saturate, report
                report_error(ws.status, kDevErrRange);
                s = fminf(fmaxf(s, -65504.0f), 65504.0f);
                b = fminf(fmaxf(b, -65504.0f), 65504.0f);
            }
            const __half2 s2 = __floats2half2_rn(s, s), b2 = __floats2half2_rn(b, b);
            const unsigned char *cr = st + off_codes + (m * kM + rr) * cb;
            uint32_t o[16];
            if (six) {
                uint32_t v[12];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const uint4 t4 = *reinterpret_cast<const uint4 *>(cr + 16 * i);
                    v[4 * i] = t4.x; v[4 * i + 1] = t4.y; v[4 * i + 2] = t4.z; v[4 * i + 3] = t4.w;
                }
                // compile-time core indices keep v[] in registers
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 r4 = half ? deq_6bit(v, 4 + j, s2, b2) : deq_6bit(v, j, s2, b2);
                    o[4 * j] = r4.x; o[4 * j + 1] = r4.y; o[4 * j + 2] = r4.z; o[4 * j + 3] = r4.w;
                }
            } else {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(cr + 16 * (half ^ code_swz(rr)));
                const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 r4 = deq_word(wv[j], s2, b2);
                    o[4 * j] = r4.x; o[4 * j + 1] = r4.y; o[4 * j + 2] = r4.z; o[4 * j + 3] = r4.w;
                }
            }
            // two f16 per 32-bit column in the stored input order
            tc::st_32x32b_x16(tmem + dq_lane + kAcol + (uint32_t)((bsel * MATS + m) * 32 + half * 16), o);
        }
        tc::fence_before_sync();
        __syncthreads();
        if ((tid >> 5) == 0) {
            // warp 0 forms the descriptors (warp-uniform), one elected lane issues
            const uint64_t bd0 = descB0 + (uint64_t)(((idx % S) * stage_stride) >> 4);
            const uint32_t a0 = tmem + kAcol + (uint32_t)(bsel * MATS * 32);
            if (tc::elect_one()) {
                tc::fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < kK / 16; ++ks) {
#pragma unroll
                    for (int m = 0; m < MATS; ++m)
                        tc::mma_f16_ts(tmem + m * kN, a0 + (uint32_t)(m * 32 + ks * 8), bd0 + 2 * ks, idesc,
                                       (c > 0 || ks > 0) ? 1u : 0u);
                }
                tc::commit(&bar[bsel]);
            }
            __syncwarp();
        }
        issued = idx;
        // the MMAs of chunk idx - 1 have read their A tile and ring stage: the
        // stage takes chunk idx + S - 1, the A tile chunk idx + 1
        if (idx >= 1 && !wait_bar(&bar[(idx - 1) & 1], (uint32_t)(((idx - 1) >> 1) & 1), ws.status))
            *abort_flag = 1;
        issue(idx + S - 1);
        if (c == nchunks - 1) {
            // epilogue of this token block, once its last MMAs have completed
            if (!wait_bar(&bar[bsel], (uint32_t)((idx >> 1) & 1), ws.status)) *abort_flag = 1;
            tc::fence_after_sync();
            const int rr = 32 * (warp & 3) + lane;          // this thread's TMEM lane = weight row
            constexpr int kTokW = kN / (kThr / 128);         // tokens per warp (32 or 16)
            const int t0 = kTokW * (warp >> 2);              // tokens [t0, t0 + kTokW) of the block
            const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
            const int r = r0 + rr;
#pragma unroll
            for (int half = 0; half < kTokW / 16; ++half) {
                const int tc0 = t0 + 16 * half;
                float g[16];
                tc::ld_32x32b_x16(ta + tc0, g);
                if (GATEUP) {
                    float uu[16];
                    tc::ld_32x32b_x16(ta + kN + tc0, uu);
                    // h row of the slot, f16 in the core order, in the first half of the f32 row
                    const int pos = (r & ~7) | core_pos(r & 7);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int j = blk * kN + tc0 + i;
                        if (j < cnt_e)
                            reinterpret_cast<__half *>(ws.h + (size_t)(off_e + j) * F)[pos] =
                                sat_h(glu_act<true>(a.s.act, a.s.act_limit, g[i], uu[i]), ws.status);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int j = blk * kN + tc0 + i;
                        if (j < cnt_e) ws.y[(size_t)(off_e + j) * D + r] = g[i];
                    }
                }
            }
            tc::fence_before_sync();
        }
        __syncthreads();  // abort flag; the next block's MMAs overwrite the accumulators
        if (*abort_flag) break;
    }
    // after a timeout: wait (bounded) for the MMAs still in flight before the
    // tensor memory is freed
    if (*abort_flag && issued >= 0) wait_bar(&bar[issued & 1], (uint32_t)((issued >> 1) & 1), ws.status);
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if ((tid >> 5) == 0) tc::tmem_dealloc(tmem, kCols);
}

// ring stages per variant (the ring is all of the shared memory)
constexpr int kStagesGateUp = 8;   // 8 x 18 KB
constexpr int kStagesDown = 8;     // 8 x 13 KB (two CTAs per SM) or 15 KB (6-bit)

size_t tc_smem_bytes(bool gateup, int cb) {
    const int mats = gateup ? 2 : 1;
    const int S = gateup ? kStagesGateUp : kStagesDown;
    return 1024 + (size_t)S * stage_bytes_of(mats, cb) + 64;
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
    const int cb = (down && a.s.down_bits == 6) ? 48 : 32;
    const size_t smem = tc_smem_bytes(!down, cb);
    const void *k = down ? (const void *)expert_tc_kernel<false, kStagesDown>
                         : (const void *)expert_tc_kernel<true, kStagesGateUp>;
    if ((err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return err;
    const int maxU = min(a.s.E, a.s.n * a.s.k);
    // token-block slices: about 1.5x the mean tokens per selected expert, in
    // blocks of 64 (a CTA loops over its slice's blocks; empty CTAs exit)
    const long mean = ((long)a.s.n * a.s.k + maxU - 1) / maxU;
    const int zb = (int)max(1L, min(8L, (3 * mean / 2 + kN - 1) / kN));
    if (!down)
        expert_tc_kernel<true, kStagesGateUp><<<dim3(a.s.F / kM, maxU, zb), 512, smem, st>>>(a, ws, thr);
    else
        expert_tc_kernel<false, kStagesDown><<<dim3(a.s.D / kM, maxU, zb), 256, smem, st>>>(a, ws, thr);
    launched += 1;
    return cudaGetLastError();
}

}  // namespace moe
