// expert_tile_kernels.cu -- the tile variant of the expert MLP, for experts
// that at least mma_min_tokens tokens of the cohort selected.
//
// Where an expert serves many tokens the step is a real (small) matrix product,
// so these kernels dequantise each weight tile once into shared memory as f16
// (w = s*q + b in f32, rounded once; f16 keeps three more mantissa bits than
// bf16). A weight or activation beyond f16's range saturates at +-65504 and is
// reported (MOE_ERR_RANGE on the plan's next call); the f32 check path
// (MOE_FLAG_F32_DEBUG) has no such limit.
// and multiply it on the tensor cores against all of the expert's tokens at
// once: weights on M, tokens on N in n8 tiles (up to 64 tokens), f32
// accumulation. The GEMV kernels of the same launch sequence
// skip these experts, and these kernels skip the others, so every selected
// expert plane is still read once per step.
//
//   gate/up : h[p, f] = silu(sum_d Wg[e,f,d] x[t,d]) * sum_d Wu[e,f,d] x[t,d]
//   down    : y[p, d] = sum_f Wd[e,d,f] h[p,f]
// for the slots p of expert e (t = slot_token[p]); the combine kernel then sums
// y over each token's k slots in rank order.
//
// Sources: mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against
// 3.25x on dense" -- Leading hypothesis (group the cohort's rows by expert so
// that a wide expert becomes one matrix product, the sorted gather), and issue
// #1859 "perf(moe): attribute the MoE decode gap at the M = 1 expert gather" --
// Problem / Background (the slot-count switch between the gather GEMV and the
// sorted matrix path, taken here per expert instead of per call).
#include <cuda_fp16.h>

#include "activation.cuh"
#include "device_status.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {
namespace {

constexpr int kTR = 64;                // weight-tile rows per block (one MMA row tile per warp)
constexpr int kTT = 2 * kTR;           // threads per block: two per tile row (4 warps)
constexpr int kKC = 128;               // inputs per K chunk (two groups)
constexpr int kRowB = kKC * 2 + 16;    // shared row stride in bytes (ldmatrix without bank conflicts)
constexpr int kTokB = 64;              // tokens of one block pass (an expert's tokens in blocks of 64)
constexpr int kMaxNT = kTokB / 8;      // token tiles
constexpr int kSmemA = kTR * kRowB;    // weights: kTR rows x kKC f16
constexpr int kSmemX = kTokB * kRowB;
constexpr int kSmem = kSmemA + kSmemX;
static_assert(kTR * 65 * 4 <= kSmem, "the gate/up epilogue reuses the tile's shared memory");

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// two values as f16x2; a magnitude beyond the largest f16 saturates to
// +-65504 and is reported (MOE_ERR_RANGE on the plan's next call)
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi, unsigned *status) {
    if (fabsf(lo) > 65504.0f || fabsf(hi) > 65504.0f) {
        report_error(status, kDevErrRange);
        lo = fminf(fmaxf(lo, -65504.0f), 65504.0f);
        hi = fminf(fmaxf(hi, -65504.0f), 65504.0f);
    }
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// one group of one row (8 packed words, 64 inputs) dequantised to f16 at dst
__device__ __forceinline__ void dequant_group(const uint32_t *q, float s, float b, unsigned char *dst,
                                              unsigned *status) {
    const uint4 w0 = __ldg(reinterpret_cast<const uint4 *>(q));
    const uint4 w1 = __ldg(reinterpret_cast<const uint4 *>(q) + 1);
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = fmaf(s, (float)((w[i] >> (8 * j)) & 0xFu), b);
            const float hi = fmaf(s, (float)((w[i] >> (8 * j + 4)) & 0xFu), b);
            o[j] = pack_f16(lo, hi, status);
        }
        *reinterpret_cast<uint4 *>(dst + i * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// one group of one 6-bit row (48 bytes, a little-endian bit stream of 64
// codes) dequantised to f16 at dst
__device__ __forceinline__ void dequant_group6(const unsigned char *q, float s, float b, unsigned char *dst,
                                               unsigned *status) {
    const uint4 c0 = __ldg(reinterpret_cast<const uint4 *>(q));
    const uint4 c1 = __ldg(reinterpret_cast<const uint4 *>(q) + 1);
    const uint4 c2 = __ldg(reinterpret_cast<const uint4 *>(q) + 2);
    const uint32_t v[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float w2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int bit = 6 * (8 * i + 2 * j + h), wi = bit >> 5, sh = bit & 31;
                const uint32_t code = __funnelshift_r(v[wi], wi + 1 < 12 ? v[wi + 1] : 0u, sh) & 0x3Fu;
                w2[h] = fmaf(s, (float)code, b);
            }
            o[j] = pack_f16(w2[0], w2[1], status);
        }
        *reinterpret_cast<uint4 *>(dst + i * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// 8 consecutive activations as f16 (x may be f32 or bf16; h is f32)
__device__ __forceinline__ uint4 load8_f16(const void *p, size_t i, int dtype, unsigned *status) {
    float v[8];
    if (dtype == MOE_DTYPE_BF16) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + i));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        const float4 a = __ldg(q), b = __ldg(q + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    return make_uint4(pack_f16(v[0], v[1], status), pack_f16(v[2], v[3], status), pack_f16(v[4], v[5], status),
                      pack_f16(v[6], v[7], status));
}

// The shared K-chunk loop of both kernels: rows [16 w, 16 w + 16) of the
// kTR-row weight tile against the expert's NT token tiles.
//   load_w(r, half, dst): dequantise group `half` of the chunk for tile row r
//   load_x(j, piece, dst): 8 inputs (piece of the chunk) of the expert's j-th token
template <typename LW, typename LX>
__device__ __forceinline__ void tile_product(unsigned char *As, unsigned char *Xs, int K, int NT,
                                             LW load_w, LX load_x, float (&acc)[kMaxNT][4]) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k0 = 0; k0 < K; k0 += kKC) {
        {
            const int r = tid >> 1, half = tid & 1;
            load_w(r, k0 + half * kGroup, As + r * kRowB + half * 128);
        }
        for (int i = tid; i < NT * 8 * (kKC / 8); i += kTT) {
            const int j = i / (kKC / 8), piece = i - j * (kKC / 8);
            *reinterpret_cast<uint4 *>(Xs + j * kRowB + piece * 16) = load_x(j, k0 + piece * 8);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kKC; kk += 16) {
            uint32_t af[4];
            ptx::ldsm_x4(af, As + (16 * warp + (lane & 15)) * kRowB + (kk + (lane >> 4) * 8) * 2);
#pragma unroll
            for (int nt = 0; nt < kMaxNT; ++nt) {
                if (nt < NT) {
                    uint32_t bfr[2];
                    ptx::ldsm_x2(bfr, Xs + (nt * 8 + (lane & 7)) * kRowB + (kk + ((lane >> 3) & 1) * 8) * 2);
                    ptx::mma_f16_16816(acc[nt], af, bfr[0], bfr[1]);
                }
            }
        }
        __syncthreads();
    }
}

// block (kTR / 2 rows f of expert unique[blockIdx.y]): tile rows [0, kTR / 2) gate,
// [kTR / 2, kTR) up; the expert's tokens in blocks of 64 (blocks z, z + gridDim.z,
// ... for z = blockIdx.z), so a prefill expert with hundreds of tokens reuses
// each weight tile across them
__global__ void __launch_bounds__(kTT) gateup_tile_kernel(StepArgs a, Workspace ws, int thr) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int u = blockIdx.y;
    if (u >= *ws.U) return;
    const int e = ws.unique[u];
    const int off_e = ws.offsets[e], cnt_e = ws.offsets[e + 1] - off_e;
    if (cnt_e < thr) return;
    for (int tb = blockIdx.z; tb * kTokB < cnt_e; tb += gridDim.z) {
    const int off = off_e + tb * kTokB, cnt = min(kTokB, cnt_e - tb * kTokB);
    const int D = a.s.D, F = a.s.F, f0 = blockIdx.x * (kTR / 2);
    const int NT = (cnt + 7) / 8;
    unsigned char *As = sm, *Xs = sm + kSmemA;
    float acc[kMaxNT][4];
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    auto load_w = [&](int r, int k, unsigned char *dst) {
        const size_t row = (size_t)e * F + f0 + (r % (kTR / 2));
        const bool up = r >= kTR / 2;
        const uint32_t *q = (up ? a.planes.up_q : a.planes.gate_q) + row * (D / 8) + k / 8;
        const size_t gi = row * (D / kGroup) + k / kGroup;
        const float s = bf16f((up ? a.planes.up_s : a.planes.gate_s)[gi]);
        const float b = bf16f((up ? a.planes.up_b : a.planes.gate_b)[gi]);
        dequant_group(q, s, b, dst, ws.status);
    };
    auto load_x = [&](int j, int k) -> uint4 {
        if (j >= cnt) return make_uint4(0, 0, 0, 0);
        return load8_f16(a.x, (size_t)ws.slot_token[off + j] * D + k, a.s.x_dtype, ws.status);
    };
    tile_product(As, Xs, D, NT, load_w, load_x, acc);
    // accumulators -> shared [kTR rows][65] f32, then h = silu(gate) * up per (slot, f)
    float *E = reinterpret_cast<float *>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) {
        if (nt < NT) {
            const int r = 16 * warp + g, j = nt * 8 + 2 * c;
            E[r * 65 + j] = acc[nt][0];
            E[r * 65 + j + 1] = acc[nt][1];
            E[(r + 8) * 65 + j] = acc[nt][2];
            E[(r + 8) * 65 + j + 1] = acc[nt][3];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < cnt * (kTR / 2); i += kTT) {
        const int j = i / (kTR / 2), fr = i % (kTR / 2);
        const float gv = E[fr * 65 + j], uv = E[(kTR / 2 + fr) * 65 + j];
        ws.h[(size_t)(off + j) * F + f0 + fr] = glu_act<true>(a.s.act, a.s.act_limit, gv, uv);
    }
    __syncthreads();  // the next block's tiles overwrite the epilogue's shared memory
    }
}

// block (kTR rows d of expert unique[blockIdx.y]); token blocks as above
__global__ void __launch_bounds__(kTT) down_tile_kernel(StepArgs a, Workspace ws, int thr) {
    extern __shared__ __align__(16) unsigned char sm[];
    const int u = blockIdx.y;
    if (u >= *ws.U) return;
    const int e = ws.unique[u];
    const int off_e = ws.offsets[e], cnt_e = ws.offsets[e + 1] - off_e;
    if (cnt_e < thr) return;
    for (int tb = blockIdx.z; tb * kTokB < cnt_e; tb += gridDim.z) {
    const int off = off_e + tb * kTokB, cnt = min(kTokB, cnt_e - tb * kTokB);
    const int D = a.s.D, F = a.s.F, d0 = blockIdx.x * kTR;
    const int NT = (cnt + 7) / 8;
    unsigned char *As = sm, *Xs = sm + kSmemA;
    float acc[kMaxNT][4];
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    auto load_w = [&](int r, int k, unsigned char *dst) {
        const size_t row = (size_t)e * D + d0 + r;
        const size_t gi = row * (F / kGroup) + k / kGroup;
        if (a.s.down_bits == 6)
            dequant_group6(reinterpret_cast<const unsigned char *>(a.planes.down_q) + row * (3 * F / 4) + k / 64 * 48,
                           bf16f(a.planes.down_s[gi]), bf16f(a.planes.down_b[gi]), dst, ws.status);
        else
            dequant_group(a.planes.down_q + row * (F / 8) + k / 8, bf16f(a.planes.down_s[gi]),
                          bf16f(a.planes.down_b[gi]), dst, ws.status);
    };
    auto load_x = [&](int j, int k) -> uint4 {
        if (j >= cnt) return make_uint4(0, 0, 0, 0);
        return load8_f16(ws.h, (size_t)(off + j) * F + k, MOE_DTYPE_F32, ws.status);
    };
    tile_product(As, Xs, F, NT, load_w, load_x, acc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) {
        if (nt < NT) {
            const int r = d0 + 16 * warp + g, j = nt * 8 + 2 * c;
            if (j < cnt) {
                ws.y[(size_t)(off + j) * D + r] = acc[nt][0];
                ws.y[(size_t)(off + j) * D + r + 8] = acc[nt][2];
            }
            if (j + 1 < cnt) {
                ws.y[(size_t)(off + j + 1) * D + r] = acc[nt][1];
                ws.y[(size_t)(off + j + 1) * D + r + 8] = acc[nt][3];
            }
        }
    }
    }
}

}  // namespace

bool tile_variant_supported(const Shape &s) { return s.D % 128 == 0 && s.F % 128 == 0; }

cudaError_t launch_expert_tiles(const StepArgs &a, const Workspace &ws, int thr, bool down,
                                cudaStream_t st, int &launched) {
    cudaError_t err = cudaFuncSetAttribute(down ? (const void *)down_tile_kernel : (const void *)gateup_tile_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (err != cudaSuccess) return err;
    const int maxU = min(a.s.E, a.s.n * a.s.k);
    // token blocks per expert in the grid (each block loops over the rest): an
    // expert holds at most n tokens
    const int zb = min((a.s.n + kTokB - 1) / kTokB, 8);
    if (!down) {
        gateup_tile_kernel<<<dim3(a.s.F / (kTR / 2), maxU, zb), kTT, kSmem, st>>>(a, ws, thr);
    } else {
        down_tile_kernel<<<dim3(a.s.D / kTR, maxU, zb), kTT, kSmem, st>>>(a, ws, thr);
    }
    launched += 1;
    return cudaGetLastError();
}

}  // namespace moe
