// expert_f32_kernels.cu -- the GEMV variant of the grouped path's expert half.
// Every weight is dequantised exactly to f32 (w = s*q + b) and every product
// is accumulated in f32 on the CUDA cores. It serves the experts below the
// tensor-core threshold (mma_min_tokens) of the grouped and prefill paths, every
// expert of a shape the tcgen05 GEMMs decline, and every expert under
// MOE_FLAG_F32_DEBUG, where it is held to 1e-4 of RMS(out) against the oracle.
// launch_experts (end of this file) runs the tcgen05 GEMMs, these kernels and
// the combine for a step.
//
// Stages (one launch each), over the de-duplicated expert list:
//   gate/up : h[p, f] = act(sum_d Wg[e,f,d] x[t,d], sum_d Wu[e,f,d] x[t,d])
//             (activation.cuh; SwiGLU by default)
//   down    : y[p, d] = sum_f Wd[e,d,f] h[p,f]
//   combine : out[t, d] = sum_{j<k} w[t,j] * y[slot_of(t,j), d], j ascending
// where p runs over the slots grouped under expert e and t = slot_token[p].
//
// Sources: mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against
// 3.25x on dense" -- Current Behavior (SwitchGLU experts, moe_weighted_sum,
// 4-bit group 64), Implementation Notes (f32 partials, a single final
// rounding, parity against an all-f32 dense reference).
#include <cuda_bf16.h>

#include "activation.cuh"
#include "moe_internal.h"
#include "prefill_tc.h"
#include "routing.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

template <int DT>
__device__ __forceinline__ void ld8(const void *p, size_t i, float (&v)[8]) {
    if (DT == MOE_DTYPE_F32) {
        const float4 *q = reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        float4 a = __ldg(q), b = __ldg(q + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        uint4 a = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(p) + i));
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

// exact f32 value of a 4-bit code: the code ORed into the mantissa of 2^23,
// minus 2^23
__device__ __forceinline__ float code_f32(uint32_t word, int j) {
    return __uint_as_float(0x4B000000u | ((word >> (4 * j)) & 0xFu)) - 8388608.0f;
}

// w[j] = s * q_j + b for the 8 codes of one packed word
__device__ __forceinline__ void deq8(uint32_t q, float s, float b, float (&w)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = fmaf(s, code_f32(q, j), b);
}

constexpr int kTok = 8;             // tokens per pass (accumulators per thread and matrix)
constexpr int kRowThreads = 256;    // one thread per weight row
constexpr int kStageBytes = 65536;  // activations of one pass in shared memory, at most

// tokens per pass for a K-long activation row staged as f32
__host__ __device__ inline int pass_tokens(int K) {
    const int t = kStageBytes / (K * 4);
    return t < 1 ? 1 : t > kTok ? kTok : t;
}

// One thread's gate and up rows against NT staged tokens (cnt <= NT of them
// real): accumulators ag/au per token. The next group's codes and scales are
// loaded before the current group is computed.
template <int NT>
__device__ __forceinline__ void gateup_row(const uint4 *gq, const uint4 *uq, const uint16_t *gs,
                                           const uint16_t *gb, const uint16_t *us, const uint16_t *ub,
                                           const float *xs, int D, int cnt, float (&ag)[kTok],
                                           float (&au)[kTok]) {
    const int G = D / kGroup;
    uint4 ng0 = __ldg(gq), ng1 = __ldg(gq + 1), nu0 = __ldg(uq), nu1 = __ldg(uq + 1);
    uint16_t nsg = gs[0], nbg = gb[0], nsu = us[0], nbu = ub[0];
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const uint4 cg[2] = {ng0, ng1}, cu[2] = {nu0, nu1};
        const float sg = bf16f(nsg), bg = bf16f(nbg), su = bf16f(nsu), bu = bf16f(nbu);
        if (g + 1 < G) {
            ng0 = __ldg(gq + 2 * g + 2);
            ng1 = __ldg(gq + 2 * g + 3);
            nu0 = __ldg(uq + 2 * g + 2);
            nu1 = __ldg(uq + 2 * g + 3);
            nsg = gs[g + 1];
            nbg = gb[g + 1];
            nsu = us[g + 1];
            nbu = ub[g + 1];
        }
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const uint32_t wg4[4] = {cg[hq].x, cg[hq].y, cg[hq].z, cg[hq].w};
            const uint32_t wu4[4] = {cu[hq].x, cu[hq].y, cu[hq].z, cu[hq].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float wg[8], wu[8];
                deq8(wg4[w], sg, bg, wg);
                deq8(wu4[w], su, bu, wu);
                const int k0 = g * kGroup + hq * 32 + w * 8;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (NT == 1 || t < cnt) {
                        const float4 x0 = *reinterpret_cast<const float4 *>(xs + (size_t)t * D + k0);
                        const float4 x1 = *reinterpret_cast<const float4 *>(xs + (size_t)t * D + k0 + 4);
                        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            ag[t] = fmaf(wg[j], xv[j], ag[t]);
                            au[t] = fmaf(wu[j], xv[j], au[t]);
                        }
                    }
                }
            }
        }
    }
}

// Thread per gate/up row f of expert unique[blockIdx.y] (experts with at
// least `thr` tokens are left to the tcgen05 GEMMs when thr > 0). Per pass of up
// to T of the expert's slots, the block stages their activations as f32 in
// shared memory; every thread then walks its two rows (gate and up) in 16-byte
// code loads, dequantises each weight exactly and accumulates its products
// with every staged token (the warp's threads read the same activation, so the
// shared-memory reads are broadcasts and no cross-thread sum is needed). The
// token loop is specialised for 1, 2, 4 or 8 tokens, so a pass issues work for
// at most twice its tokens.
template <int XT>
__global__ void __launch_bounds__(kRowThreads) gateup_f32_kernel(StepArgs a, Workspace ws, int thr, int T) {
    extern __shared__ float4 xs4[];
    float *xs = reinterpret_cast<float *>(xs4);  // [T][D]
    const int u = blockIdx.y;
    const int D = a.s.D, F = a.s.F;
    if (u >= *ws.U) return;
    const int e = ws.unique[u];
    const int p_begin = ws.offsets[e], p_end = ws.offsets[e + 1];
    if (thr > 0 && p_end - p_begin >= thr) return;
    const int f = blockIdx.x * kRowThreads + threadIdx.x;
    const bool has_row = f < F;
    const size_t row = (size_t)e * F + (has_row ? f : F - 1);
    const uint4 *gq = reinterpret_cast<const uint4 *>(a.planes.gate_q + row * (D / 8));
    const uint4 *uq = reinterpret_cast<const uint4 *>(a.planes.up_q + row * (D / 8));
    const uint16_t *gs = a.planes.gate_s + row * (D / kGroup);
    const uint16_t *gb = a.planes.gate_b + row * (D / kGroup);
    const uint16_t *us = a.planes.up_s + row * (D / kGroup);
    const uint16_t *ub = a.planes.up_b + row * (D / kGroup);
    for (int p0 = p_begin; p0 < p_end; p0 += T) {
        const int cnt = min(T, p_end - p0);
        __syncthreads();  // the previous pass is done with xs
        for (int i = threadIdx.x; i < cnt * (D / 8); i += kRowThreads) {
            const int t = i / (D / 8), c8 = i - t * (D / 8);
            float v[8];
            ld8<XT>(a.x, (size_t)ws.slot_token[p0 + t] * D + (size_t)c8 * 8, v);
            float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)t * D + c8 * 8);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        __syncthreads();
        if (!has_row) continue;
        float ag[kTok], au[kTok];
#pragma unroll
        for (int t = 0; t < kTok; ++t) ag[t] = au[t] = 0.f;
        if (cnt == 1)
            gateup_row<1>(gq, uq, gs, gb, us, ub, xs, D, cnt, ag, au);
        else if (cnt == 2)
            gateup_row<2>(gq, uq, gs, gb, us, ub, xs, D, cnt, ag, au);
        else if (cnt <= 4)
            gateup_row<4>(gq, uq, gs, gb, us, ub, xs, D, cnt, ag, au);
        else
            gateup_row<kTok>(gq, uq, gs, gb, us, ub, xs, D, cnt, ag, au);
#pragma unroll
        for (int t = 0; t < kTok; ++t)
            if (t < cnt) ws.h[(size_t)(p0 + t) * F + f] = glu_act<true>(a.s.act, a.s.act_limit, ag[t], au[t]);
    }
}

// One thread's down row against NT staged h rows (cnt <= NT of them real).
template <int NT>
__device__ __forceinline__ void down_row(const uint4 *dq, const uint16_t *ds, const uint16_t *db,
                                         const float *hs, int F, int cnt, float (&acc)[kTok]) {
    const int G = F / kGroup;
    uint4 n0 = __ldg(dq), n1 = __ldg(dq + 1);
    uint16_t ns = ds[0], nb = db[0];
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const uint4 c[2] = {n0, n1};
        const float sd = bf16f(ns), bd = bf16f(nb);
        if (g + 1 < G) {
            n0 = __ldg(dq + 2 * g + 2);
            n1 = __ldg(dq + 2 * g + 3);
            ns = ds[g + 1];
            nb = db[g + 1];
        }
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            const uint32_t w4[4] = {c[hq].x, c[hq].y, c[hq].z, c[hq].w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                float wd[8];
                deq8(w4[w], sd, bd, wd);
                const int k0 = g * kGroup + hq * 32 + w * 8;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (NT == 1 || t < cnt) {
                        const float4 h0 = *reinterpret_cast<const float4 *>(hs + (size_t)t * F + k0);
                        const float4 h1 = *reinterpret_cast<const float4 *>(hs + (size_t)t * F + k0 + 4);
                        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[t] = fmaf(wd[j], hv[j], acc[t]);
                    }
                }
            }
        }
    }
}

// 6-bit down rows: one group of 64 codes is 48 bytes of a little-endian bit
// stream (code j at bits 6j..6j+5); w = s * q + b exactly in f32.
__device__ __forceinline__ void deq64_6bit(const uint4 (&c)[3], float s, float b, float (&w)[64]) {
    const uint32_t v[12] = {c[0].x, c[0].y, c[0].z, c[0].w, c[1].x, c[1].y,
                            c[1].z, c[1].w, c[2].x, c[2].y, c[2].z, c[2].w};
#pragma unroll
    for (int j = 0; j < 64; ++j) {
        const int bit = 6 * j, wi = bit >> 5, sh = bit & 31;
        const uint32_t lo = v[wi], hi = wi + 1 < 12 ? v[wi + 1] : 0u;
        const uint32_t q = __funnelshift_r(lo, hi, sh) & 0x3Fu;
        w[j] = fmaf(s, __uint_as_float(0x4B000000u | q) - 8388608.0f, b);
    }
}

template <int NT>
__device__ __forceinline__ void down_row6(const unsigned char *dq, const uint16_t *ds, const uint16_t *db,
                                          const float *hs, int F, int cnt, float (&acc)[kTok]) {
    const int G = F / kGroup;
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const uint4 *p = reinterpret_cast<const uint4 *>(dq + (size_t)g * 48);
        const uint4 c[3] = {__ldg(p), __ldg(p + 1), __ldg(p + 2)};
        float wd[64];
        deq64_6bit(c, bf16f(ds[g]), bf16f(db[g]), wd);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (NT == 1 || t < cnt) {
                const float *hr = hs + (size_t)t * F + g * kGroup;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const float4 h4 = *reinterpret_cast<const float4 *>(hr + j);
                    acc[t] = fmaf(wd[j], h4.x, acc[t]);
                    acc[t] = fmaf(wd[j + 1], h4.y, acc[t]);
                    acc[t] = fmaf(wd[j + 2], h4.z, acc[t]);
                    acc[t] = fmaf(wd[j + 3], h4.w, acc[t]);
                }
            }
        }
    }
}

// Thread per down row d of expert unique[blockIdx.y]: the same scheme over the
// f32 h rows of the expert's slots (4-bit or 6-bit down codes).
__global__ void __launch_bounds__(kRowThreads) down_f32_kernel(StepArgs a, Workspace ws, int thr, int T) {
    extern __shared__ float4 hs4[];
    float *hs = reinterpret_cast<float *>(hs4);  // [T][F]
    const int u = blockIdx.y;
    const int D = a.s.D, F = a.s.F;
    if (u >= *ws.U) return;
    const int e = ws.unique[u];
    const int p_begin = ws.offsets[e], p_end = ws.offsets[e + 1];
    if (thr > 0 && p_end - p_begin >= thr) return;
    const int d = blockIdx.x * kRowThreads + threadIdx.x;
    const bool has_row = d < D;
    const size_t row = (size_t)e * D + (has_row ? d : D - 1);
    const uint4 *dq = reinterpret_cast<const uint4 *>(a.planes.down_q + row * (F / 8));
    const unsigned char *dq6 = reinterpret_cast<const unsigned char *>(a.planes.down_q) + row * (3 * F / 4);
    const bool six = a.s.down_bits == 6;
    const uint16_t *ds = a.planes.down_s + row * (F / kGroup);
    const uint16_t *db = a.planes.down_b + row * (F / kGroup);
    for (int p0 = p_begin; p0 < p_end; p0 += T) {
        const int cnt = min(T, p_end - p0);
        __syncthreads();
        for (int i = threadIdx.x; i < cnt * (F / 4); i += kRowThreads) {
            const int t = i / (F / 4), c4 = i - t * (F / 4);
            hs4[(size_t)t * (F / 4) + c4] =
                *reinterpret_cast<const float4 *>(ws.h + (size_t)(p0 + t) * F + (size_t)c4 * 4);
        }
        __syncthreads();
        if (!has_row) continue;
        float acc[kTok];
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = 0.f;
        if (six) {
            if (cnt == 1)
                down_row6<1>(dq6, ds, db, hs, F, cnt, acc);
            else
                down_row6<kTok>(dq6, ds, db, hs, F, cnt, acc);
        } else if (cnt == 1)
            down_row<1>(dq, ds, db, hs, F, cnt, acc);
        else if (cnt == 2)
            down_row<2>(dq, ds, db, hs, F, cnt, acc);
        else if (cnt <= 4)
            down_row<4>(dq, ds, db, hs, F, cnt, acc);
        else
            down_row<kTok>(dq, ds, db, hs, F, cnt, acc);
#pragma unroll
        for (int t = 0; t < kTok; ++t)
            if (t < cnt) ws.y[(size_t)(p0 + t) * D + d] = acc[t];
    }
}

// thread per 4 consecutive output elements (D % 4 == 0); for each, the
// rank-ordered weighted sum and one final rounding
template <int OT>
__global__ void combine_kernel(StepArgs a, Workspace ws) {
    const int i4 = blockIdx.x * blockDim.x + threadIdx.x;
    const int D = a.s.D, k = a.s.k;
    if (i4 >= a.s.n * (D / 4)) return;
    const int t = i4 / (D / 4), d = 4 * (i4 - t * (D / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int p = ws.slot_of[t * k + j];
        if (p < 0) continue;  // an expert this plan does not own
        const float wj = ws.topk_w[t * k + j];
        const float4 yv = *reinterpret_cast<const float4 *>(ws.y + (size_t)p * D + d);
        acc.x = fmaf(wj, yv.x, acc.x);
        acc.y = fmaf(wj, yv.y, acc.y);
        acc.z = fmaf(wj, yv.z, acc.z);
        acc.w = fmaf(wj, yv.w, acc.w);
    }
    const size_t i = (size_t)t * D + d;
    if (OT == MOE_DTYPE_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(a.out) + i) = acc;
    } else {
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out) + i;
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(o) = pk;
    }
}

}  // namespace

cudaError_t launch_experts(const StepArgs &a, const Workspace &ws, int mma_thr, cudaStream_t st,
                           int &launched) {
    const int maxU = min(a.s.E, a.s.n * a.s.k);
    // experts from mma_thr tokens on the tcgen05 GEMMs, where the shape allows
    const int thr = mma_thr > 0 && tc_variant_supported(a.s) ? mma_thr : 0;
    auto gemms = [&](bool down) { return launch_expert_tc(a, ws, thr, down, st, launched); };
    // with a threshold of one token every selected expert takes the
    // tensor-core kernels: the GEMV kernels would have nothing to do
    const bool gemv = thr != 1;
    dim3 block(256);
    cudaError_t err;
    if (thr > 0 && (err = gemms(false)) != cudaSuccess) return err;
    const int T1 = pass_tokens(a.s.D), T2 = pass_tokens(a.s.F);
    const int sm1 = T1 * a.s.D * 4, sm2 = T2 * a.s.F * 4;
    dim3 g1((a.s.F + kRowThreads - 1) / kRowThreads, maxU);
    if (!gemv) {
    } else if (a.s.x_dtype == MOE_DTYPE_F32) {
        if ((err = cudaFuncSetAttribute(gateup_f32_kernel<MOE_DTYPE_F32>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, sm1)) != cudaSuccess)
            return err;
        gateup_f32_kernel<MOE_DTYPE_F32><<<g1, kRowThreads, sm1, st>>>(a, ws, thr, T1);
    } else {
        if ((err = cudaFuncSetAttribute(gateup_f32_kernel<MOE_DTYPE_BF16>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, sm1)) != cudaSuccess)
            return err;
        gateup_f32_kernel<MOE_DTYPE_BF16><<<g1, kRowThreads, sm1, st>>>(a, ws, thr, T1);
    }
    if (gemv) {
        launched += 1;
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if (thr > 0 && (err = gemms(true)) != cudaSuccess) return err;
    if (gemv) {
        if ((err = cudaFuncSetAttribute(down_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm2)) !=
            cudaSuccess)
            return err;
        dim3 g2((a.s.D + kRowThreads - 1) / kRowThreads, maxU);
        down_f32_kernel<<<g2, kRowThreads, sm2, st>>>(a, ws, thr, T2);
        launched += 1;
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    const int total = a.s.n * (a.s.D / 4);
    dim3 g3((total + 255) / 256);
    if (a.s.out_dtype == MOE_DTYPE_F32)
        combine_kernel<MOE_DTYPE_F32><<<g3, block, 0, st>>>(a, ws);
    else
        combine_kernel<MOE_DTYPE_BF16><<<g3, block, 0, st>>>(a, ws);
    launched += 1;
    return cudaGetLastError();
}

}  // namespace moe
