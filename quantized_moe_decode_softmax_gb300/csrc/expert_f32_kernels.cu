// expert_f32_kernels.cu -- the f32 check path of the expert half of the step.
// Every weight is dequantised exactly to f32 (w = s*q + b) and every product
// is accumulated in f32 on the CUDA cores. Slow by design; it is the path that
// MOE_FLAG_F32_DEBUG selects, held to 1e-4 of RMS(out) against the oracle.
//
// Stages (one launch each), over the de-duplicated expert list:
//   gate/up : h[p, f] = silu(sum_d Wg[e,f,d] x[t,d]) * sum_d Wu[e,f,d] x[t,d]
//   down    : y[p, d] = sum_f Wd[e,d,f] h[p,f]
//   combine : out[t, d] = sum_{j<k} w[t,j] * y[slot_of(t,j), d], j ascending
// where p runs over the slots grouped under expert e and t = slot_token[p].
//
// Sources: mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against
// 3.25x on dense" -- Current Behavior (SwitchGLU experts, moe_weighted_sum,
// 4-bit group 64), Implementation Notes (f32 partials, a single final
// rounding, parity against an all-f32 dense reference).
#include <cuda_bf16.h>

#include "moe_internal.h"
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

__device__ __forceinline__ void deq8(uint32_t q, float s, float b, float (&w)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = fmaf(s, (float)((q >> (4 * j)) & 0xFu), b);
}

constexpr int kTok = 8;  // tokens per register tile

// warp per gate/up row f of expert unique[blockIdx.y]
// (experts with at least `thr` tokens are left to the tile kernels when thr > 0)
template <int XT>
__global__ void __launch_bounds__(256) gateup_f32_kernel(StepArgs a, Workspace ws, int thr) {
    const int lane = threadIdx.x & 31;
    const int f = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int u = blockIdx.y;
    const int D = a.s.D, F = a.s.F;
    if (u >= *ws.U || f >= F) return;
    const int e = ws.unique[u];
    const int p_begin = ws.offsets[e], p_end = ws.offsets[e + 1];
    if (thr > 0 && p_end - p_begin >= thr) return;
    const size_t row = (size_t)e * F + f;
    const uint32_t *gq = a.planes.gate_q + row * (D / 8);
    const uint32_t *uq = a.planes.up_q + row * (D / 8);
    const uint16_t *gs = a.planes.gate_s + row * (D / kGroup);
    const uint16_t *gb = a.planes.gate_b + row * (D / kGroup);
    const uint16_t *us = a.planes.up_s + row * (D / kGroup);
    const uint16_t *ub = a.planes.up_b + row * (D / kGroup);
    for (int p0 = p_begin; p0 < p_end; p0 += kTok) {
        const int cnt = min(kTok, p_end - p0);
        int tok[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) tok[i] = i < cnt ? ws.slot_token[p0 + i] : 0;
        float ag[kTok], au[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) ag[i] = au[i] = 0.f;
        for (int wi = lane; wi < D / 8; wi += 32) {
            float wg[8], wu[8];
            deq8(__ldg(gq + wi), bf16f(gs[wi / 8]), bf16f(gb[wi / 8]), wg);
            deq8(__ldg(uq + wi), bf16f(us[wi / 8]), bf16f(ub[wi / 8]), wu);
#pragma unroll
            for (int i = 0; i < kTok; ++i) {
                if (i < cnt) {
                    float xv[8];
                    ld8<XT>(a.x, (size_t)tok[i] * D + (size_t)wi * 8, xv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        ag[i] = fmaf(wg[j], xv[j], ag[i]);
                        au[i] = fmaf(wu[j], xv[j], au[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
            const float g = warp_sum(ag[i]);
            const float uu = warp_sum(au[i]);
            if (lane == 0 && i < cnt) ws.h[(size_t)(p0 + i) * F + f] = g / (1.0f + expf(-g)) * uu;
        }
    }
}

// warp per down row d of expert unique[blockIdx.y]
__global__ void __launch_bounds__(256) down_f32_kernel(StepArgs a, Workspace ws, int thr) {
    const int lane = threadIdx.x & 31;
    const int d = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int u = blockIdx.y;
    const int D = a.s.D, F = a.s.F;
    if (u >= *ws.U || d >= D) return;
    const int e = ws.unique[u];
    const int p_begin = ws.offsets[e], p_end = ws.offsets[e + 1];
    if (thr > 0 && p_end - p_begin >= thr) return;
    const size_t row = (size_t)e * D + d;
    const uint32_t *dq = a.planes.down_q + row * (F / 8);
    const uint16_t *ds = a.planes.down_s + row * (F / kGroup);
    const uint16_t *db = a.planes.down_b + row * (F / kGroup);
    for (int p0 = p_begin; p0 < p_end; p0 += kTok) {
        const int cnt = min(kTok, p_end - p0);
        float acc[kTok];
#pragma unroll
        for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
        for (int wi = lane; wi < F / 8; wi += 32) {
            float wd[8];
            deq8(__ldg(dq + wi), bf16f(ds[wi / 8]), bf16f(db[wi / 8]), wd);
#pragma unroll
            for (int i = 0; i < kTok; ++i) {
                if (i < cnt) {
                    const float4 *hp = reinterpret_cast<const float4 *>(ws.h + (size_t)(p0 + i) * F + wi * 8);
                    const float4 h0 = hp[0], h1 = hp[1];
                    const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i] = fmaf(wd[j], hv[j], acc[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kTok; ++i) {
            const float v = warp_sum(acc[i]);
            if (lane == 0 && i < cnt) ws.y[(size_t)(p0 + i) * D + d] = v;
        }
    }
}

// thread per output element; rank-ordered weighted sum, one final rounding
template <int OT>
__global__ void combine_kernel(StepArgs a, Workspace ws) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int D = a.s.D, k = a.s.k;
    if (i >= a.s.n * D) return;
    const int t = i / D, d = i - t * D;
    float acc = 0.f;
    for (int j = 0; j < k; ++j)
        acc = fmaf(ws.topk_w[t * k + j], ws.y[(size_t)ws.slot_of[t * k + j] * D + d], acc);
    if (OT == MOE_DTYPE_F32)
        static_cast<float *>(a.out)[i] = acc;
    else
        static_cast<__nv_bfloat16 *>(a.out)[i] = __float2bfloat16_rn(acc);
}

}  // namespace

cudaError_t launch_experts_f32(const StepArgs &a, const Workspace &ws, int tile_thr, cudaStream_t st,
                               int &launched) {
    const int maxU = min(a.s.E, a.s.n * a.s.k);
    const int thr = tile_thr > 0 && tile_variant_supported(a.s) ? tile_thr : 0;
    dim3 block(256);
    cudaError_t err;
    if (thr > 0 && (err = launch_expert_tiles(a, ws, thr, false, st, launched)) != cudaSuccess) return err;
    dim3 g1((a.s.F + 7) / 8, maxU);
    if (a.s.x_dtype == MOE_DTYPE_F32)
        gateup_f32_kernel<MOE_DTYPE_F32><<<g1, block, 0, st>>>(a, ws, thr);
    else
        gateup_f32_kernel<MOE_DTYPE_BF16><<<g1, block, 0, st>>>(a, ws, thr);
    launched += 1;
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (thr > 0 && (err = launch_expert_tiles(a, ws, thr, true, st, launched)) != cudaSuccess) return err;
    dim3 g2((a.s.D + 7) / 8, maxU);
    down_f32_kernel<<<g2, block, 0, st>>>(a, ws, thr);
    launched += 1;
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const int total = a.s.n * a.s.D;
    dim3 g3((total + 255) / 256);
    if (a.s.out_dtype == MOE_DTYPE_F32)
        combine_kernel<MOE_DTYPE_F32><<<g3, block, 0, st>>>(a, ws);
    else
        combine_kernel<MOE_DTYPE_BF16><<<g3, block, 0, st>>>(a, ws);
    launched += 1;
    return cudaGetLastError();
}

}  // namespace moe
