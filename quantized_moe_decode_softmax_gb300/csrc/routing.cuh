// routing.cuh -- block-cooperative device routines for the routing half of the
// decode step: softmax over all experts, top-k with renormalised weights, and
// the grouping of (token, rank) slots by expert.
//
// Sources: mlxcel issue #1616 "perf(moe): batched decode scales 1.55x against
// 3.25x on dense" (Leading hypothesis: the per-slot expert traffic that
// grouping by expert id removes; Proposed Solution: de-duplicate expert ids
// across the cohort) and issue #1859 "perf(moe): attribute the MoE decode gap
// at the M = 1 expert gather" (Problem / Background: the unsorted per-slot
// gather below 64 slots).
//
// Conventions shared with the rest of the library:
//   * top-k order is descending logit, ties to the lower expert index
//   * w_j = p_j / sum_{j'} p_j' with p = softmax over all E experts
//   * grouped order: expert ascending, token ascending within an expert (a
//     token selects an expert at most once)
#pragma once

#include <stdint.h>

namespace moe {

struct ValIdx {
    float v;
    int i;
};

// larger value wins; equal values -> lower index
__device__ __forceinline__ ValIdx vi_better(ValIdx a, ValIdx b) {
    return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ ValIdx warp_argmax(ValIdx a) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        ValIdx b;
        b.v = __shfl_xor_sync(0xffffffffu, a.v, o);
        b.i = __shfl_xor_sync(0xffffffffu, a.i, o);
        a = vi_better(a, b);
    }
    return a;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Softmax + top-k + renormalisation of one token's logits held in registers:
// lane l holds experts l + 32*i for i < NPL (entries past E are -inf).
template <int NPL>
__device__ __forceinline__ void warp_topk_token(const float *lt, int E, int k, int lane,
                                                int *idx_out, float *w_out) {
    float v[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        const float x = e < E ? __ldcg(lt + e) : -INFINITY;
        v[i] = x == x ? x : -INFINITY;  // NaN ranks as -inf
    }
    float m = v[0];
#pragma unroll
    for (int i = 1; i < NPL; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        if (lane + 32 * i < E) z += expf(v[i] - m);
    z = warp_sum(z);
    // lane-local best of the untaken entries, refreshed only on the lane that
    // loses its best to the warp-wide winner
    ValIdx lb{-INFINITY, 0x7fffffff};
#pragma unroll
    for (int i = 0; i < NPL; ++i)
        if (lane + 32 * i < E) lb = vi_better(lb, ValIdx{v[i], lane + 32 * i});
    uint32_t taken = 0;
    float psum = 0.f;
    for (int j = 0; j < k; ++j) {
        const ValIdx best = warp_argmax(lb);
        if (lane == 0) {
            const float p = expf(best.v - m) / z;
            idx_out[j] = best.i;
            w_out[j] = p;  // renormalised below
            psum += p;
        }
        if ((best.i & 31) == lane) {
            taken |= 1u << (best.i >> 5);
            lb = ValIdx{-INFINITY, 0x7fffffff};
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (lane + 32 * i < E && !(taken & (1u << i)))
                    lb = vi_better(lb, ValIdx{v[i], lane + 32 * i});
        }
    }
    if (lane == 0)
        for (int j = 0; j < k; ++j) w_out[j] = w_out[j] / psum;
}

// Softmax + top-k + renormalisation for tokens t = warp, warp + nwarps, ...
// logits: [n, E] in global memory, read once through L2 (they may have been
// written by other CTAs of the same kernel). Writes s_idx / s_w [n*k]
// (shared). Requires E <= 1024 and k <= 16.
__device__ inline void block_topk(const float *logits, int n, int E, int k, int *s_idx,
                                  float *s_w) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    for (int t = warp; t < n; t += nwarps) {
        const float *lt = logits + (size_t)t * E;
        int *io = s_idx + t * k;
        float *wo = s_w + t * k;
        if (E <= 32) warp_topk_token<1>(lt, E, k, lane, io, wo);
        else if (E <= 64) warp_topk_token<2>(lt, E, k, lane, io, wo);
        else if (E <= 128) warp_topk_token<4>(lt, E, k, lane, io, wo);
        else if (E <= 256) warp_topk_token<8>(lt, E, k, lane, io, wo);
        else if (E <= 512) warp_topk_token<16>(lt, E, k, lane, io, wo);
        else warp_topk_token<32>(lt, E, k, lane, io, wo);
    }
}

// Grouping of the n*k slots by expert (block-cooperative, all threads), over
// the experts [e_lo, e_hi) only (an expert-parallel shard; the other slots get
// slot_of = -1 and no grouped position).
// s_mask: [E] u64 scratch (token bitmask per expert, n <= 64).
// Outputs (shared): counts[E], offsets[E+1], slot_token/slot_k[n*k] in grouped
// order, slot_of[n*k] (t*k + j -> grouped position), unique[E], *U.
__device__ inline void block_group(const int *s_idx, int n, int E, int k, int e_lo, int e_hi,
                                   unsigned long long *s_mask, int *counts, int *offsets,
                                   int *slot_token, int *slot_k, int *slot_of, int *unique,
                                   int *U) {
    const int S = n * k;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0ull;
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int e = s_idx[s];
        if ((unsigned)e < (unsigned)E && e >= e_lo && e < e_hi) atomicOr(&s_mask[e], 1ull << (s / k));
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = __popcll(s_mask[e]);
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive scans of counts and of (counts > 0)
        const int lane = threadIdx.x;
        int base = 0, ubase = 0;
        for (int c0 = 0; c0 < E; c0 += 32) {
            int e = c0 + lane;
            int c = e < E ? counts[e] : 0;
            int u = c > 0 ? 1 : 0;
            int ic = c, iu = u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int a = __shfl_up_sync(0xffffffffu, ic, o);
                int b = __shfl_up_sync(0xffffffffu, iu, o);
                if (lane >= o) {
                    ic += a;
                    iu += b;
                }
            }
            if (e < E) {
                offsets[e] = base + ic - c;
                if (u) unique[ubase + iu - 1] = e;
            }
            base += __shfl_sync(0xffffffffu, ic, 31);
            ubase += __shfl_sync(0xffffffffu, iu, 31);
        }
        if (lane == 0) {
            offsets[E] = base;
            *U = ubase;
        }
    }
    __syncthreads();
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int e = s_idx[s];
        if ((unsigned)e >= (unsigned)E || e < e_lo || e >= e_hi) {
            slot_of[s] = -1;
            continue;
        }
        const int t = s / k;
        const unsigned long long below = (t == 0) ? 0ull : (s_mask[e] & ((1ull << t) - 1ull));
        const int pos = offsets[e] + __popcll(below);
        slot_token[pos] = t;
        slot_k[pos] = s - t * k;
        slot_of[s] = pos;
    }
    __syncthreads();
}

}  // namespace moe
