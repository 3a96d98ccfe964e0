// topk.cuh -- one warp's top-k over one token's router logits, shared by the
// routing kernels and the fused decode kernel.
//
// Rule (the layer's routing): rank by fp32 logit, larger first, equal logits
// -> lower expert id first, a NaN logit counts as -infinity; the weights over
// the k picks are a softmax, or each pick's sigmoid divided by their sum.
#pragma once

#include "ds4g_common.cuh"

namespace ds4g {

constexpr int kMaxPerLane = 8;   // 256 experts / 32 lanes

__device__ __forceinline__ float canon(float v) { return v != v ? -INFINITY : v; }

// a ranks before b
__device__ __forceinline__ bool before(float va, int ia, float vb, int ib)
{
    return ib < 0 || (ia >= 0 && (va > vb || (va == vb && ia < ib)));
}

// One token, one warp.  Writes ids[k], wts[k] (lane 0).
__device__ __forceinline__ void topk_warp(const float *__restrict__ row, int E, int k, int score,
                                          int32_t *__restrict__ ids, float *__restrict__ wts)
{
    const int lane = threadIdx.x & 31;
    float v[kMaxPerLane];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
        int e = lane + 32 * j;
        v[j] = -INFINITY;
        if (e < E) {
            v[j] = canon(__ldg(row + e));
            avail |= 1u << j;
        }
    }
    float sel_v[DS4G_MAX_TOPK];
    int sel_i[DS4G_MAX_TOPK];
#pragma unroll
    for (int i = 0; i < DS4G_MAX_TOPK; ++i) {
        if (i >= k) break;
        float bv = -INFINITY;
        int bi = -1;
#pragma unroll
        for (int j = 0; j < kMaxPerLane; ++j) {
            if ((avail >> j) & 1u) {
                int e = lane + 32 * j;
                if (before(v[j], e, bv, bi)) { bv = v[j]; bi = e; }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
        sel_v[i] = bv;
        sel_i[i] = bi;
    }
    if (lane == 0) {
        float p[DS4G_MAX_TOPK];
        float sum = 0.0f;
        if (score == DS4G_SCORE_SOFTMAX) {
            float m = sel_v[0];
#pragma unroll
            for (int i = 0; i < DS4G_MAX_TOPK; ++i)
                if (i < k) { p[i] = expf(sel_v[i] - m); sum += p[i]; }
        } else {
#pragma unroll
            for (int i = 0; i < DS4G_MAX_TOPK; ++i)
                if (i < k) { p[i] = 1.0f / (1.0f + expf(-sel_v[i])); sum += p[i]; }
        }
#pragma unroll
        for (int i = 0; i < DS4G_MAX_TOPK; ++i)
            if (i < k) { ids[i] = sel_i[i]; wts[i] = p[i] / sum; }
    }
}

}  // namespace ds4g
