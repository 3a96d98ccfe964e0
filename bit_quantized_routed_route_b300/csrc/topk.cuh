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

// Order-preserving map of a non-NaN float to an unsigned key (larger float,
// larger key; -0 is mapped as +0 so that the two zeros tie as they compare
// equal), and back.  Every key of a real logit, -inf included, is above 0.
__device__ __forceinline__ uint32_t order_key(float v)
{
    const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t o)
{
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// One token, one warp.  Writes ids[k], wts[k] (lanes 0..k-1).  Each round the
// warp takes the largest remaining key with two warp reductions (the largest
// key, then the smallest expert id holding it), so the order is: larger
// logit first, equal logits -> lower id first.  Lane i keeps pick i; the
// weights are formed with the picks' fp32 values and summed in pick order.
__device__ __forceinline__ void topk_warp(const float *__restrict__ row, int E, int k, int score,
                                          int32_t *__restrict__ ids, float *__restrict__ wts)
{
    const int lane = threadIdx.x & 31;
    uint32_t key[kMaxPerLane];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
        const int e = lane + 32 * j;
        key[j] = 0u;
        if (e < E) {
            key[j] = order_key(canon(__ldg(row + e)));
            avail |= 1u << j;
        }
    }
    float my_v = 0.0f;
    int my_id = 0;
#pragma unroll
    for (int i = 0; i < DS4G_MAX_TOPK; ++i) {
        if (i >= k) break;
        // this lane's best remaining key; equal keys keep the lower j (lower id)
        uint32_t bk = 0u;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < kMaxPerLane; ++j)
            if (((avail >> j) & 1u) && key[j] > bk) { bk = key[j]; bj = j; }
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t win = __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
        if ((int)(win & 31u) == lane) avail &= ~(1u << (win >> 5));
        if (lane == i) { my_v = key_value(m); my_id = (int)win; }
    }
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    float p = 0.0f;
    if (lane < k) p = score == DS4G_SCORE_SOFTMAX ? expf(my_v - top) : 1.0f / (1.0f + expf(-my_v));
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum += __shfl_sync(0xffffffffu, p, i);
    if (lane < k) {
        ids[lane] = my_id;
        wts[lane] = p / sum;
    }
}

}  // namespace ds4g
