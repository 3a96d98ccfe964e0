// route.cu -- top-k routing, routing weights, per-expert counts, segment
// offsets and the token-by-expert permutation.
//
// Routing is what makes the experts "routed" (ds4 README mirror, "Model
// Weights": only the routed MoE experts are quantized).  Rule used here and
// in the reference: rank by fp32 logit, larger first, equal logits -> lower
// expert id first, a NaN logit counts as -infinity; weights over the k picks
// are a softmax, or each pick's sigmoid divided by their sum.
//
// Kernels:
//   topk_kernel   one warp per token; each lane holds E/32 logits in
//                 registers; k rounds of two warp reductions (largest
//                 order key, then lowest expert id holding it).
//   scan_kernel   one CTA: a stable counting sort of the assignments
//                 a = t*k + i by expert: each warp counts, then places, one
//                 contiguous chunk (warp match-any ranks + per-warp,
//                 per-expert bases), with the counts, the exclusive scan over
//                 the experts and the active list in between, so the order
//                 inside each segment is ascending a.  No atomics.
//   route_small   both phases in one CTA for small T (decode), one launch.
//
// With an activation pointer the kernels also write the decode path's
// activation operand: xp = fp16(x) with every aligned group of 4 stored in the
// order (0, 2, 1, 3), and xs = fp32 sums of each 16 consecutive fp16 values.
#include "ds4g_common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace ds4g {
namespace {

// Four activations x[4g..4g+3] -> fp16, stored permuted (0,2,1,3); returns
// their fp32 sum.
__device__ __forceinline__ float prep4(const uint16_t *__restrict__ x, __half *__restrict__ xp,
                                       size_t g)
{
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x) + g);
    const __half h0 = __float2half_rn(bf16_bits(raw.x & 0xFFFFu));
    const __half h1 = __float2half_rn(bf16_bits(raw.x >> 16));
    const __half h2 = __float2half_rn(bf16_bits(raw.y & 0xFFFFu));
    const __half h3 = __float2half_rn(bf16_bits(raw.y >> 16));
    __half2 *o = reinterpret_cast<__half2 *>(xp + 4 * g);
    o[0] = __halves2half2(h0, h2);
    o[1] = __halves2half2(h1, h3);
    return __half2float(h0) + __half2float(h1) + __half2float(h2) + __half2float(h3);
}

// One group of 4 per lane; lanes 4j..4j+3 of a warp cover one sub-block of
// 16 and reduce its sum.  n_groups must be a multiple of 32 per warp pass.
__device__ __forceinline__ void prep_groups(const uint16_t *x, __half *xp, float *xs, size_t g)
{
    float v = prep4(x, xp, g);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    if ((g & 3) == 0) xs[g >> 2] = v;
}

__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int T, int E,
                                                   int k, int score, int32_t *__restrict__ ids,
                                                   float *__restrict__ wts,
                                                   const uint16_t *__restrict__ x, int H,
                                                   __half *__restrict__ xp, float *__restrict__ xs,
                                                   int32_t *status, int32_t *sync, int n_sync)
{
    if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = DS4G_OK;
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_sync; i += blockDim.x) sync[i] = 0;
    int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_warp(logits + (size_t)t * E, E, k, score, ids + (size_t)t * k, wts + (size_t)t * k);
    if (x) {
        const size_t g0 = (size_t)t * (H / 4);
        for (int g = threadIdx.x & 31; g < H / 4; g += 32) prep_groups(x, xp, xs, g0 + g);
    }
}

// Shared state of the counting sort (one CTA of NW >= 8 warps).
template <int NW>
struct ScanSmem {
    int offset[DS4G_MAX_EXPERTS + 1];
    int warp_base[NW][DS4G_MAX_EXPERTS];
    int warp_sum[8];
    int act_sum[8];
};

// counts / offsets / perm / slot_pos / active from ids[A].  Called by all
// NW * 32 threads of the CTA.  `ids` may have been written earlier in the same
// kernel, so it is read through the coherent path (no __restrict__).
//
// Warp w takes the contiguous chunk [w*C, (w+1)*C) of the assignments.  Pass 1
// counts its chunk per expert (warp match-any, warp-private table); the
// counts per expert are the sums over the warps; an exclusive scan over the
// experts gives the offsets; a prefix over the warps (in chunk order) turns
// each warp's counts into its first position per expert; pass 2 places the
// chunk in order (lanes of equal expert ranked by lane), so each segment is
// in ascending a.  The ids of a chunk are read eight loads at a time.
constexpr int kScanBatch = 8;

__device__ __forceinline__ void load_ids(const int32_t *ids, int a0, int a_end, int E, int lane,
                                         int (&eb)[kScanBatch])
{
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
        const int a = a0 + 32 * u + lane;
        const int e = a < a_end ? ids[a] : -1;
        eb[u] = e >= 0 && e < E ? e : -1;
    }
}

template <int NW>
__device__ void scan_body(ScanSmem<NW> &sm, const int32_t *ids, int A, int E,
                          int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                          int32_t *active, int32_t *n_active)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned below = (1u << lane) - 1u;
    for (int i = tid; i < NW * DS4G_MAX_EXPERTS; i += blockDim.x) (&sm.warp_base[0][0])[i] = 0;
    __syncthreads();
    const int C = ((A + NW - 1) / NW + 31) / 32 * 32;
    const int a_beg = warp * C, a_end = min(A, (warp + 1) * C);
    for (int a0 = a_beg; a0 < a_end; a0 += 32 * kScanBatch) {
        int eb[kScanBatch];
        load_ids(ids, a0, a_end, E, lane, eb);
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const unsigned same = __match_any_sync(0xffffffffu, eb[u]);
            if (eb[u] >= 0 && (same & below) == 0) sm.warp_base[warp][eb[u]] += __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
    // exclusive scan over E <= 256 experts: 8 warps x 32
    int c = 0;
    if (tid < E)
        for (int w = 0; w < NW; ++w) c += sm.warp_base[w][tid];
    int incl = c;
    if (warp < 8) {
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) sm.warp_sum[warp] = incl;
    }
    __syncthreads();
    if (warp < 8) {
        int base = 0;
        for (int w = 0; w < warp; ++w) base += sm.warp_sum[w];
        if (tid < E) sm.offset[tid] = base + incl - c;
        if (tid == E - 1) sm.offset[E] = base + incl;
    }
    // active experts (count > 0) in id order
    if (warp < 8) {
        bool act = (tid < E) && c > 0;
        unsigned b = __ballot_sync(0xffffffffu, act);
        if (lane == 0) sm.act_sum[warp] = __popc(b);
    }
    __syncthreads();
    if (warp < 8) {
        bool act = (tid < E) && c > 0;
        unsigned b = __ballot_sync(0xffffffffu, act);
        int base = 0;
        for (int w = 0; w < warp; ++w) base += sm.act_sum[w];
        if (act && active) active[base + __popc(b & below)] = tid;
        if (tid == 255 && n_active) {
            int tot = 0;
            for (int w = 0; w < 8; ++w) tot += sm.act_sum[w];
            *n_active = tot;
        }
    }
    if (tid < E) {
        if (counts) counts[tid] = c;
        if (offsets) offsets[tid] = sm.offset[tid];
        // each warp's first position per expert
        int run = sm.offset[tid];
        for (int w = 0; w < NW; ++w) {
            const int cnt = sm.warp_base[w][tid];
            sm.warp_base[w][tid] = run;
            run += cnt;
        }
    }
    if (tid == 0 && offsets) offsets[E] = sm.offset[E];
    __syncthreads();
    for (int a0 = a_beg; a0 < a_end; a0 += 32 * kScanBatch) {
        int eb[kScanBatch];
        load_ids(ids, a0, a_end, E, lane, eb);
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const int e = eb[u];
            const unsigned same = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(same & below);
            if (e >= 0) {
                const int a = a0 + 32 * u + lane;
                const int pos = sm.warp_base[warp][e] + rank;
                if (perm) perm[pos] = a;
                if (slot_pos) slot_pos[a] = pos;
            }
            __syncwarp();
            if (e >= 0 && rank == 0) sm.warp_base[warp][e] += __popc(same);
            __syncwarp();
        }
    }
}

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t *ids, int A, int E,
                                                    int32_t *counts, int32_t *offsets,
                                                    int32_t *perm, int32_t *slot_pos,
                                                    int32_t *active, int32_t *n_active)
{
    __shared__ ScanSmem<32> sm;
    scan_body<32>(sm, ids, A, E, counts, offsets, perm, slot_pos, active, n_active);
}

// Small T: top-k by the 8 warps of the CTA, then the scan, one launch.
constexpr int kSmallWarps = 8;
__global__ void __launch_bounds__(kSmallWarps * 32) route_small_kernel(
    const float *__restrict__ logits, int T, int E, int k, int score, int32_t *ids, float *wts,
    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos, int32_t *active,
    int32_t *n_active, const uint16_t *__restrict__ x, int H, __half *__restrict__ xp,
    float *__restrict__ xs, int32_t *status, int32_t *sync, int n_sync)
{
    __shared__ ScanSmem<kSmallWarps> sm;
    ptx::grid_dep_launch();    // the consumer kernels may become resident and wait
    if (status && threadIdx.x == 0) *status = DS4G_OK;
    for (int i = threadIdx.x; i < n_sync; i += blockDim.x) sync[i] = 0;
    for (int t = threadIdx.x >> 5; t < T; t += kSmallWarps)
        topk_warp(logits + (size_t)t * E, E, k, score, ids + (size_t)t * k, wts + (size_t)t * k);
    if (x) {
        const size_t groups = (size_t)T * (H / 4);
        for (size_t g = threadIdx.x; g < groups; g += blockDim.x) prep_groups(x, xp, xs, g);
    }
    __threadfence_block();
    __syncthreads();
    scan_body<kSmallWarps>(sm, ids, T * k, E, counts, offsets, perm, slot_pos, active, n_active);
}

}  // namespace

cudaError_t launch_route(const float *logits, int T, int E, int k, int score, int32_t *ids,
                         float *wts, int32_t *counts, int32_t *offsets, int32_t *perm,
                         int32_t *slot_pos, int32_t *active, int32_t *n_active,
                         const uint16_t *x, int H, __half *xp, float *xs, int32_t *status,
                         int32_t *sync, int n_sync, cudaStream_t s)
{
    if (T <= kRouteSmallT) {
        route_small_kernel<<<1, kSmallWarps * 32, 0, s>>>(logits, T, E, k, score, ids, wts, counts, offsets,
                                             perm, slot_pos, active, n_active, x, H, xp, xs,
                                             status, sync, n_sync);
    } else {
        int warps = 8;
        topk_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, s>>>(logits, T, E, k, score, ids,
                                                                  wts, x, H, xp, xs, status, sync, n_sync);
        scan_kernel<<<1, 1024, 0, s>>>(ids, T * k, E, counts, offsets, perm, slot_pos, active,
                                       n_active);
    }
    return cudaGetLastError();
}

}  // namespace ds4g
