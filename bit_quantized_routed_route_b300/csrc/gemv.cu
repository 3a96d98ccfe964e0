// gemv.cu -- the general expert path: grouped dequant-and-dot on CUDA cores,
// correct for every segment size and every weight format (Q2_K, codebook,
// and the Q4_K / Q5_K / Q6_K and MXFP4 routed formats, which only this path
// runs).
//
// Per active expert e with segment tokens t_0..t_{n-1} (the assignments
// perm[offsets[e] .. offsets[e+1]-1]):
//   gateup_kernel:  h[p, n] = SiLU(W_gate[e][n,:] . x_t) * (W_up[e][n,:] . x_t)
//                   for every row n < inter (rows inter..I_pad-1 get 0), where
//                   p = offsets[e] + i is the segment position of assignment i;
//   down_kernel:    yslot[p, m] = w_a * (W_down[e][m,:] . h[p, :]);
//   combine_kernel: y[t, m] = sum_{i<k} yslot[slot_pos[t*k+i], m], slot order.
// (the SiLU-gated expert FFN over routed experts; ds4 README mirror, "Model
// Weights", names the routed up/gate and down projections.)
//
// Weights are dequantized to fp32 exactly as the block definitions state and
// accumulated in fp32.  One warp per weight row; lanes stride over the row's
// 16-weight units; a warp-shuffle sum finishes each dot product.  Work items
// (active expert, 8-row tile) are claimed by a persistent grid from the device
// list written by the routing kernels, so the host never reads the routing.
#include "ds4g_common.cuh"
#include "kquant.cuh"

namespace ds4g {
namespace {

constexpr int kWarps = 8;       // rows per work item
constexpr int kTokChunk = 8;    // tokens accumulated per pass over a row

// fp32 weights 16u .. 16u+15 of one super-block.
template <int FMT>
__device__ __forceinline__ void dequant16(const uint8_t *__restrict__ blk, int u,
                                          const int8_t *__restrict__ scb, float (&w)[16])
{
    if constexpr (FMT == DS4G_FMT_Q2K) {
        uint32_t dd = __ldg(reinterpret_cast<const uint32_t *>(blk + 80));
        float d = half_bits(dd & 0xFFFFu), dmin = half_bits(dd >> 16);
        int sc = __ldg(blk + u);
        int h = u >> 3, g = (u & 7) >> 1;
        const uint32_t *q4 = reinterpret_cast<const uint32_t *>(blk + 16 + 32 * h + 16 * (u & 1));
        float scale_part = d * (float)(sc & 15);
        float min_part = dmin * (float)(sc >> 4);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t word = __ldg(q4 + v);
#pragma unroll
            for (int by = 0; by < 4; ++by) {
                int q = (word >> (8 * by + 2 * g)) & 3;
                w[4 * v + by] = scale_part * (float)q - min_part;
            }
        }
    } else if constexpr (FMT != DS4G_FMT_CB2) {
        kquant_unit16<FMT>(blk, u, w);
    } else {
        uint32_t dbits = (uint32_t)__ldg(blk + 68) | ((uint32_t)__ldg(blk + 69) << 8);
        int G = u >> 1;
        int scale = (__ldg(blk + 64 + (G >> 1)) >> (4 * (G & 1))) & 15;
        float ds = half_bits(dbits) * (float)scale;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            int o = 2 * u + half;
            int idx = __ldg(blk + o);
            int sgn = __ldg(blk + 32 + o);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float v = ds * (float)scb[8 * idx + j];
                w[8 * half + j] = ((sgn >> j) & 1) ? -v : v;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ void load_x16(const uint16_t *__restrict__ x, float (&xv)[16])
{
    const uint4 *p = reinterpret_cast<const uint4 *>(x);
    uint4 a = __ldg(p), b = __ldg(p + 1);
    uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        xv[2 * i] = bf16_bits(wd[i] & 0xFFFFu);
        xv[2 * i + 1] = bf16_bits(wd[i] >> 16);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32) gateup_kernel(LayerArgs a)
{
    __shared__ int8_t scb[256 * 8];
    if constexpr (FMT == DS4G_FMT_CB2) {
        for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) scb[i] = a.codebook[i];
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bb = block_bytes_of(FMT);
    const int tiles = a.I_pad / kWarps;
    const int n_items = *a.n_active * tiles;
    const int units = (a.H / kQK) * 16;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int e = a.active[item / tiles];
        const int n = (item % tiles) * kWarps + warp;
        const int seg0 = a.offsets[e], seg_n = a.offsets[e + 1] - seg0;
        if (n >= a.I) {
            for (int i = lane; i < seg_n; i += 32) a.hbuf[(size_t)(seg0 + i) * a.I_pad + n] = 0.0f;
            continue;
        }
        const int we = weight_slot(a.wslot, a.n_wslots, e, a.status);
        const uint8_t *rg = a.w_gate + (size_t)we * a.gu_stride + (size_t)n * a.gu_row;
        const uint8_t *ru = a.w_up + (size_t)we * a.gu_stride + (size_t)n * a.gu_row;
        for (int c0 = 0; c0 < seg_n; c0 += kTokChunk) {
            const int nt = min(kTokChunk, seg_n - c0);
            const uint16_t *xr[kTokChunk];
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j) {
                int jj = j < nt ? j : 0;
                int asg = a.perm[seg0 + c0 + jj];
                xr[j] = a.x + (size_t)(asg / a.k) * a.H;
            }
            float ag[kTokChunk], au[kTokChunk];
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j) { ag[j] = 0.0f; au[j] = 0.0f; }
            for (int u = lane; u < units; u += 32) {
                const int b = u >> 4, su = u & 15;
                float wg[16], wu[16];
                dequant16<FMT>(rg + (size_t)b * bb, su, scb, wg);
                dequant16<FMT>(ru + (size_t)b * bb, su, scb, wu);
#pragma unroll
                for (int j = 0; j < kTokChunk; ++j) {
                    if (j < nt) {
                        float xv[16];
                        load_x16(xr[j] + (size_t)u * 16, xv);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            ag[j] = fmaf(wg[i], xv[i], ag[j]);
                            au[j] = fmaf(wu[i], xv[i], au[j]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j) {
                if (j < nt) {
                    float g = warp_sum(ag[j]);
                    float uu = warp_sum(au[j]);
                    if (lane == 0) a.hbuf[(size_t)(seg0 + c0 + j) * a.I_pad + n] = silu_mul(g, uu);
                }
            }
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kWarps * 32) down_kernel(LayerArgs a)
{
    __shared__ int8_t scb[256 * 8];
    if constexpr (FMT == DS4G_FMT_CB2) {
        for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) scb[i] = a.codebook[i];
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int bb = block_bytes_of(FMT);
    const int tiles = a.H / kWarps;
    const int n_items = *a.n_active * tiles;
    const int units = (a.I_pad / kQK) * 16;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int e = a.active[item / tiles];
        const int m = (item % tiles) * kWarps + warp;
        const int seg0 = a.offsets[e], seg_n = a.offsets[e + 1] - seg0;
        const int we = weight_slot(a.wslot, a.n_wslots, e, a.status);
        const uint8_t *rd = a.w_down + (size_t)we * a.dn_stride + (size_t)m * a.dn_row;
        for (int c0 = 0; c0 < seg_n; c0 += kTokChunk) {
            const int nt = min(kTokChunk, seg_n - c0);
            float acc[kTokChunk];
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j) acc[j] = 0.0f;
            for (int u = lane; u < units; u += 32) {
                const int b = u >> 4, su = u & 15;
                float wd[16];
                dequant16<FMT>(rd + (size_t)b * bb, su, scb, wd);
#pragma unroll
                for (int j = 0; j < kTokChunk; ++j) {
                    if (j < nt) {
                        const float4 *hp = reinterpret_cast<const float4 *>(
                            a.hbuf + (size_t)(seg0 + c0 + j) * a.I_pad + (size_t)u * 16);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            float4 hv = hp[v];
                            acc[j] = fmaf(wd[4 * v], hv.x, acc[j]);
                            acc[j] = fmaf(wd[4 * v + 1], hv.y, acc[j]);
                            acc[j] = fmaf(wd[4 * v + 2], hv.z, acc[j]);
                            acc[j] = fmaf(wd[4 * v + 3], hv.w, acc[j]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j) {
                if (j < nt) {
                    float o = warp_sum(acc[j]);
                    if (lane == 0) {
                        int p = seg0 + c0 + j;
                        a.yslot[(size_t)p * a.H + m] = a.wts[a.perm[p]] * o;
                    }
                }
            }
        }
    }
}

// y[t, m..m+3] = sum_i yslot[slot_pos[t*k+i], m..m+3], slot order.
__global__ void __launch_bounds__(256) combine_kernel(LayerArgs a)
{
    const int q = a.H / 4;
    const int64_t total = (int64_t)a.T * q;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / q), c = (int)(i % q);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < a.k; ++s) {
            int p = a.slot_pos[t * a.k + s];
            float4 v = reinterpret_cast<const float4 *>(a.yslot + (size_t)p * a.H)[c];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4 *>(a.y + (size_t)t * a.H)[c] = acc;
    }
}

}  // namespace

cudaError_t launch_combine(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s)
{
    int64_t quads = (int64_t)a.T * (a.H / 4);
    int64_t want = (quads + 255) / 256, cap = (int64_t)dev.sm_count * 8;
    int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
    combine_kernel<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// Gate/up in the W_gate / W_up format, down in the W_down format (they may
// differ: the shipping mix has codebook gate/up and Q2_K down; Q6_K is a
// down-only format).
cudaError_t launch_gemv_gateup(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s)
{
    const int grid = min(min(a.E, a.A) * (a.I_pad / kWarps), dev.sm_count * 8);
    switch (a.gu_format) {
    case DS4G_FMT_Q2K: gateup_kernel<DS4G_FMT_Q2K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_CB2: gateup_kernel<DS4G_FMT_CB2><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_Q4K: gateup_kernel<DS4G_FMT_Q4K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_Q5K: gateup_kernel<DS4G_FMT_Q5K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_MXFP4: gateup_kernel<DS4G_FMT_MXFP4><<<grid, kWarps * 32, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gemv_down(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s)
{
    const int grid = min(min(a.E, a.A) * (a.H / kWarps), dev.sm_count * 8);
    switch (a.dn_format) {
    case DS4G_FMT_Q2K: down_kernel<DS4G_FMT_Q2K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_CB2: down_kernel<DS4G_FMT_CB2><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_Q4K: down_kernel<DS4G_FMT_Q4K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_Q5K: down_kernel<DS4G_FMT_Q5K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_Q6K: down_kernel<DS4G_FMT_Q6K><<<grid, kWarps * 32, 0, s>>>(a); break;
    case DS4G_FMT_MXFP4: down_kernel<DS4G_FMT_MXFP4><<<grid, kWarps * 32, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_gemv_path(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s,
                             const cudaEvent_t *ev)
{
    cudaError_t e;
    if ((e = launch_gemv_gateup(a, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[2], s)) != cudaSuccess) return e;
    if ((e = launch_gemv_down(a, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[3], s)) != cudaSuccess) return e;
    if ((e = launch_combine(a, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[4], s)) != cudaSuccess) return e;
    return cudaGetLastError();
}

int32_t gemv_path_launches(const Plan &) { return 3; }

}  // namespace ds4g
