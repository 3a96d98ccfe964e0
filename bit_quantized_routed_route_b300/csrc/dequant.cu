// dequant.cu -- standalone dequantization of Q2_K, codebook-2-bit and the
// Q4_K / Q5_K / Q6_K super-blocks (the block layouts are GGUF's K-quants and
// an IQ2_XXS-style codebook format; ds4 README mirror, "Model Weights" and
// "Acknowledgements to llama.cpp and GGML").
//
// Pure HBM streams: one super-block in (84, 70, 144, 176 or 210 bytes), 1 KB
// (fp32) or 512 B (fp16/bf16) out.  One thread per 16 weights (Q2_K and the
// K-quants) or per 8 weights (codebook group); the fp32 value is formed
// exactly as the definition states (exact products, at most one rounding, in
// the subtraction), so fp32 output is bit-exact and fp16/bf16 output is its
// round-to-nearest-even.
#include "ds4g_common.cuh"
#include "kquant.cuh"

namespace ds4g {
namespace {

template <int DT>
__device__ __forceinline__ void store16(void *out, size_t first, const float (&w)[16])
{
    if constexpr (DT == DS4G_F32) {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + first);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = make_float4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            unsigned short lo, hi;
            if constexpr (DT == DS4G_F16) {
                lo = __half_as_ushort(__float2half_rn(w[2 * i]));
                hi = __half_as_ushort(__float2half_rn(w[2 * i + 1]));
            } else {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(w[2 * i]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(w[2 * i + 1]));
            }
            packed[i] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + first);
        o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
}

// One thread = sub-block s of block b (weights 16s .. 16s+15).
template <int DT>
__global__ void __launch_bounds__(256) q2k_dequant_kernel(const uint8_t *__restrict__ blocks,
                                                          int64_t n_blocks, void *__restrict__ out)
{
    int64_t total = n_blocks * 16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = i >> 4;
        int s = (int)(i & 15);
        const uint8_t *blk = blocks + b * kQ2KBytes;
        uint32_t dd = __ldg(reinterpret_cast<const uint32_t *>(blk + 80));
        float d = half_bits(dd & 0xFFFFu), dmin = half_bits(dd >> 16);
        int sc = __ldg(blk + s);
        // weights 16s..16s+15: half h = s/8, shift group g = (s%8)/2,
        // lanes 16*(s%2) .. +15 -> qs bytes 32h + 16(s%2) + (0..15)
        int h = s >> 3, g = (s & 7) >> 1;
        const uint32_t *q4 = reinterpret_cast<const uint32_t *>(blk + 16 + 32 * h + 16 * (s & 1));
        float scale_part = d * (float)(sc & 15);
        float min_part = dmin * (float)(sc >> 4);
        float w[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t word = __ldg(q4 + v);
#pragma unroll
            for (int by = 0; by < 4; ++by) {
                int q = (word >> (8 * by + 2 * g)) & 3;
                w[4 * v + by] = scale_part * (float)q - min_part;
            }
        }
        store16<DT>(out, (size_t)b * kQK + 16 * s, w);
    }
}

// One thread = group o (weights 8o .. 8o+7) of block b.  The codebook is
// staged in shared memory once per CTA.
template <int DT>
__global__ void __launch_bounds__(256) cb2_dequant_kernel(const uint8_t *__restrict__ blocks,
                                                          int64_t n_blocks,
                                                          const int8_t *__restrict__ cb,
                                                          void *__restrict__ out)
{
    __shared__ int8_t scb[256 * 8];
    for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) scb[i] = cb[i];
    __syncthreads();
    int64_t total = n_blocks * 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = i >> 5;
        int o = (int)(i & 31);
        const uint8_t *blk = blocks + b * kCB2Bytes;
        int idx = __ldg(blk + o);
        int sgn = __ldg(blk + 32 + o);
        int G = o >> 2;
        int scale = (__ldg(blk + 64 + (G >> 1)) >> (4 * (G & 1))) & 15;
        uint32_t dbits = (uint32_t)__ldg(blk + 68) | ((uint32_t)__ldg(blk + 69) << 8);
        float ds = half_bits(dbits) * (float)scale;
        float w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float v = ds * (float)scb[8 * idx + j];
            w[j] = ((sgn >> j) & 1) ? -v : v;
        }
        size_t first = (size_t)b * kQK + 8 * o;
        if constexpr (DT == DS4G_F32) {
            float4 *po = reinterpret_cast<float4 *>(static_cast<float *>(out) + first);
            po[0] = make_float4(w[0], w[1], w[2], w[3]);
            po[1] = make_float4(w[4], w[5], w[6], w[7]);
        } else {
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                unsigned short lo, hi;
                if constexpr (DT == DS4G_F16) {
                    lo = __half_as_ushort(__float2half_rn(w[2 * j]));
                    hi = __half_as_ushort(__float2half_rn(w[2 * j + 1]));
                } else {
                    lo = __bfloat16_as_ushort(__float2bfloat16_rn(w[2 * j]));
                    hi = __bfloat16_as_ushort(__float2bfloat16_rn(w[2 * j + 1]));
                }
                p[j] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + first) =
                make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

// One thread = weights 16u .. 16u+15 of block b (a K-quant format).
template <int FMT, int DT>
__global__ void __launch_bounds__(256) kquant_dequant_kernel(const uint8_t *__restrict__ blocks,
                                                             int64_t n_blocks,
                                                             void *__restrict__ out)
{
    const int64_t total = n_blocks * 16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i >> 4;
        const int u = (int)(i & 15);
        float w[16];
        kquant_unit16<FMT>(blocks + b * block_bytes_of(FMT), u, w);
        store16<DT>(out, (size_t)b * kQK + 16 * u, w);
    }
}

template <int FMT>
void launch_kquant_fmt(const uint8_t *blocks, int64_t n_blocks, void *out, int dtype, int grid,
                       cudaStream_t s)
{
    if (dtype == DS4G_F32)
        kquant_dequant_kernel<FMT, DS4G_F32><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
    else if (dtype == DS4G_F16)
        kquant_dequant_kernel<FMT, DS4G_F16><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
    else
        kquant_dequant_kernel<FMT, DS4G_BF16><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
}

int grid_for(int64_t threads_needed)
{
    DeviceInfo dev;
    int sms = device_info(&dev) == DS4G_OK ? dev.sm_count : 148;
    int64_t blocks = (threads_needed + 255) / 256;
    int64_t cap = (int64_t)sms * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_q2k_dequant(const uint8_t *blocks, int64_t n_blocks, void *out, int dtype,
                               cudaStream_t s)
{
    int grid = grid_for(n_blocks * 16);
    if (dtype == DS4G_F32)
        q2k_dequant_kernel<DS4G_F32><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
    else if (dtype == DS4G_F16)
        q2k_dequant_kernel<DS4G_F16><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
    else
        q2k_dequant_kernel<DS4G_BF16><<<grid, 256, 0, s>>>(blocks, n_blocks, out);
    return cudaGetLastError();
}

cudaError_t launch_cb2_dequant(const uint8_t *blocks, int64_t n_blocks, const int8_t *cb,
                               void *out, int dtype, cudaStream_t s)
{
    int grid = grid_for(n_blocks * 32);
    if (dtype == DS4G_F32)
        cb2_dequant_kernel<DS4G_F32><<<grid, 256, 0, s>>>(blocks, n_blocks, cb, out);
    else if (dtype == DS4G_F16)
        cb2_dequant_kernel<DS4G_F16><<<grid, 256, 0, s>>>(blocks, n_blocks, cb, out);
    else
        cb2_dequant_kernel<DS4G_BF16><<<grid, 256, 0, s>>>(blocks, n_blocks, cb, out);
    return cudaGetLastError();
}

cudaError_t launch_kquant_dequant(int fmt, const uint8_t *blocks, int64_t n_blocks, void *out,
                                  int dtype, cudaStream_t s)
{
    const int grid = grid_for(n_blocks * 16);
    if (fmt == DS4G_FMT_Q4K)
        launch_kquant_fmt<DS4G_FMT_Q4K>(blocks, n_blocks, out, dtype, grid, s);
    else if (fmt == DS4G_FMT_Q5K)
        launch_kquant_fmt<DS4G_FMT_Q5K>(blocks, n_blocks, out, dtype, grid, s);
    else if (fmt == DS4G_FMT_MXFP4)
        launch_kquant_fmt<DS4G_FMT_MXFP4>(blocks, n_blocks, out, dtype, grid, s);
    else
        launch_kquant_fmt<DS4G_FMT_Q6K>(blocks, n_blocks, out, dtype, grid, s);
    return cudaGetLastError();
}

}  // namespace ds4g
