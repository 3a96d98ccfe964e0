// kquant.cuh -- device decoders of the routed-expert formats beyond the
// 2-bit ones: Q4_K and Q5_K (routed gate/up and down) and Q6_K (routed down),
// the GGUF K-quant super-blocks of 256 weights, and MXFP4 (ds4 README mirror,
// "Model Weights", which lists the routed expert formats and the ds4f-mxfp4
// download, and "Acknowledgements to llama.cpp and GGML" for the GGUF
// layouts).  MXFP4 (OCP microscaling FP4): 17-byte blocks of 32 weights, an
// E8M0 scale byte then 16 bytes of E2M1 codes (weight i low nibble of byte
// 1 + i, weight i + 16 high nibble); w = 2^(e-127) * value.
//
//   Q4_K (144 B): d fp16 @0, dmin fp16 @2, 12 packed scale bytes @4, qs @16
//   Q5_K (176 B): d @0, dmin @2, packed scales @4, qh[32] @16, qs @48
//   Q6_K (210 B): ql[128] @0, qh[64] @128, int8 scales[16] @192, d fp16 @208
//
// Q4_K / Q5_K: eight 32-weight sub-blocks with 6-bit scale sc_s and min m_s
// (sub-blocks 0..3 in the low six bits of bytes 0..3 / 4..7, sub-blocks 4..7
// in the nibbles of bytes 8..11 with their top two bits in the top bits of
// bytes 0..7); weight 64c + l / 64c + 32 + l in the low / high nibble of
// qs[32c + l]; Q5_K's fifth bit of weight 32s + l is bit s of qh[l];
//   w = d * sc_s * q - dmin * m_s.
// Q6_K: weight j (h = j/128, u = (j%128)/32, l = j%32) has its low nibble in
// nibble u>>1 of ql[64h + 32(u&1) + l], its top two bits in bits 2u, 2u+1 of
// qh[32h + l]; q = that 6-bit value - 32;  w = d * scales[j/16] * q.
// Every product is exact in fp32 (at most 24 significant bits), so the
// values below are exactly the definitions' (one rounding, in the
// subtraction, for Q4_K / Q5_K; none for Q6_K).
#pragma once

#include "ds4g_common.cuh"

namespace ds4g {

// 6-bit scale and min of sub-block s of a Q4_K / Q5_K block (p = byte 4).
__device__ __forceinline__ void k4_scale_min(const uint8_t *__restrict__ p, int s, int &sc, int &m)
{
    if (s < 4) {
        sc = __ldg(p + s) & 63;
        m = __ldg(p + s + 4) & 63;
    } else {
        const int b = __ldg(p + s + 4);
        sc = (b & 15) | ((__ldg(p + s - 4) >> 6) << 4);
        m = (b >> 4) | ((__ldg(p + s) >> 6) << 4);
    }
}

// 16 consecutive bytes starting at a 16-byte offset of a block that is at
// least 2-byte aligned (Q6_K) or 4-byte aligned (Q4_K, Q5_K).
template <int ALIGN4>
__device__ __forceinline__ void load16(const uint8_t *__restrict__ p, uint32_t (&v)[4])
{
    if (ALIGN4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(reinterpret_cast<const uint32_t *>(p) + i);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = __ldg(reinterpret_cast<const uint16_t *>(p) + 2 * i);
            const uint32_t hi = __ldg(reinterpret_cast<const uint16_t *>(p) + 2 * i + 1);
            v[i] = lo | (hi << 16);
        }
    }
}

__device__ __forceinline__ int byte_of(const uint32_t (&v)[4], int i)
{
    return (v[i >> 2] >> (8 * (i & 3))) & 0xFF;
}

// E2M1 value of a 4-bit code: bit 3 the sign, bits 0..2 the magnitude
// 0, 0.5, 1, 1.5, 2, 3, 4, 6: exponent field m >> 1, mantissa bit m & 1;
// exponent 0 is the subnormal 0 / 0.5, exponent x >= 1 gives
// (2 + mantissa) * 2^(x-1) / 2 (integer arithmetic, then an exact halving).
__device__ __forceinline__ float e2m1_value(int code)
{
    const int m = code & 7;
    const float mag = m < 2 ? 0.5f * (float)m : 0.5f * (float)((2 + (m & 1)) << ((m >> 1) - 1));
    return (code & 8) ? -mag : mag;
}

// fp32 weights 16u .. 16u+15 of one K-quant super-block (FMT = DS4G_FMT_Q4K,
// DS4G_FMT_Q5K or DS4G_FMT_Q6K) or MXFP4 unit of eight blocks (the low (u
// even) or high (u odd) nibbles of block u/2: weights 16 (u&1) .. +15 of it).
template <int FMT>
__device__ __forceinline__ void kquant_unit16(const uint8_t *__restrict__ blk, int u, float (&w)[16])
{
    if constexpr (FMT == DS4G_FMT_MXFP4) {
        // the unit (eight 17-byte blocks) is 4-byte aligned: block b's codes
        // start at byte 17b + 1, (b + 1) & 3 bytes into an aligned word, and
        // the aligned words that hold them end inside the unit
        const int b = u >> 1;
        const uint32_t e = __ldg(blk + 17 * b);
        // 2^(e-127): e = 0 is the subnormal 2^-127, e = 255 NaN
        const float scale = e == 0 ? __uint_as_float(0x00400000u)
                          : e == 255 ? __uint_as_float(0x7FC00000u)
                                     : __uint_as_float(e << 23);
        const int mis = (b + 1) & 3;
        const uint32_t *w4 = reinterpret_cast<const uint32_t *>(blk + ((17 * b + 1) & ~3));
        uint32_t v[5];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(w4 + i);
        v[4] = mis ? __ldg(w4 + 4) : 0u;
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __funnelshift_r(v[i], v[i + 1], 8 * mis);
        const int sh = 4 * (u & 1);
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = scale * e2m1_value((byte_of(q, i) >> sh) & 15);
    } else if constexpr (FMT == DS4G_FMT_Q4K || FMT == DS4G_FMT_Q5K) {
        const int s = u >> 1;                       // 32-weight sub-block
        const int c = u >> 2;                       // 64-weight chunk
        const int l0 = 16 * (u & 1);                // first lane
        const int hi = (u >> 1) & 1;                // high nibble for odd sub-blocks
        const uint32_t dd = (uint32_t)__ldg(reinterpret_cast<const uint16_t *>(blk)) |
                            ((uint32_t)__ldg(reinterpret_cast<const uint16_t *>(blk) + 1) << 16);
        const float d = half_bits(dd & 0xFFFFu), dmin = half_bits(dd >> 16);
        int sc, m;
        k4_scale_min(blk + 4, s, sc, m);
        const float scale_part = d * (float)sc;
        const float min_part = dmin * (float)m;
        uint32_t qs[4];
        load16<1>(blk + (FMT == DS4G_FMT_Q4K ? 16 : 48) + 32 * c + l0, qs);
        uint32_t qh[4] = {0, 0, 0, 0};
        if constexpr (FMT == DS4G_FMT_Q5K) load16<1>(blk + 16 + l0, qh);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            int q = (byte_of(qs, i) >> (4 * hi)) & 15;
            if constexpr (FMT == DS4G_FMT_Q5K) q += 16 * ((byte_of(qh, i) >> s) & 1);
            w[i] = scale_part * (float)q - min_part;
        }
    } else {
        static_assert(FMT == DS4G_FMT_Q6K, "K-quant format");
        const int h = u >> 3;                       // 128-weight half
        const int uq = (u & 7) >> 1;                // 32-weight quarter of the half
        const int l0 = 16 * (u & 1);
        const float d = half_bits(__ldg(reinterpret_cast<const uint16_t *>(blk + 208)));
        const float scale_part = d * (float)(int8_t)__ldg(blk + 192 + u);
        uint32_t ql[4], qh[4];
        load16<0>(blk + 64 * h + 32 * (uq & 1) + l0, ql);
        load16<0>(blk + 128 + 32 * h + l0, qh);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int low = (byte_of(ql, i) >> (4 * (uq >> 1))) & 15;
            const int high = (byte_of(qh, i) >> (2 * uq)) & 3;
            w[i] = scale_part * (float)(low + 16 * high - 32);
        }
    }
}

}  // namespace ds4g
