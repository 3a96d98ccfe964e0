// tc.cu -- the tensor-core path for Q2_K and codebook-2-bit experts: expert
// segments long enough that the layer is a dense contraction (prefill; ds4
// README mirror, "So, what can I do with this software?" names micro-batched
// prefill on CUDA).
//
// Per active expert e with segment rows P = offsets[e] .. offsets[e+1]-1
// (assignments in segment order):
//   gate/up kernel:  h[p, n] = SiLU(W_gate[e][n,:] . x_p) * (W_up[e][n,:] . x_p)
//   down kernel:     yslot[p, m] = w_p * (W_down[e][m,:] . h[p, :])
//   combine:         y[t, m] = sum_{i<k} yslot[slot(t,i), m]   (slot order)
//
// One work item is (token tile of up to 128 rows of one segment, 128 weight
// rows).  The weights are the MMA's M side, the tokens its N side, so one
// dequantized weight serves every token of the tile.
//
// Roles inside a CTA (one CTA per SM, persistent over the items):
//   warp 0     TMA producer: per 256-wide K step, the 16-byte aligned window
//              of each weight row's 84-byte super-block (a 3-D tensor map
//              over [experts][rows][row words]) and the activation tile (a
//              2-D tensor map over [segment rows][K], fp16, 128-byte swizzle)
//              land in a two-stage shared-memory ring;
//   warp 1     MMA issuer: tcgen05.mma kind::f16, A (dequantized weights)
//              from tensor memory, B (activations) from shared memory, fp32
//              accumulators in tensor memory;
//   warps 2-9  dequantizers, two warpgroups: each thread owns one weight row,
//              reads its block from shared memory, forms fp16 weights in
//              registers and stores them to tensor memory (tcgen05.st) as
//              the next A buffer.  In the gate/up kernel they are also the
//              epilogue after each item (tcgen05.ld of the accumulators,
//              SiLU*up, fp16 stores of h);
//   warps 10-13  down kernel only: the epilogue (tcgen05.ld, routing weight,
//              fp32 stores of yslot), on double-buffered accumulators so
//              the next item's MMAs overlap it.
//
// Weight values.  w = d*(sc&15)*q - dmin*(sc>>4) is formed on half2 pairs
// with two roundings, each relative to w (q2k_half below); the per-token
// relative L2 error of the layer stays near 5e-4.  The pair order inside
// each aligned group of 4 weights is (0, 2, 1, 3), the order the lop3
// extraction yields; the activation operand is stored in the same permuted
// order, so the contraction is unchanged.  Codebook-2-bit weights keep the
// natural order: each 8-weight codebook row comes from a 16-way replicated
// copy of the codebook in shared memory, c*s is formed exactly in fp16 and
// the single rounding is the multiply by d.
//
// Tensor memory (512 columns): columns 0..255 are two A buffers of 128
// columns (K = 128 fp16 per matrix-half pair, or K = 256 of one matrix);
// columns 256..383 and 384..511 are the fp32 accumulators (gate and up, or
// the down kernel's two alternating accumulators).  Every mbarrier wait is bounded; on expiry the kernel records
// DS4G_ERR_TIMEOUT in the status word, lets every role leave its loop,
// drains its own copies and MMAs (bounded) and frees its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ds4g_common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace ds4g {
namespace {

constexpr int kBM = 128;                  // weight rows per item (MMA M)
constexpr int kNT = kTcTileTokens;        // tokens per item at most (MMA N)
constexpr int kBoxRows = 16;              // token rows per activation TMA box
constexpr int kStages = 2;
constexpr int kWinWords = 28;             // 112-byte window per weight row
constexpr int kAqBytes = kWinWords * 4 * kBM;
constexpr int kChunkBytes = kNT * 128;    // one 64-wide K chunk of the activation tile
constexpr int kBBytes = 4 * kChunkBytes;
constexpr int kDequantWarps = 8;
constexpr int kEpilogueWarps = 4;          // down kernel: dedicated epilogue warps
__host__ __device__ constexpr int tc_threads(int mode)
{
    return (2 + kDequantWarps + (mode == 1 ? kEpilogueWarps : 0)) * 32;
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;

struct TcArgs {
    int K;                      // contraction length: hidden, or I_pad
    int m_tiles;                // weight-row tiles per expert
    int H, I_pad;
    const int32_t *tiles;       // [n][4]: expert, first segment row, rows, 0
    const int32_t *n_tiles;
    const float *wseg;          // routing weight of each segment row
    __half *hp;                 // gate/up output [A][I_pad] (permuted order)
    float *yslot;               // down output [A][H]
    const int8_t *codebook;     // [256 x 8] int8 (codebook format)
    int32_t *status;
    uint64_t wait_ns;
    int stall;                  // debug: the producer issues nothing (tests the bounded waits)
};

__device__ __forceinline__ int perm4(int n) { return (n & ~3) | ((n & 1) << 1) | ((n >> 1) & 1); }

__device__ __forceinline__ void set_status(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                         volatile int *abort_flag)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The 64 packed fp16 pairs (128 weights) of half `h` of one Q2_K block for
// this thread's row.  `w`: the block's 21 words (scales 0..3, qs 4..19,
// d|dmin 20).
//
// Per weight, with exact fp16 operands throughout:
//   v  = 1024 + q*4^g           lop3 of the 2-bit field in place (no shift)
//   n  = v*S + C = q*sc         S = sc*4^-g, C = -1024*S; exact (integer <= 45)
//   w1 = fp16(n*d + c_hi)       one rounding, relative to w itself
//   w  = fp16(w1 + c_lo)        c_hi + c_lo = -dmin*m exactly (c_lo from an fma)
// Rounding d*sc or dmin*m to fp16 before the subtraction instead would be
// amplified by the cancellation between the two terms of a Q2_K weight.
__device__ __forceinline__ void q2k_half(const uint32_t *w, int h, uint32_t (&out)[64])
{
    const uint32_t dd = w[20];
    const uint32_t d2 = __byte_perm(dd, 0, 0x1010);                    // (d, d)
    const uint32_t ndmin2 = __byte_perm(dd, 0, 0x3232) ^ 0x80008000u;  // (-dmin, -dmin)
    const uint32_t k1024 = 0x64006400u, kn1024 = 0xE400E400u;
    // 4^-g and -1024 * 4^-g, g = 0..3, replicated fp16
    const uint32_t p4[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};
    const uint32_t c4[4] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u};
    uint32_t S2[8], C2[8], HI2[8], LO2[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint32_t sw = w[2 * h + (s >> 2)];
        const uint32_t j = (uint32_t)(s & 3);
        const uint32_t rep = __byte_perm(sw, 0, 0x4040u | j | (j << 8));   // byte j twice
        const uint32_t sc2 = ptx::lop3_and_or(rep, 0x000F000Fu, k1024);       // 1024 + sc
        const uint32_t mn2 = ptx::lop3_and_or(rep >> 4, 0x000F000Fu, k1024);  // 1024 + m
        S2[s] = ptx::hfma2_u(sc2, p4[s >> 1], c4[s >> 1]);                   // sc * 4^-g
        C2[s] = ptx::hmul2_u(S2[s], kn1024);
        const uint32_t mnf = ptx::hsub2_u(mn2, k1024);                       // m
        HI2[s] = ptx::hmul2_u(mnf, ndmin2);
        LO2[s] = ptx::hfma2_u(mnf, ndmin2, HI2[s] ^ 0x80008000u);
    }
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
        const uint32_t qw = w[4 + 8 * h + wd];
        const uint32_t qh = qw >> 8;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int s = 2 * g + (wd >> 2);
            const uint32_t mask = 0x00030003u << (2 * g);
            const uint32_t v0 = ptx::lop3_and_or(qw, mask, k1024);
            const uint32_t v1 = ptx::lop3_and_or(qh, mask, k1024);
            const uint32_t n0 = ptx::hfma2_u(v0, S2[s], C2[s]);
            const uint32_t n1 = ptx::hfma2_u(v1, S2[s], C2[s]);
            out[16 * g + 2 * wd] = ptx::hadd2_u(ptx::hfma2_u(n0, d2, HI2[s]), LO2[s]);
            out[16 * g + 2 * wd + 1] = ptx::hadd2_u(ptx::hfma2_u(n1, d2, HI2[s]), LO2[s]);
        }
    }
}

// Dequantizes half HALF of this thread's row block (the block starts at word
// SH of the 112-byte window `win`) and stores it to tensor-memory columns
// taddr.col .. +63 of this warp's 32 lanes.
template <int SH, int HALF>
__device__ __forceinline__ void dequant_store(const uint32_t (&win)[24], uint32_t taddr)
{
    uint32_t out[64];
    q2k_half(win + SH, HALF, out);
    ptx::tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&out[0]));
    ptx::tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&out[32]));
}

// Register arrays are only indexed with constants: dispatch on the
// (warp-uniform) word offset and half.
__device__ __forceinline__ void dequant_store_sh(const uint32_t (&win)[24], int sh, int half,
                                                 uint32_t taddr)
{
    switch (sh * 2 + half) {
    case 0: dequant_store<0, 0>(win, taddr); break;
    case 1: dequant_store<0, 1>(win, taddr); break;
    case 2: dequant_store<1, 0>(win, taddr); break;
    case 3: dequant_store<1, 1>(win, taddr); break;
    case 4: dequant_store<2, 0>(win, taddr); break;
    case 5: dequant_store<2, 1>(win, taddr); break;
    case 6: dequant_store<3, 0>(win, taddr); break;
    default: dequant_store<3, 1>(win, taddr); break;
    }
}

// ---------------------------------------------------------------------------
// Codebook-2-bit blocks (70 bytes: idx[32], sgn[32], 4-bit scales sc[4], d).
// Per group of 8 weights one 8-byte codebook row is read from a shared-memory
// copy replicated 16 times, so the 16 lanes of a half-warp never share a bank
// whatever their indices.  Per pair of weights:
//   v = 1024 + (c + 128)          byte-biased int8 OR-ed into fp16 1024 (prmt)
//   n = v * s - 1152 * s = c * s  exact (|c * s| <= 645)
//   n ^= sign bits                the weight's sign from the sign byte
//   w = fp16(n * d)               one rounding, relative to w
// Weights stay in natural order; the activation operand is stored likewise.
// ---------------------------------------------------------------------------
constexpr int kCbCopies = 16;
constexpr int kCbRepBytes = 256 * kCbCopies * 8;

template <int WO, int HALF>
__device__ __forceinline__ void cb2_store(const uint32_t (&win)[24], uint32_t fs, uint32_t cb_lane,
                                          uint32_t taddr)
{
    // the block's words (it starts fs/8 bytes into word WO of the window)
    auto word = [&](int i) -> uint32_t { return __funnelshift_r(win[WO + i], win[WO + i + 1], fs); };
    const uint32_t d2 = __byte_perm(word(17), 0, 0x1010);
    const uint32_t scw = word(16);
    uint32_t s2[4], ns2[4], idxw[4], sgnw[4];
#pragma unroll
    for (int G = 0; G < 4; ++G) {
        const float sf = (float)((scw >> (4 * (4 * HALF + G))) & 15u);
        s2[G] = ptx::pack_half2(sf, sf);
        ns2[G] = ptx::pack_half2(-1152.0f * sf, -1152.0f * sf);
        idxw[G] = word(4 * HALF + G);
        sgnw[G] = word(8 + 4 * HALF + G);
    }
    uint32_t out[64];
#pragma unroll
    for (int o = 0; o < 16; ++o) {
        const uint32_t idx = (idxw[o >> 2] >> (8 * (o & 3))) & 0xFFu;
        const uint32_t sg = (sgnw[o >> 2] >> (8 * (o & 3))) & 0xFFu;
        const int G = o >> 2;
        uint32_t cw[2];
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(cw[0]), "=r"(cw[1]) : "r"(cb_lane + idx * (kCbCopies * 8)));
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t wb = cw[q] ^ 0x80808080u;
            const uint32_t v0 = __byte_perm(wb, 0x64646464u, 0x4140);
            const uint32_t v1 = __byte_perm(wb, 0x64646464u, 0x4342);
            const uint32_t x = sg >> (4 * q);
            const uint32_t m0 = ((x & 1u) << 15) | ((x & 2u) << 30);
            const uint32_t m1 = ((x & 4u) << 13) | ((x & 8u) << 28);
            out[4 * o + 2 * q] = ptx::hmul2_u(ptx::hfma2_u(v0, s2[G], ns2[G]) ^ m0, d2);
            out[4 * o + 2 * q + 1] = ptx::hmul2_u(ptx::hfma2_u(v1, s2[G], ns2[G]) ^ m1, d2);
        }
    }
    ptx::tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&out[0]));
    ptx::tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&out[32]));
}

__device__ __forceinline__ void cb2_store_off(const uint32_t (&win)[24], int byteoff, int half,
                                              uint32_t cb_lane, uint32_t taddr)
{
    const uint32_t fs = (uint32_t)(byteoff & 3) * 8;
    switch ((byteoff >> 2) * 2 + half) {
    case 0: cb2_store<0, 0>(win, fs, cb_lane, taddr); break;
    case 1: cb2_store<0, 1>(win, fs, cb_lane, taddr); break;
    case 2: cb2_store<1, 0>(win, fs, cb_lane, taddr); break;
    case 3: cb2_store<1, 1>(win, fs, cb_lane, taddr); break;
    case 4: cb2_store<2, 0>(win, fs, cb_lane, taddr); break;
    case 5: cb2_store<2, 1>(win, fs, cb_lane, taddr); break;
    case 6: cb2_store<3, 0>(win, fs, cb_lane, taddr); break;
    default: cb2_store<3, 1>(win, fs, cb_lane, taddr); break;
    }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(tc_threads(MODE), 1)
    tc_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
              const __grid_constant__ CUtensorMap tm_b, const TcArgs a)
{
    constexpr int NMAT = MODE == 0 ? 2 : 1;
    constexpr uint32_t kStageBytes = kBBytes + NMAT * kAqBytes;
    constexpr int kFills = MODE == 0 ? 2 : 1;     // A buffers per K step
    constexpr int kBlockBytes = FMT == DS4G_FMT_Q2K ? kQ2KBytes : kCB2Bytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], afull[2], aempty[2];
    __shared__ __align__(8) uint64_t accfull[2], accempty[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_issued;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&afull[b], kDequantWarps);
            ptx::mbar_init(&aempty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&accfull[b], 1);
            ptx::mbar_init(&accempty[b], MODE == 0 ? kDequantWarps : kEpilogueWarps);
        }
        ptx::mbar_init(&drain, 1);
        ptx::fence_mbar_init();
        s_abort = 0;
        s_issued = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(&s_tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    uint8_t *cbrep = smem + (size_t)kStages * kStageBytes;    // codebook format only
    if (FMT == DS4G_FMT_CB2) {
        for (int i = threadIdx.x; i < 256 * kCbCopies; i += blockDim.x) {
            const int r = i / kCbCopies, cpy = i % kCbCopies;
            uint8_t *dst = cbrep + r * (kCbCopies * 8) + cpy * 8;
#pragma unroll
            for (int b = 0; b < 8; ++b) dst[b] = (uint8_t)a.codebook[8 * r + b];
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int *abort_flag = &s_abort;

    const int n_items = *a.n_tiles * a.m_tiles;
    const int KB = a.K / kQK;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0 && !a.stall) {
            ptx::prefetch_tmap(&tm_a0);
            if (NMAT == 2) ptx::prefetch_tmap(&tm_a1);
            ptx::prefetch_tmap(&tm_b);
            int sc = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int tile = it / a.m_tiles, mt = it % a.m_tiles;
                const int e = a.tiles[4 * tile], row0 = a.tiles[4 * tile + 1];
                const int nb = (a.tiles[4 * tile + 2] + kBoxRows - 1) / kBoxRows;
                const uint32_t bytes = NMAT * kAqBytes + 4u * nb * kBoxRows * 128u;
                for (int kb = 0; kb < KB; ++kb, ++sc) {
                    const int s = sc % kStages;
                    if (sc >= kStages &&
                        !wait_bar(&empty[s], ((sc / kStages) - 1) & 1, a.wait_ns, abort_flag)) {
                        set_status(a.status, DS4G_ERR_TIMEOUT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + (size_t)s * kStageBytes;
                    ptx::mbar_arrive_expect_tx(&full[s], bytes);
                    for (int kc = 0; kc < 4; ++kc)
                        for (int r = 0; r < nb; ++r)
                            ptx::tma_load_2d(st + kc * kChunkBytes + r * kBoxRows * 128, &tm_b,
                                             kb * kQK + 64 * kc, row0 + kBoxRows * r, &full[s]);
                    const int x = ((kBlockBytes * kb) & ~15) / 4;
                    ptx::tma_load_3d(st + kBBytes, &tm_a0, x, mt * kBM, e, &full[s]);
                    if (NMAT == 2)
                        ptx::tma_load_3d(st + kBBytes + kAqBytes, &tm_a1, x, mt * kBM, e, &full[s]);
                    s_issued = sc + 1;
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int sc = 0, fc = 0, ic = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++ic) {
                const int tile = it / a.m_tiles;
                const int nb = (a.tiles[4 * tile + 2] + kBoxRows - 1) / kBoxRows;
                const uint32_t idesc = ptx::idesc_f16(kBM, nb * kBoxRows);
                // gate/up: one accumulator pair; down: two accumulators, so the
                // epilogue warps drain one while the next item accumulates
                const int ab = MODE == 1 ? (ic & 1) : 0;
                const int uses = MODE == 1 ? (ic >> 1) : ic;
                if (uses > 0 && !wait_bar(&accempty[ab], (uses - 1) & 1, a.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t acc_col = kAccCol + 128u * ab;
                for (int kb = 0; ok && kb < KB; ++kb, ++sc) {
                    const int s = sc % kStages;
                    if (!wait_bar(&full[s], (sc / kStages) & 1, a.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t b_base = ptx::smem_addr(smem + (size_t)s * kStageBytes);
                    for (int h = 0; h < kFills; ++h, ++fc) {
                        const int buf = fc & 1;
                        if (!wait_bar(&afull[buf], (fc >> 1) & 1, a.wait_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t a_buf = tmem + (uint32_t)buf * 128u;
                        if (MODE == 0) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int kk = 128 * h + 16 * i;
                                const uint64_t bd = ptx::sw128_desc(
                                    b_base + (kk >> 6) * kChunkBytes + (kk & 63) * 2);
                                const bool acc = !(kb == 0 && h == 0 && i == 0);
                                ptx::mma_f16_ts(tmem + kAccCol, a_buf + 8 * i, bd, idesc, acc);
                                ptx::mma_f16_ts(tmem + kAccCol + 128, a_buf + 64 + 8 * i, bd, idesc,
                                                acc);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int kk = 16 * i;
                                const uint64_t bd = ptx::sw128_desc(
                                    b_base + (kk >> 6) * kChunkBytes + (kk & 63) * 2);
                                ptx::mma_f16_ts(tmem + acc_col, a_buf + 8 * i, bd, idesc,
                                                !(kb == 0 && i == 0));
                            }
                        }
                        ptx::mma_commit(&aempty[buf]);
                    }
                    if (!ok) break;
                    ptx::mma_commit(&empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&accfull[ab]);
            }
            if (!ok) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread is complete before the CTA
            // frees its tensor memory
            ptx::mma_commit(&drain);
            ptx::mbar_wait(&drain, 0, a.wait_ns);
        }
    } else if (warp >= 2 + kDequantWarps) {
        // ---------------- down epilogue warps (MODE 1) ----------------
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        int ic = 0;
        bool ok = true;
        for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++ic) {
            const int tile = it / a.m_tiles, mt = it % a.m_tiles;
            const int row0 = a.tiles[4 * tile + 1], nlen = a.tiles[4 * tile + 2];
            const int ab = ic & 1;
            ok = wait_bar(&accfull[ab], (ic >> 1) & 1, a.wait_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int m = mt * kBM + row;
            const uint32_t acc = tmem + lane_base + kAccCol + 128u * ab;
            for (int c = 0; 8 * c < nlen; ++c) {
                float o[8];
                ptx::tmem_ld8(acc + 8 * c, o);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = 8 * c + j;
                    if (t < nlen) {
                        const int pos = row0 + t;
                        a.yslot[(size_t)pos * a.H + m] = __ldg(a.wseg + pos) * o[j];
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&accempty[ab]);
        }
        if (!ok) {
            if (lane == 0) set_status(a.status, DS4G_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ---------------- dequantizers / gate-up epilogue ----------------
        const int dw = warp - 2;                 // 0..7
        const int wg = dw >> 2;                  // warpgroup: matrix (gate/up) or half
        const int quarter = warp & 3;            // tensor-memory lane quarter
        const int row = 32 * quarter + lane;
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        int sc = 0, fc = 0, ic = 0;
        bool ok = true;
        for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++ic) {
            const int tile = it / a.m_tiles, mt = it % a.m_tiles;
            const int row0 = a.tiles[4 * tile + 1], nlen = a.tiles[4 * tile + 2];
            for (int kb = 0; ok && kb < KB; ++kb, ++sc) {
                const int s = sc % kStages;
                ok = wait_bar(&full[s], (sc / kStages) & 1, a.wait_ns, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint8_t *aq = smem + (size_t)s * kStageBytes + kBBytes +
                                    (MODE == 0 ? wg * kAqBytes : 0) + row * (kWinWords * 4);
                uint32_t win[24];
#pragma unroll
                for (int v = 0; v < 6; ++v) {
                    const uint4 q = reinterpret_cast<const uint4 *>(aq)[v];
                    win[4 * v] = q.x;
                    win[4 * v + 1] = q.y;
                    win[4 * v + 2] = q.z;
                    win[4 * v + 3] = q.w;
                }
                const int sh = kb & 3;       // (84 * kb) mod 16, in words (Q2_K)
                const int boff = (kBlockBytes * kb) & 15;   // block start in the window, bytes
                for (int h = 0; h < kFills; ++h, ++fc) {
                    const int buf = fc & 1;
                    if (fc >= 2) {
                        ok = wait_bar(&aempty[buf], ((fc >> 1) - 1) & 1, a.wait_ns, abort_flag);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ptx::tc_fence_after();
                    }
                    const uint32_t taddr = tmem + lane_base + (uint32_t)buf * 128u + 64u * wg;
                    if (FMT == DS4G_FMT_Q2K)
                        dequant_store_sh(win, sh, MODE == 0 ? h : wg, taddr);
                    else
                        cb2_store_off(win, boff, MODE == 0 ? h : wg,
                                      ptx::smem_addr(cbrep) + (uint32_t)(lane & 15) * 8, taddr);
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&afull[buf]);
                }
            }
            if (!ok) break;
            if (MODE == 1) continue;                 // the epilogue warps finish down items
            // epilogue of the item
            ok = wait_bar(&accfull[0], ic & 1, a.wait_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int chunks = (nlen + 7) / 8;
            for (int c = wg; c < chunks; c += 2) {
                if (MODE == 0) {
                    float g[8], u[8];
                    ptx::tmem_ld8(tmem + lane_base + kAccCol + 8 * c, g);
                    ptx::tmem_ld8(tmem + lane_base + kAccCol + 128 + 8 * c, u);
                    ptx::tmem_ld_wait();
                    const int n = mt * kBM + row;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int t = 8 * c + j;
                        if (t < nlen)
                            a.hp[(size_t)(row0 + t) * a.I_pad + (FMT == DS4G_FMT_Q2K ? perm4(n) : n)] =
                                __float2half_rn(silu_mul(g[j], u[j]));
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&accempty[0]);
        }
        if (!ok) {
            if (lane == 0) set_status(a.status, DS4G_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    // after an abort: the copies this CTA issued land before it exits
    if (threadIdx.x == 0 && *abort_flag) {
        const int issued = s_issued;
        for (int q = issued - kStages; q < issued; ++q) {
            if (q < 0) continue;
            if (!ptx::mbar_wait(&full[q % kStages], (q / kStages) & 1, a.wait_ns)) break;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Token tiles of every active segment and the activation gather:
//   tiles[j] = (expert, first segment row, rows <= kNT, 0), heaviest expert
//   segments are not reordered; *n_tiles = count; wseg[p] = wts[perm[p]];
//   xseg[p, :] = fp16(x[perm[p] / k, :]), in the (0, 2, 1, 3) order per 4
//   for Q2_K (permute4), in natural order for the codebook format.
__global__ void __launch_bounds__(256) tc_prep_kernel(const uint16_t *__restrict__ x, int H, int k,
                                                      int A, const int32_t *__restrict__ perm,
                                                      const int32_t *counts,
                                                      const int32_t *offsets, int E,
                                                      __half *__restrict__ xseg, int32_t *tiles,
                                                      int32_t *n_tiles, int permute4,
                                                      const float *__restrict__ wts,
                                                      float *__restrict__ wseg)
{
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < A; p += gridDim.x * blockDim.x)
        wseg[p] = wts[perm[p]];
    if (blockIdx.x == 0) {
        __shared__ int s_nt[DS4G_MAX_EXPERTS];
        __shared__ int s_base[DS4G_MAX_EXPERTS + 1];
        const int e = threadIdx.x;
        if (e < DS4G_MAX_EXPERTS) s_nt[e] = e < E ? (counts[e] + kNT - 1) / kNT : 0;
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = 0;
            for (int i = 0; i < E; ++i) {
                s_base[i] = run;
                run += s_nt[i];
            }
            s_base[E] = run;
            *n_tiles = run;
        }
        __syncthreads();
        if (e < E) {
            const int c = counts[e], o = offsets[e];
            for (int j = 0; j < s_nt[e]; ++j) {
                int32_t *t = tiles + 4 * (s_base[e] + j);
                t[0] = e;
                t[1] = o + j * kNT;
                t[2] = min(kNT, c - j * kNT);
                t[3] = 0;
            }
        }
    }
    const int per_row = H / 8;
    const int64_t total = (int64_t)A * per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / per_row), c = (int)(i % per_row);
        const int t = perm[p] / k;
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * H) + c);
        const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
        __half hv[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hv[2 * j] = __float2half_rn(bf16_bits(wv[j] & 0xFFFFu));
            hv[2 * j + 1] = __float2half_rn(bf16_bits(wv[j] >> 16));
        }
        // Q2_K: (0, 2, 1, 3) inside each group of 4; codebook format: natural
        const __half2 o0 = permute4 ? __halves2half2(hv[0], hv[2]) : __halves2half2(hv[0], hv[1]);
        const __half2 o1 = permute4 ? __halves2half2(hv[1], hv[3]) : __halves2half2(hv[2], hv[3]);
        const __half2 o2 = permute4 ? __halves2half2(hv[4], hv[6]) : __halves2half2(hv[4], hv[5]);
        const __half2 o3 = permute4 ? __halves2half2(hv[5], hv[7]) : __halves2half2(hv[6], hv[7]);
        uint4 out;
        out.x = *reinterpret_cast<const uint32_t *>(&o0);
        out.y = *reinterpret_cast<const uint32_t *>(&o1);
        out.z = *reinterpret_cast<const uint32_t *>(&o2);
        out.w = *reinterpret_cast<const uint32_t *>(&o3);
        reinterpret_cast<uint4 *>(xseg + (size_t)p * H)[c] = out;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// 2-D map over [rows][K] fp16 activations: box = 64 (128 bytes) x 16 rows,
// 128-byte swizzle, zero fill beyond the last row.
cudaError_t act_map(CUtensorMap *m, const void *base, int64_t K, int64_t rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kBoxRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE, int FMT>
cudaError_t launch_tc(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                      const TcArgs &args, int grid, cudaStream_t s)
{
    constexpr int NMAT = MODE == 0 ? 2 : 1;
    const size_t smem = (size_t)kStages * (kBBytes + NMAT * kAqBytes) + 1024 +
                        (FMT == DS4G_FMT_CB2 ? kCbRepBytes : 0);
    cudaError_t e = cudaFuncSetAttribute(tc_kernel<MODE, FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tc_kernel<MODE, FMT><<<grid, tc_threads(MODE), smem, s>>>(a0, a1, b, args);
    return cudaGetLastError();
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

// 3-D map over [experts][rows][row words] of one quantized weight tensor:
// box = 28 words (112 bytes) x 128 rows x 1 expert, no swizzle, zero fill.
cudaError_t weight_map(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows,
                       int64_t expert_stride, int64_t experts, int phases)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    // `phases` consecutive rows form one super-row (phases * row_bytes is a
    // multiple of 16); the box covers 128 / phases super-rows
    cuuint64_t dims[3] = {(cuuint64_t)(phases * row_bytes / 4), (cuuint64_t)(rows / phases),
                          (cuuint64_t)experts};
    cuuint64_t strides[2] = {(cuuint64_t)(phases * row_bytes), (cuuint64_t)expert_stride};
    cuuint32_t box[3] = {(cuuint32_t)kWinWords, (cuuint32_t)(kBM / phases), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_path_supported(const Plan &p, const ds4g_moe_desc *d)
{
    return p.A > 0 && d->gate_up_row_bytes % 16 == 0 && d->down_row_bytes % 16 == 0 &&
           p.H % kBM == 0;
}

int32_t tc_max_tiles(int32_t E, int32_t A) { return E + A / kNT + 1; }

cudaError_t launch_tc_prep(const LayerArgs &la, const TcBufs &tb, const DeviceInfo &dev,
                           cudaStream_t s)
{
    const int prep_grid = dev.sm_count * 4;
    tc_prep_kernel<<<prep_grid, 256, 0, s>>>(la.x, la.H, la.k, la.A, la.perm, la.counts,
                                             la.offsets, la.E, tb.xseg, tb.tiles, tb.n_tiles,
                                             la.format == DS4G_FMT_Q2K ? 1 : 0, la.wts, tb.wseg);
    return cudaGetLastError();
}

cudaError_t launch_tc_path(const LayerArgs &la, const TcBufs &tb, const DeviceInfo &dev,
                           cudaStream_t s, const cudaEvent_t *ev, uint64_t wait_ns,
                           bool stall)
{
    CUtensorMap m_gate, m_up, m_down, m_x, m_h;
    cudaError_t e;
    if ((e = weight_map(&m_gate, la.w_gate, la.gu_row, la.I, la.gu_stride, la.E, 1)) != cudaSuccess ||
        (e = weight_map(&m_up, la.w_up, la.gu_row, la.I, la.gu_stride, la.E, 1)) != cudaSuccess ||
        (e = weight_map(&m_down, la.w_down, la.dn_row, la.H, la.dn_stride, la.E, 1)) != cudaSuccess ||
        (e = act_map(&m_x, tb.xseg, la.H, la.A)) != cudaSuccess ||
        (e = act_map(&m_h, tb.hp, la.I_pad, la.A)) != cudaSuccess)
        return e;

    TcArgs a{};
    a.H = la.H;
    a.I_pad = la.I_pad;
    a.tiles = tb.tiles;
    a.n_tiles = tb.n_tiles;
    a.wseg = tb.wseg;
    a.hp = tb.hp;
    a.yslot = la.yslot;
    a.status = tb.status;
    a.wait_ns = wait_ns;
    a.stall = stall ? 1 : 0;

    a.K = la.H;
    a.m_tiles = la.I_pad / kBM;
    a.codebook = la.codebook;
    const bool cb2 = la.format == DS4G_FMT_CB2;
    if ((e = cb2 ? launch_tc<0, DS4G_FMT_CB2>(m_gate, m_up, m_x, a, dev.sm_count, s)
                 : launch_tc<0, DS4G_FMT_Q2K>(m_gate, m_up, m_x, a, dev.sm_count, s)) != cudaSuccess)
        return e;
    if (ev && (e = record_phase(ev[2], s)) != cudaSuccess) return e;

    a.K = la.I_pad;
    a.m_tiles = la.H / kBM;
    if ((e = cb2 ? launch_tc<1, DS4G_FMT_CB2>(m_down, m_down, m_h, a, dev.sm_count, s)
                 : launch_tc<1, DS4G_FMT_Q2K>(m_down, m_down, m_h, a, dev.sm_count, s)) != cudaSuccess)
        return e;
    if (ev && (e = record_phase(ev[3], s)) != cudaSuccess) return e;

    if ((e = launch_combine(la, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[4], s)) != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ds4g
