// tc.cu -- the tensor-core path for every routed-expert format (Q2_K,
// codebook-2-bit, Q4_K, Q5_K, Q6_K for W_down, MXFP4; any mix per matrix):
// the weights are dequantized to fp16 into tensor memory and contracted with
// tcgen05 MMAs, for every call above three tokens whose rows can be staged
// (ds4 README mirror, "So, what can I do with this software?" names
// micro-batched decode and prefill on CUDA; "Model Weights" the formats).
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
// The pipeline unit is the half block: 128 weights of every row of the item
// (one half of a 256-weight super-block), one fill of a 64-column A buffer in
// tensor memory, eight K = 16 MMAs.  Each team of dequantizing warps has its
// own two A buffers, so a buffer is dequantized again only after the team's
// other fill: the time one thread needs to issue a fill's MMAs (about 100-150
// cycles per tcgen05.mma while the dequantizing warps run, whatever the token
// count) and their completion overlap the dequantization of the next fill,
// and the two teams' hand-off latencies (tensor-memory stores, barrier
// arrivals and waits) overlap each other's arithmetic.  In the gate/up kernel
// each team feeds its own issuer (one per matrix), so the teams never wait for
// each other's fills.
//
// Roles inside a CTA (one CTA per SM, persistent over the items):
//   warp 0     weight producer: per 256-wide K step, the 16-byte aligned
//              window of each weight row's super-block (a 3-D tensor map
//              over [experts][rows][row words]) into a ring of window stages
//              that the dequantizers release once they have read them; the
//              windows a few K steps ahead are prefetched into L2;
//   warp 1     activation producer: per half K step, the activation tile
//              (a 2-D tensor map over [segment rows][K], fp16, 128-byte
//              swizzle) into a ring of half stages that the MMAs release;
//   warps 2-3  MMA issuers: tcgen05.mma kind::f16, A (dequantized weights)
//              from tensor memory, B (activations) from shared memory, fp32
//              accumulators in tensor memory.  Gate/up kernel: warp 2 issues
//              every W_gate fill, warp 3 every W_up fill.  Down kernel: warp
//              2 alone;
//   warps 4-19 dequantizers, two teams of two warpgroups (gate/up kernel:
//              team t dequantizes matrix t; Q2_K down kernel: team t the K
//              steps of parity t): each thread owns one weight row and, per
//              fill (one half of the block), the field pair 2*gh, 2*gh+1
//              (Q2_K) or weights 64*gh .. +63 (codebook) of the half: 64
//              weights, 32 fp16 pairs formed in registers and stored to
//              tensor memory (tcgen05.st).  In the gate/up kernel the sixteen warps are
//              also the epilogue after each item (tcgen05.ld of the
//              accumulators, SiLU*up, fp16 stores of h);
//   warps 20-23  down kernel only: the epilogue (tcgen05.ld, routing weight,
//              fp32 stores of yslot), on double-buffered accumulators so
//              the next item's MMAs overlap it.
//
// Weight values.  w = d*(sc&15)*q - dmin*(sc>>4) is formed on half2 pairs
// with two roundings, each relative to w (q2k_quarter below); the per-token
// relative L2 error of the layer stays near 5e-4.  A pair holds weights l
// and l+16 of one 32-weight field group: they lie in the two sub-blocks of
// the group, so one half2 of scales serves both lanes without replication.
// Inside every aligned group of 32, weight 16b + l is stored at K position
// 2l + b (the activation operand and h use the same order, so the
// contraction is unchanged).  MXFP4 follows the same order (a code byte is
// the pair i, i + 16 of its block).  Codebook-2-bit weights keep the natural
// order: each 8-weight codebook row comes from a 16-way replicated copy of
// the codebook in shared memory, c*s is formed exactly in fp16 and the single
// rounding is the multiply by d.  So do the K-quant formats (the quarter
// decoders below state their arithmetic).
//
// Tensor memory (512 columns): columns 0..255 are the four A buffers of 64
// columns (K = 128 fp16), 2t and 2t+1 for team t; columns 256..383 and 384..511 are the fp32
// accumulators (gate and up, or the down kernel's two alternating
// accumulators).  Every mbarrier wait is bounded; on expiry the kernel
// records DS4G_ERR_TIMEOUT in the status word, lets every role leave its
// loop, drains its own copies and MMAs (bounded) and frees its tensor memory.
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
// The window of one weight row per K step: the 16-byte aligned bytes that
// hold its 256-weight unit (Q2_K 84 and codebook 70 bytes: 112; MXFP4 136
// and Q4_K 144 bytes: 144; Q5_K 176; Q6_K 210 bytes at an even offset: 224).
// win_bytes: the windows of all kBM rows of an item.
__host__ __device__ constexpr int win_words(int fmt)
{
    return fmt == DS4G_FMT_MXFP4 || fmt == DS4G_FMT_Q4K ? 36
         : fmt == DS4G_FMT_Q5K                          ? 44
         : fmt == DS4G_FMT_Q6K                          ? 56
                                                        : 28;
}
__host__ __device__ constexpr int win_bytes(int fmt) { return 4 * win_words(fmt) * kBM; }
constexpr int kChunkBytes = kNT * 128;    // one 64-wide K chunk of the activation tile
constexpr int kHalfBytes = 2 * kChunkBytes;   // activation half stage: K = 128
constexpr int kHalfMmas = 8;              // K = 16 MMAs per half block
constexpr int kABufs = 4;                 // A buffers of 64 columns
constexpr int kDequantWarps = 16;         // two teams of two warpgroups
constexpr int kTeamWarps = 8;             // one team fills half hh = team of every block
constexpr int kEpilogueWarps = 4;         // down kernel: dedicated epilogue warps
constexpr int kIssuers = 2;
// warps: 0 weight producer, 1 activation producer, 2-3 MMA issuers, then the
// dequantizers, then (down kernel) the epilogue warps
constexpr int kFirstIssuerWarp = 2;
constexpr int kFirstDequantWarp = kFirstIssuerWarp + kIssuers;
__host__ __device__ constexpr int tc_threads(int mode)
{
    return (kFirstDequantWarp + kDequantWarps + (mode == 1 ? kEpilogueWarps : 0)) * 32;
}
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;
constexpr int kCbCopies = 16;
constexpr int kCbRepBytes = 256 * kCbCopies * 8;

// Shared-memory rings of one kernel: kW window stages (one K step of every
// matrix's windows), kB activation half stages; the codebook copy last.
template <int MODE, int FMT>
struct Ring {
    static constexpr int NMAT = MODE == 0 ? 2 : 1;
    static constexpr int kW = MODE == 0 ? (FMT == DS4G_FMT_Q2K ? 3 : 2) : (FMT == DS4G_FMT_Q6K ? 3 : 4);
    static constexpr int kB = MODE == 1 && FMT == DS4G_FMT_Q2K ? 5 : 4;
    static constexpr uint32_t kWStageBytes = NMAT * win_bytes(FMT);
    static constexpr size_t kWOff = (size_t)kB * kHalfBytes;
    static constexpr size_t kCbOff = kWOff + (size_t)kW * kWStageBytes;
    static constexpr size_t kBytes = kCbOff + (FMT == DS4G_FMT_CB2 ? kCbRepBytes : 0);
    static_assert(kBytes + 1024 <= 225 * 1024, "shared-memory rings exceed the per-CTA limit");
};

struct TcArgs {
    int K;                      // contraction length: hidden, or I_pad
    int m_tiles;                // weight-row tiles per expert
    int H, I_pad;
    const int32_t *tiles;       // [n][4]: expert, first segment row, rows, 0
    const int32_t *n_tiles;
    const float *wseg;          // routing weight of each segment row
    const int32_t *eseg;        // activation exponent of each segment row
    __half *hp;                 // gate/up output [A][I_pad] (permuted order)
    int h_perm32;               // h in the perm32 order of a Q2_K W_down (else natural)
    float *yslot;               // down output [A][H]
    const int8_t *codebook;     // [256 x 8] int8 (codebook format)
    const int32_t *wslot;       // [E] weight slot of each expert, or null
    int n_wslots;
    int32_t *status;
    uint64_t wait_ns;
    int stall;                  // debug: the producers issue nothing (tests the bounded waits)
};

// K position of element n inside its aligned group of 32 (Q2_K operands):
// element 16b + l goes to 2l + b.
__host__ __device__ __forceinline__ int perm32(int n)
{
    return (n & ~31) | ((n & 15) << 1) | ((n >> 4) & 1);
}

// The formats whose dequantized pairs follow perm32 (Q2_K, MXFP4); the
// codebook keeps the natural order.
__host__ __device__ constexpr bool perm32_format(int fmt)
{
    return fmt == DS4G_FMT_Q2K || fmt == DS4G_FMT_MXFP4;
}

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

// Per-warp constants of the dequantizing role: this warp's quarter of every
// block is half HH, field pair GH (Q2_K) / 64-weight half GH (codebook),
// columns 32 * GH .. +31 of the half's A buffer.
struct QuarterConst {
    int hh, gh;
    uint32_t mask[2];           // Q2_K: 2-bit field masks of g = 2*gh, 2*gh+1 (both lanes)
    uint32_t p4[2], c4[2];      // Q2_K: 4^-g and -1024 * 4^-g, replicated fp16
};

__device__ __forceinline__ QuarterConst quarter_const(int hh, int gh)
{
    QuarterConst q;
    q.hh = hh;
    q.gh = gh;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        const int g = 2 * gh + gi;
        q.mask[gi] = 0x00030003u << (2 * g);
        // fp16 4^-g: exponent 15 - 2g; -1024 * 4^-g: sign, exponent 25 - 2g
        q.p4[gi] = 0x3C003C00u - (uint32_t)g * 0x08000800u;
        q.c4[gi] = 0xE400E400u - (uint32_t)g * 0x08000800u;
    }
    return q;
}

// One quarter of a fill for this thread's row of a Q2_K block: the field
// pair g = 2*gh, 2*gh+1 of half hh, 64 weights as 32 fp16 pairs.  `qw`: the
// three 16-byte units of the window from word 4 + 8*hh (the half's qs bytes
// start SH words into it); `sw`: the scale word of sub-blocks 8*hh + 4*gh
// .. +3; `dd`: the d | dmin word.
//
// Pair (l, l+16) of field g (l = 0..15) holds weights 32g + l and 32g + l + 16
// of the half: sub-blocks 2g and 2g+1, so each lane of the half2 has its own
// sub-block scale.  Per weight, with exact fp16 operands throughout:
//   v  = 1024 + q*4^g           lop3 of the 2-bit field in place (no shift)
//   n  = v*S + C = q*sc         S = sc*4^-g, C = -1024*S; exact (integer <= 45)
//   w1 = fp16(n*d + c_hi)       one rounding, relative to w itself
//   w  = fp16(w1 + c_lo)        c_hi + c_lo = -dmin*m exactly (c_lo from an fma)
// Rounding d*sc or dmin*m to fp16 before the subtraction instead would be
// amplified by the cancellation between the two terms of a Q2_K weight.
// out[16*gi + l] = the pair of field 2*gh + gi (column 16g + l of the half).
template <int SH>
__device__ __forceinline__ void q2k_quarter(const uint32_t (&qw)[12], uint32_t sw, uint32_t dd,
                                            const QuarterConst &k, uint32_t (&out)[32])
{
    const uint32_t d2 = __byte_perm(dd, 0, 0x1010);                    // (d, d)
    const uint32_t ndmin2 = __byte_perm(dd, 0, 0x3232) ^ 0x80008000u;  // (-dmin, -dmin)
    const uint32_t k1024 = 0x64006400u, kn1024 = 0xE400E400u;
    uint32_t S2[2], C2[2], HI2[2], LO2[2];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        // scale bytes 2gi and 2gi+1 of the word (sub-blocks 2g, 2g+1) -> the two halves
        const uint32_t rep = __byte_perm(sw, 0, gi == 0 ? 0x4140u : 0x4342u);
        const uint32_t sc2 = ptx::lop3_and_or(rep, 0x000F000Fu, k1024);       // 1024 + sc
        const uint32_t mn2 = ptx::lop3_and_or(rep >> 4, 0x000F000Fu, k1024);  // 1024 + m
        S2[gi] = ptx::hfma2_u(sc2, k.p4[gi], k.c4[gi]);                      // sc * 4^-g
        C2[gi] = ptx::hmul2_u(S2[gi], kn1024);
        const uint32_t mnf = ptx::hsub2_u(mn2, k1024);                      // m
        HI2[gi] = ptx::hmul2_u(mnf, ndmin2);
        LO2[gi] = ptx::hfma2_u(mnf, ndmin2, HI2[gi] ^ 0x80008000u);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t A = qw[SH + i];                      // qs bytes 4i .. 4i+3 of the half
        const uint32_t B = qw[SH + 4 + i];                  // qs bytes 16+4i .. 16+4i+3
        const uint32_t W1 = __byte_perm(A, B, 0x5410);      // A0 A1 B0 B1
        const uint32_t W2 = __byte_perm(A, B, 0x7632);      // A2 A3 B2 B3
        const uint32_t Wu[4] = {W1, W1 >> 8, W2, W2 >> 8};  // pairs (4i+u, 4i+u+16)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int gi = 0; gi < 2; ++gi) {
                const uint32_t v = ptx::lop3_and_or(Wu[u], k.mask[gi], k1024);
                const uint32_t n = ptx::hfma2_u(v, S2[gi], C2[gi]);
                out[16 * gi + 4 * i + u] = ptx::hadd2_u(ptx::hfma2_u(n, d2, HI2[gi]), LO2[gi]);
            }
        }
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
// One quarter of a fill: weights 128*hh + 64*gh .. +63 of the block (groups
// of 8 o = 16hh + 8gh .. +7, 32-weight scale groups 4hh + 2gh, +1).  `iw`,
// `gw`: the window words holding idx / sgn bytes of those groups (three each,
// for the funnel shift), `tw`: the words holding sc and d; `fs`: the block's
// bit offset inside its first word.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cb2_quarter(const uint32_t (&iw)[3], const uint32_t (&gw)[3],
                                            const uint32_t (&tw)[3], uint32_t fs, int hh, int gh,
                                            uint32_t cb_lane, uint32_t (&out)[32])
{
    const uint32_t d2 = __byte_perm(__funnelshift_r(tw[1], tw[2], fs), 0, 0x1010);
    const uint32_t scw = __funnelshift_r(tw[0], tw[1], fs);
    uint32_t s2[2], ns2[2];
#pragma unroll
    for (int Gi = 0; Gi < 2; ++Gi) {
        const int G = 4 * hh + 2 * gh + Gi;
        const float sf = (float)((scw >> (4 * G)) & 15u);
        s2[Gi] = ptx::pack_half2(sf, sf);
        ns2[Gi] = ptx::pack_half2(-1152.0f * sf, -1152.0f * sf);
    }
    const uint32_t idxw[2] = {__funnelshift_r(iw[0], iw[1], fs), __funnelshift_r(iw[1], iw[2], fs)};
    const uint32_t sgnw[2] = {__funnelshift_r(gw[0], gw[1], fs), __funnelshift_r(gw[1], gw[2], fs)};
#pragma unroll
    for (int oi = 0; oi < 8; ++oi) {
        const uint32_t idx = (idxw[oi >> 2] >> (8 * (oi & 3))) & 0xFFu;
        const uint32_t sg = (sgnw[oi >> 2] >> (8 * (oi & 3))) & 0xFFu;
        const int Gi = oi >> 2;
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
            out[4 * oi + 2 * q] = ptx::hmul2_u(ptx::hfma2_u(v0, s2[Gi], ns2[Gi]) ^ m0, d2);
            out[4 * oi + 2 * q + 1] = ptx::hmul2_u(ptx::hfma2_u(v1, s2[Gi], ns2[Gi]) ^ m1, d2);
        }
    }
}

// Shared state of one CTA of tc_kernel (barriers, tensor memory, abort flag).
struct TcCta {
    uint8_t *wring;             // window stages
    uint64_t *wfull, *wempty, *afull, *aempty, *accfull, *accempty;
    uint32_t tmem;
    uint32_t cbrep;             // shared address of the replicated codebook
    volatile int *abort_flag;
    int n_items, KB;
};

// One thread's quarter of a block from its row window `win` of K step kb:
// half hh, field pair k.gh (Q2_K; the block's offset inside the 16-byte
// aligned window repeats every 4 K steps and is dispatched once per fill to
// a body where it is a compile-time constant, so all warps share the same
// few bodies) or weights 64*gh .. +63 of the half (codebook, `cb_lane` =
// this lane's copy of the replicated codebook).
template <int SH>
__device__ __forceinline__ void q2k_window_quarter(const uint8_t *win, int hh, const QuarterConst &k,
                                                   uint32_t (&out)[32])
{
    // 16-byte units 1 + 2hh .. 3 + 2hh hold the half's qs words (from word SH)
    uint32_t qw[12];
    const uint4 *u = reinterpret_cast<const uint4 *>(win) + 1 + 2 * hh;
#pragma unroll
    for (int v = 0; v < 3; ++v) {
        const uint4 q = u[v];
        qw[4 * v] = q.x;
        qw[4 * v + 1] = q.y;
        qw[4 * v + 2] = q.z;
        qw[4 * v + 3] = q.w;
    }
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(win);
    const uint32_t sw = w32[SH + 2 * hh + k.gh];
    const uint32_t dd = w32[SH + 20];
    q2k_quarter<SH>(qw, sw, dd, k, out);
}

__device__ __forceinline__ void cb2_window_quarter(const uint8_t *win, int boff, int hh, int gh,
                                                   uint32_t cb_lane, uint32_t (&out)[32])
{
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(win) + (boff >> 2);
    const int o = 4 * hh + 2 * gh;
    uint32_t iw[3], gw[3], tw[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        iw[j] = w32[o + j];
        gw[j] = w32[8 + o + j];
        tw[j] = w32[16 + j];
    }
    cb2_quarter(iw, gw, tw, (uint32_t)(boff & 3) * 8, hh, gh, cb_lane, out);
}

// ---------------------------------------------------------------------------
// MXFP4 units (eight 17-byte blocks of 32 weights: an E8M0 scale byte e, then
// 16 bytes of E2M1 codes, weight i in the low nibble of byte 1 + i and weight
// i + 16 in the high one; w = 2^(e-127) * value).  One quarter of a fill:
// blocks b0 = 4hh + 2gh and b0 + 1, weights 64gh .. +63 of half hh.  A code
// byte is the weight pair (i, i + 16) of its block, stored at K positions
// 2i, 2i + 1 of the block's 32: the perm32 order of the Q2_K operands, which
// the activations and h follow.  cvt.rn.f16x2.e2m1x2 gives both values
// exactly in fp16; the multiply by the block scale, an fp16 power of two, is
// exact while e - 127 lies in [-23, 13] (every product then stays between
// 2^-24 and 49152).  `boff`: the unit's byte offset in its 16-byte aligned
// window (0 or 8).  Returns false when a scale outside that range (other than
// e = 255, NaN, which propagates as the definition says) met a nonzero code,
// so that a weight came out inexact (all-zero blocks, such as the zero-filled
// rows past `inter`, stay exact whatever their scale byte).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t mx_scale2(uint32_t e, bool &in_range)
{
    const int s = (int)e - 127;
    const uint32_t bits = e == 255 ? 0x7E00u
                        : s > 15   ? 0x7C00u
                        : s >= -14 ? (uint32_t)(s + 15) << 10
                        : s >= -24 ? 1u << (s + 24)
                                   : 0u;
    in_range = e == 255 || (s >= -23 && s <= 13);
    return bits | (bits << 16);
}

__device__ __forceinline__ bool mx_window_quarter(const uint8_t *win, int boff, int hh, int gh,
                                                  uint32_t (&out)[32])
{
    // scale byte of block b0: an even offset (17 * b0 and boff are even), so
    // the 34 bytes of the two blocks lie in nine aligned words, the last of
    // them inside the 144-byte window
    const int a0 = boff + 17 * (4 * hh + 2 * gh);
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(win) + (a0 >> 2);
    const uint32_t sh = (uint32_t)(a0 & 3) * 8;             // 0 or 16
    uint32_t W[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) W[i] = w32[i];
    bool exact = true;
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
        bool in_range;
        const uint32_t s2 = mx_scale2(bi == 0 ? (W[0] >> sh) & 0xFFu : (W[4] >> (sh + 8)) & 0xFFu,
                                      in_range);
        // code bytes 4j .. 4j+3 of block b0 + bi (stream bytes 1 + 4j and 18 + 4j)
        uint32_t cw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            cw[j] = bi == 0 ? __funnelshift_r(W[j], W[j + 1], sh + 8)
                            : __funnelshift_rc(W[4 + j], W[5 + j], sh + 16);
        if (!in_range && ((cw[0] | cw[1] | cw[2] | cw[3]) & 0x77777777u) != 0) exact = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t h[4];
            ptx::e2m1x8_to_half2(cw[j], h);
#pragma unroll
            for (int u = 0; u < 4; ++u) out[16 * bi + 4 * j + u] = ptx::hmul2_u(h[u], s2);
        }
    }
    return exact;
}

// ---------------------------------------------------------------------------
// Q4_K / Q5_K super-blocks (144 / 176 bytes: d, dmin, 12 bytes of packed
// 6-bit scales and mins of eight 32-weight sub-blocks, Q5_K's qh[32] of
// fifth bits, qs[128] of nibbles; weight 64c + l / 64c + 32 + l in the low /
// high nibble of qs[32c + l], the fifth bit of weight 32s + l bit s of
// qh[l]).  Both sizes are multiples of 16, so a block starts its window.
// One quarter: chunk c = 2hh + gh, weights 64c .. +63 in natural order;
// pairs 0..15 come from the low nibbles of qs[32c + 2j], qs[32c + 2j + 1]
// (sub-block 2c), pairs 16..31 from their high nibbles (sub-block 2c + 1),
// read in place.  Per pair, with exact fp16 operands:
//   v = 1024 + q  (low nibble)  or  1024 + 16 q  (high nibble, fifth bit at 256)
//   n = v * S + C = q * sc         S = sc or sc / 16, C = -1024 * S; exact (<= 1953)
//   w = fp16(fp16(n * d + HI) + LO)   HI + LO = -dmin * m exactly (as Q2_K)
// ---------------------------------------------------------------------------
struct SubConst {
    uint32_t S2, C2, HI2, LO2;
};

__device__ __forceinline__ SubConst k45_sub_const(int sc, int m, float inv, uint32_t ndmin2)
{
    SubConst k;
    const float s = (float)sc * inv;
    k.S2 = ptx::pack_half2(s, s);
    k.C2 = ptx::pack_half2(-1024.0f * s, -1024.0f * s);
    const uint32_t m2 = ptx::pack_half2((float)m, (float)m);
    k.HI2 = ptx::hmul2_u(m2, ndmin2);
    k.LO2 = ptx::hfma2_u(m2, ndmin2, k.HI2 ^ 0x80008000u);
    return k;
}

__device__ __forceinline__ uint32_t k45_weight(uint32_t v, const SubConst &k, uint32_t d2)
{
    return ptx::hadd2_u(ptx::hfma2_u(ptx::hfma2_u(v, k.S2, k.C2), d2, k.HI2), k.LO2);
}

template <int Q5>
__device__ __forceinline__ void k45_window_quarter(const uint8_t *win, int hh, int gh,
                                                   uint32_t (&out)[32])
{
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(win);
    const int c = 2 * hh + gh;
    const uint32_t dd = w32[0];
    const uint32_t d2 = __byte_perm(dd, 0, 0x1010);
    const uint32_t ndmin2 = __byte_perm(dd, 0, 0x3232) ^ 0x80008000u;
    // scale bytes q[0..11] in w32[1..3]; sub-block s = 2c + t.  s < 4 (hh 0):
    // sc = q[s] & 63, m = q[s+4] & 63; s >= 4 (hh 1): sc = (q[s+4] & 15) |
    // (q[s-4] >> 6) << 4, m = (q[s+4] >> 4) | (q[s] >> 6) << 4.  Either way the
    // three bytes sit at position 2gh + t of words 1, 2, 3.
    SubConst k[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int sh = 8 * (2 * gh + t);
        const int b0 = (w32[1] >> sh) & 0xFF, b1 = (w32[2] >> sh) & 0xFF, b2 = (w32[3] >> sh) & 0xFF;
        const int sc = hh ? (b2 & 15) | ((b0 >> 6) << 4) : b0 & 63;
        const int m = hh ? (b2 >> 4) | ((b1 >> 6) << 4) : b1 & 63;
        k[t] = k45_sub_const(sc, m, t ? 0.0625f : 1.0f, ndmin2);
    }
    const uint32_t k1024 = 0x64006400u;
    const int qs0 = (Q5 ? 48 : 16) / 4 + 8 * c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t W = w32[qs0 + i];                   // qs bytes 32c + 4i .. +3
        const uint32_t x[2] = {__byte_perm(W, 0, 0x4140), __byte_perm(W, 0, 0x4342)};
        uint32_t y[2] = {0, 0};
        if (Q5) {
            const uint32_t Y = w32[4 + i];                 // qh bytes 4i .. 4i+3
            y[0] = __byte_perm(Y, 0, 0x4140);
            y[1] = __byte_perm(Y, 0, 0x4342);
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint32_t vlo = ptx::lop3_and_or(x[p], 0x000F000Fu, k1024);
            uint32_t vhi = ptx::lop3_and_or(x[p], 0x00F000F0u, k1024);
            if (Q5) {
                // bit 2c (value 16) and bit 2c + 1 (value 256, high nibble in place)
                vlo = ptx::lop3_and_or((y[p] << 4) >> (2 * c), 0x00100010u, vlo);
                vhi = ptx::lop3_and_or((y[p] << 8) >> (2 * c + 1), 0x01000100u, vhi);
            }
            out[2 * i + p] = k45_weight(vlo, k[0], d2);
            out[16 + 2 * i + p] = k45_weight(vhi, k[1], d2);
        }
    }
}

// ---------------------------------------------------------------------------
// Q6_K super-blocks (210 bytes: ql[128], qh[64], int8 scales[16], d; weight
// j = 128h + 32u + l has its low nibble in nibble u >> 1 of ql[64h + 32(u&1)
// + l], its top two bits in bits 2u, 2u + 1 of qh[32h + l];
// w = d * scales[j / 16] * (q - 32)).  A block sits at an even offset `boff`
// of its 224-byte window.  One quarter: half hh, weights 64gh .. +63 of it in
// natural order: pairs 0..15 (u = 2gh) from nibble gh of ql[64hh + 2j, +1]
// and bits 4gh, 4gh+1 of qh[32hh + 2j, +1]; pairs 16..31 (u = 2gh + 1) from
// ql[64hh + 32 + ..] and bits 4gh+2, 4gh+3.  Per pair:
//   v = 1024 + q exactly;  v - 1056 = q - 32 exactly;
//   w = fp16((q - 32) * fp16(d * sc))   two roundings, each relative to w.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q6k_window_quarter(const uint8_t *win, int boff, int hh, int gh,
                                                   uint32_t (&out)[32])
{
    const uint32_t *w32 = reinterpret_cast<const uint32_t *>(win) + (boff >> 2);
    const uint32_t fs = (uint32_t)(boff & 3) * 8;          // 0 or 16
    // d (bytes 208, 209) and the four scales of the quarter (bytes 192 + 8hh + 4gh ..)
    // d lies inside one aligned word (boff is even); no word past the window is read
    const float d = __half2float(__ushort_as_half((unsigned short)((w32[52] >> fs) & 0xFFFFu)));
    const int so = 48 + 2 * hh + gh;                       // word of the scale bytes
    const uint32_t sw = __funnelshift_r(w32[so], w32[so + 1], fs);
    uint32_t SD2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float sd = d * (float)(int8_t)((sw >> (8 * q)) & 0xFF);
        SD2[q] = ptx::pack_half2(sd, sd);
    }
    // qh bytes 32hh .. +31 (word 32 + 8hh on): the bits of both parts
    uint32_t QH[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) QH[i] = __funnelshift_r(w32[32 + 8 * hh + i], w32[33 + 8 * hh + i], fs);
    const uint32_t k1024 = 0x64006400u, k1056 = 0x64206420u;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        const int qw = 16 * hh + 8 * part;                 // word of ql[64hh + 32 part]
        const int hs = 4 * gh + 2 * part;                  // qh bit pair
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t L = __funnelshift_r(w32[qw + i], w32[qw + i + 1], fs) >> (4 * gh);
            const uint32_t x[2] = {__byte_perm(L, 0, 0x4140), __byte_perm(L, 0, 0x4342)};
            const uint32_t y[2] = {__byte_perm(QH[i], 0, 0x4140), __byte_perm(QH[i], 0, 0x4342)};
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t v = ptx::lop3_and_or(x[p], 0x000F000Fu, k1024);
                v = ptx::lop3_and_or((y[p] >> hs) << 4, 0x00300030u, v);
                const int j = 16 * part + 2 * i + p;       // pair index of the quarter
                out[j] = ptx::hmul2_u(ptx::hsub2_u(v, k1056), SD2[j >> 3]);
            }
        }
    }
}

// One quarter's 32 fp16 pairs of any tensor-core format; false when an MXFP4
// block scale made a weight inexact in fp16.
template <int FMT>
__device__ __forceinline__ bool quarter_values(const uint8_t *win, int kb, int hh,
                                               const QuarterConst &k, uint32_t cb_lane,
                                               uint32_t (&out)[32])
{
    if (FMT == DS4G_FMT_MXFP4) return mx_window_quarter(win, (kMXFP4Bytes * kb) & 15, hh, k.gh, out);
    if (FMT == DS4G_FMT_Q4K || FMT == DS4G_FMT_Q5K) {
        k45_window_quarter<FMT == DS4G_FMT_Q5K>(win, hh, k.gh, out);
        return true;
    }
    if (FMT == DS4G_FMT_Q6K) {
        q6k_window_quarter(win, (kQ6KBytes * kb) & 15, hh, k.gh, out);
        return true;
    }
    if (FMT == DS4G_FMT_Q2K) {
        switch (kb & 3) {           // (84 * kb) mod 16, in words
        case 0: q2k_window_quarter<0>(win, hh, k, out); break;
        case 1: q2k_window_quarter<1>(win, hh, k, out); break;
        case 2: q2k_window_quarter<2>(win, hh, k, out); break;
        default: q2k_window_quarter<3>(win, hh, k, out); break;
        }
    } else {
        cb2_window_quarter(win, (kCB2Bytes * kb) & 15, hh, k.gh, cb_lane, out);
    }
    return true;
}

// The dequantizing role of one warp (both kernels of tc_kernel).  Two teams
// of two warpgroups, each with its own two A buffers (2*team, 2*team + 1 for
// halves 0 and 1).  Gate/up: team t dequantizes matrix t (W_gate, W_up) of
// every K step, and issuer t issues its fills alone, so each matrix is a
// private pipeline of dequantizers and issuer.  Down (Q2_K): team t owns the
// K steps of parity t, so while the issuer runs one team's K step the other
// team already dequantizes its next one.
template <int MODE, int FMT>
struct DequantRole {
    using R = Ring<MODE, FMT>;

    const TcArgs &a;
    const TcCta &c;
    QuarterConst k;
    int lane, row, wg;
    uint32_t lane_base;
    int kc = 0;                 // K steps done
    bool ok = true;

    __device__ __forceinline__ DequantRole(const TcArgs &a_, const TcCta &c_, int warp, int lane_,
                                           int wg_)
        : a(a_), c(c_), lane(lane_), wg(wg_)
    {
        k = quarter_const(wg >> 1, wg & 1);
        const int quarter = warp & 3;             // tensor-memory lane quarter
        row = 32 * quarter + lane;
        lane_base = (uint32_t)(32 * quarter) << 16;
    }

    // One fill: half hh of matrix `mat`, K step kb, window stage ws, into this
    // team's buffer 2*team + hh (team = k.hh).
    __device__ __forceinline__ void fill(int ws, int mat, int kb, int hh)
    {
        const int buf = 2 * k.hh + hh;
        const int uses = MODE == 0 ? kc : (kc >> 1);      // earlier fills of the buffer
        if (uses > 0) {
            ok = wait_bar(&c.aempty[buf], (uses - 1) & 1, a.wait_ns, c.abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) return;
            ptx::tc_fence_after();
        }
        const uint8_t *win = c.wring + (size_t)ws * R::kWStageBytes + mat * win_bytes(FMT) +
                             row * (4 * win_words(FMT));
        uint32_t out[32];
        if (!quarter_values<FMT>(win, kb, hh, k, c.cbrep + (uint32_t)(lane & 15) * 8, out))
            set_status(a.status, DS4G_ERR_RANGE);
        ptx::tmem_st32(c.tmem + lane_base + (uint32_t)buf * 64u + 32u * k.gh, out);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&c.afull[buf]);
    }

    __device__ __forceinline__ void run()
    {
        int ic = 0;
        for (int it = blockIdx.x; ok && it < c.n_items; it += gridDim.x, ++ic) {
            const int tile = it / a.m_tiles, mt = it % a.m_tiles;
            const int row0 = a.tiles[4 * tile + 1], nlen = a.tiles[4 * tile + 2];
            for (int kb = 0; ok && kb < c.KB; ++kb, ++kc) {
                if (MODE == 1 && (kc & 1) != k.hh) continue;     // the other team's K step
                const int ws = kc % R::kW;
                ok = wait_bar(&c.wfull[ws], (kc / R::kW) & 1, a.wait_ns, c.abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // gate/up: team = matrix; down: the stage's only matrix
                for (int hh = 0; ok && hh < 2; ++hh) fill(ws, MODE == 0 ? k.hh : 0, kb, hh);
                if (!ok) break;
                // this warp has read the stage's windows
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&c.wempty[ws]);
            }
            if (!ok) break;
            if (MODE == 1) continue;                 // the epilogue warps finish down items
            // gate/up epilogue of the item: chunks of 8 tokens, warpgroup w
            // takes chunks w, w + 4, ...; accumulator 0 = gate, 1 = up
            ok = wait_bar(&c.accfull[0], ic & 1, a.wait_ns, c.abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int chunks = (nlen + 7) / 8;
            const int n = mt * kBM + row;
            // h is laid out for the down kernel's format
            const int col = a.h_perm32 ? perm32(n) : n;
            for (int ch = wg; ch < chunks; ch += 4) {
                float g[8], u[8];
                ptx::tmem_ld8(c.tmem + lane_base + kAccCol + 8 * ch, g);
                ptx::tmem_ld8(c.tmem + lane_base + kAccCol + 128 + 8 * ch, u);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = 8 * ch + j;
                    if (t < nlen) {
                        // undo the row's activation scale, store h scaled by 2^-f
                        const int e = __ldg(a.eseg + row0 + t);
                        const float sx = exp2i(e);
                        const float h = silu_mul(g[j] * sx, u[j] * sx);
                        a.hp[(size_t)(row0 + t) * a.I_pad + col] =
                            __float2half_rn(h * exp2i(-(2 * e + kHExpOffset)));
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&c.accempty[0]);
        }
        if (!ok) {
            if (lane == 0) set_status(a.status, DS4G_ERR_TIMEOUT);
            *c.abort_flag = 1;
        }
    }
};

// Weight-window prefetch distance of the weight producer, in K steps.
constexpr int kPrefetchSteps = 6;

// After an abort: wait (bounded) for the copies still in flight on a ring
// whose `issued` stages were armed in order.
__device__ __forceinline__ void drain_ring(uint64_t *full, int ring, int issued, uint64_t wait_ns)
{
    for (int q = issued - ring; q < issued; ++q) {
        if (q < 0) continue;
        if (!ptx::mbar_wait(&full[q % ring], (q / ring) & 1, wait_ns)) break;
    }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(tc_threads(MODE), 1)
    tc_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
              const __grid_constant__ CUtensorMap tm_b, const TcArgs a)
{
    using R = Ring<MODE, FMT>;
    constexpr int NMAT = R::NMAT;
    constexpr int kBlockBytes = block_bytes_of(FMT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *bring = smem;                      // activation half stages (1024-aligned)
    uint8_t *wring = smem + R::kWOff;           // window stages
    uint8_t *cbrep = smem + R::kCbOff;          // codebook format only
    __shared__ __align__(8) uint64_t wfull[R::kW], wempty[R::kW], bfull[R::kB], bempty[R::kB];
    __shared__ __align__(8) uint64_t afull[kABufs], aempty[kABufs];
    __shared__ __align__(8) uint64_t accfull[2], accempty[2], drain[kIssuers];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_wissued, s_bissued;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < R::kW; ++s) {
            ptx::mbar_init(&wfull[s], 1);
            // gate/up: every dequantizing warp reads every stage; down: one team
            ptx::mbar_init(&wempty[s], MODE == 0 ? kDequantWarps : kTeamWarps);
        }
        for (int s = 0; s < R::kB; ++s) {
            ptx::mbar_init(&bfull[s], 1);
            ptx::mbar_init(&bempty[s], NMAT);       // one commit per issuer
        }
        for (int b = 0; b < kABufs; ++b) {
            ptx::mbar_init(&afull[b], kTeamWarps);
            ptx::mbar_init(&aempty[b], 1);
        }
        // gate/up: one accumulator pair, both issuers commit; down: two
        // alternating accumulators, one issuer
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&accfull[b], MODE == 0 ? kIssuers : 1);
            ptx::mbar_init(&accempty[b], MODE == 0 ? kDequantWarps : kEpilogueWarps);
        }
        for (int i = 0; i < kIssuers; ++i) ptx::mbar_init(&drain[i], 1);
        ptx::fence_mbar_init();
        s_abort = 0;
        s_wissued = 0;
        s_bissued = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(&s_tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
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
        // ---------------- weight producer ----------------
        // The windows of the K step kPrefetchSteps ahead are also prefetched
        // into L2, so the ring's copies of them hit L2.
        if (lane == 0 && !a.stall) {
            ptx::prefetch_tmap(&tm_a0);
            if (NMAT == 2) ptx::prefetch_tmap(&tm_a1);
            int pf_it = blockIdx.x, pf_kb = 0;       // the prefetch cursor
            auto prefetch_next = [&]() {
                if (pf_it >= n_items) return;
                const int tile = pf_it / a.m_tiles, mt = pf_it % a.m_tiles;
                const int e = weight_slot(a.wslot, a.n_wslots, a.tiles[4 * tile], a.status);
                const int x = ((kBlockBytes * pf_kb) & ~15) / 4;
                ptx::tma_prefetch_3d(&tm_a0, x, mt * kBM, e);
                if (NMAT == 2) ptx::tma_prefetch_3d(&tm_a1, x, mt * kBM, e);
                if (++pf_kb == KB) {
                    pf_kb = 0;
                    pf_it += gridDim.x;
                }
            };
            for (int i = 0; i < kPrefetchSteps; ++i) prefetch_next();
            int wc = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int tile = it / a.m_tiles, mt = it % a.m_tiles;
                const int e = weight_slot(a.wslot, a.n_wslots, a.tiles[4 * tile], a.status);
                for (int kb = 0; kb < KB; ++kb, ++wc) {
                    const int s = wc % R::kW;
                    if (wc >= R::kW &&
                        !wait_bar(&wempty[s], ((wc / R::kW) - 1) & 1, a.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = wring + (size_t)s * R::kWStageBytes;
                    ptx::mbar_arrive_expect_tx(&wfull[s], R::kWStageBytes);
                    const int x = ((kBlockBytes * kb) & ~15) / 4;
                    ptx::tma_load_3d(st, &tm_a0, x, mt * kBM, e, &wfull[s]);
                    if (NMAT == 2) ptx::tma_load_3d(st + win_bytes(FMT), &tm_a1, x, mt * kBM, e, &wfull[s]);
                    prefetch_next();
                }
            }
            if (!ok) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            s_wissued = wc;
        }
    } else if (warp == 1) {
        // ---------------- activation producer ----------------
        if (lane == 0 && !a.stall) {
            ptx::prefetch_tmap(&tm_b);
            int bc = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const int tile = it / a.m_tiles;
                const int row0 = a.tiles[4 * tile + 1];
                const int nb = (a.tiles[4 * tile + 2] + kBoxRows - 1) / kBoxRows;
                const uint32_t bytes = 2u * nb * kBoxRows * 128u;
                for (int hs = 0; ok && hs < 2 * KB; ++hs, ++bc) {
                    const int s = bc % R::kB;
                    if (bc >= R::kB &&
                        !wait_bar(&bempty[s], ((bc / R::kB) - 1) & 1, a.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = bring + (size_t)s * kHalfBytes;
                    ptx::mbar_arrive_expect_tx(&bfull[s], bytes);
                    for (int kc = 0; kc < 2; ++kc)
                        for (int r = 0; r < nb; ++r)
                            ptx::tma_load_2d(st + kc * kChunkBytes + r * kBoxRows * 128, &tm_b,
                                             hs * 128 + 64 * kc, row0 + kBoxRows * r, &bfull[s]);
                }
            }
            if (!ok) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            s_bissued = bc;
        }
    } else if (warp < kFirstDequantWarp) {
        // ---------------- MMA issuers ----------------
        // Gate/up kernel: issuer X issues team X's fills (W_gate for X = 0,
        // W_up for X = 1), A buffers 2X and 2X + 1 (halves 0 and 1), into
        // accumulator X.
        // One thread issues tcgen05.mma far slower than the tensor pipe runs
        // them at a segment's token counts; two issuers keep it fed.  Down
        // kernel (one fill per half step, bound by its dequantizers): issuer
        // 0 alone, every A buffer in turn, with two accumulators that
        // alternate per item, so the epilogue warps drain one while the next
        // item accumulates.  The whole warp runs the loop, converged; one lane chosen by
        // elect.sync issues.
        const int X = warp - kFirstIssuerWarp;
        if (MODE == 1 && X == 1) {
            // no second issuer in the down kernel
        } else {
            const uint64_t bdesc0 = ptx::sw128_desc(ptx::smem_addr(bring));
            int hc = 0, ic = 0;                      // half steps, items
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++ic) {
                const int tile = it / a.m_tiles;
                const int nb = (a.tiles[4 * tile + 2] + kBoxRows - 1) / kBoxRows;
                const uint32_t idesc = ptx::idesc_f16(kBM, nb * kBoxRows);
                const int ab = MODE == 1 ? (ic & 1) : 0;
                const int uses = MODE == 1 ? (ic >> 1) : ic;
                if (uses > 0) {
                    ok = wait_bar(&accempty[ab], (uses - 1) & 1, a.wait_ns, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                ptx::tc_fence_after();
                const uint32_t acc = tmem + kAccCol + 128u * (uint32_t)(MODE == 1 ? ab : X);
                for (int hs = 0; ok && hs < 2 * KB; ++hs, ++hc) {
                    const int s = hc % R::kB;
                    // the fill's A buffer (half hh of K step kc) and how often
                    // it was filled before
                    const int kc = hc >> 1, hh = hc & 1;
                    const int buf = MODE == 0 ? 2 * X + hh : 2 * (kc & 1) + hh;
                    const int uses = MODE == 0 ? kc : (kc >> 1);
                    ok = wait_bar(&bfull[s], (hc / R::kB) & 1, a.wait_ns, abort_flag);
                    ok = ok && wait_bar(&afull[buf], uses & 1, a.wait_ns, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint64_t bd0 = bdesc0 + (uint64_t)((s * kHalfBytes) >> 4);
                    const uint32_t a_buf = tmem + (uint32_t)buf * 64u;
#pragma unroll
                    for (int i = 0; i < kHalfMmas; ++i) {
                        const int kk = 16 * i;
                        const uint64_t bd =
                            bd0 + (uint64_t)(((kk >> 6) * kChunkBytes + (kk & 63) * 2) >> 4);
                        ptx::mma_f16_ts_elect(acc, a_buf + 8 * i, bd, idesc, hs > 0 || i > 0);
                    }
                    ptx::mma_commit_elect(&aempty[buf]);
                    ptx::mma_commit_elect(&bempty[s]);
                    __syncwarp();
                }
                if (!ok) break;
                ptx::mma_commit_elect(&accfull[ab]);
                __syncwarp();
            }
            if (!ok && lane == 0) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread is complete before the CTA frees
            // its tensor memory
            ptx::mma_commit_elect(&drain[X]);
            ptx::mbar_wait(&drain[X], 0, a.wait_ns);
            __syncwarp();
        }
    } else if (warp >= kFirstDequantWarp + kDequantWarps) {
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
                        const float sh = exp2i(2 * __ldg(a.eseg + pos) + kHExpOffset);
                        a.yslot[(size_t)pos * a.H + m] = __ldg(a.wseg + pos) * (o[j] * sh);
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
        const TcCta cta{wring, wfull, wempty, afull, aempty, accfull, accempty, tmem,
                        ptx::smem_addr(cbrep), abort_flag, n_items, KB};
        DequantRole<MODE, FMT>(a, cta, warp, lane, (warp - kFirstDequantWarp) >> 2).run();
    }

    __syncthreads();
    // after an abort: the copies this CTA issued land before it exits
    if (threadIdx.x == 0 && *abort_flag) {
        drain_ring(wfull, R::kW, s_wissued, a.wait_ns);
        drain_ring(bfull, R::kB, s_bissued, a.wait_ns);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// The down kernel of codebook W_down: one item per dequantizing team.  yslot = w * (W_down . h)
// needs one accumulator per item, so each team takes every other item of the
// CTA with its own producer, window and activation rings, MMA issuer, two A
// buffers (half 0 and half 1 of each K step) and accumulator; the teams never
// wait for each other, and the four epilogue warps drain both accumulators
// in the CTA's item order.  Two teams' rings leave each team two activation
// half stages: enough behind the codebook dequant, too few behind the faster
// Q2_K one, whose down kernel keeps the shared issuer of tc_kernel<1, Q2_K>
// (measured 1.06 against 1.15 ms for codebook_512's down phase, 1.25 against
// 1.17 ms for prefill_2048's).
//   warps 0, 1    producer of team 0, 1: per K step of the team's item the
//                 window stage, then the two activation half stages (h tile)
//   warps 2, 3    MMA issuer of team 0, 1 (elected lane, converged warp)
//   warps 4-19    dequantizers: team t = warps 4 + 8t .. 11 + 8t, thread =
//                 weight row, quarter (half, field pair gh) of each fill
//   warps 20-23   epilogue: routing weight, token exponent, fp32 y_slot
// Tensor memory: A buffers 2t, 2t+1 of team t (64 columns each), accumulator
// of team t at column 256 + 128t.
// ---------------------------------------------------------------------------
template <int FMT>
struct DownRing {
    static constexpr int kW = FMT == DS4G_FMT_Q2K ? 3 : 2;     // window stages per team
    static constexpr int kB = 2;                               // activation half stages per team
    static constexpr size_t kTeamBytes = (size_t)kW * win_bytes(FMT) + (size_t)kB * kHalfBytes;
    // per team: [B half stages][window stages]; the codebook copy last
    static constexpr size_t kBOff(int t) { return (size_t)t * kTeamBytes; }
    static constexpr size_t kWOff(int t) { return (size_t)t * kTeamBytes + (size_t)kB * kHalfBytes; }
    static constexpr size_t kCbOff = 2 * kTeamBytes;
    static constexpr size_t kBytes = kCbOff + (FMT == DS4G_FMT_CB2 ? kCbRepBytes : 0);
    static_assert(kTeamBytes % 1024 == 0, "team rings keep the 1024-byte swizzle alignment");
    static_assert(kBytes + 1024 <= 225 * 1024, "shared-memory rings exceed the per-CTA limit");
};

constexpr int kDownThreads = (kFirstDequantWarp + kDequantWarps + kEpilogueWarps) * 32;

template <int FMT>
__global__ void __launch_bounds__(kDownThreads, 1)
    tc_down_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h,
                   const TcArgs a)
{
    using R = DownRing<FMT>;
    constexpr int kBlockBytes = block_bytes_of(FMT);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *cbrep = smem + R::kCbOff;
    __shared__ __align__(8) uint64_t wfull[2][R::kW], wempty[2][R::kW], bfull[2][R::kB],
        bempty[2][R::kB];
    __shared__ __align__(8) uint64_t afull[kABufs], aempty[kABufs], accfull[2], accempty[2],
        drain[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_wissued[2], s_bissued[2];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            for (int s = 0; s < R::kW; ++s) {
                ptx::mbar_init(&wfull[t][s], 1);
                ptx::mbar_init(&wempty[t][s], kTeamWarps);
            }
            for (int s = 0; s < R::kB; ++s) {
                ptx::mbar_init(&bfull[t][s], 1);
                ptx::mbar_init(&bempty[t][s], 1);
            }
            ptx::mbar_init(&accfull[t], 1);
            ptx::mbar_init(&accempty[t], kEpilogueWarps);
            ptx::mbar_init(&drain[t], 1);
            s_wissued[t] = 0;
            s_bissued[t] = 0;
        }
        for (int b = 0; b < kABufs; ++b) {
            ptx::mbar_init(&afull[b], kTeamWarps);
            ptx::mbar_init(&aempty[b], 1);
        }
        ptx::fence_mbar_init();
        s_abort = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(&s_tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
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
    // the CTA's items: it_j = blockIdx.x + j * gridDim.x; team t takes j = t, t + 2, ...
    const int my_items = n_items > (int)blockIdx.x ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto team_items = [&](int t) { return my_items > t ? (my_items - 1 - t) / 2 + 1 : 0; };
    auto item_of = [&](int t, int q) { return (int)blockIdx.x + (2 * q + t) * (int)gridDim.x; };

    if (warp < 2) {
        // ---------------- producer of team t ----------------
        const int t = warp;
        if (lane == 0 && !a.stall) {
            ptx::prefetch_tmap(&tm_w);
            ptx::prefetch_tmap(&tm_h);
            const int nk = team_items(t) * KB;           // K steps of the team
            uint8_t *bring = smem + R::kBOff(t);
            uint8_t *wring = smem + R::kWOff(t);
            int wc = 0, bc = 0;
            bool ok = true;
            // the windows of K step w (weight producer part), L2 prefetch ahead
            auto issue_w = [&](int w) -> bool {
                const int s = w % R::kW;
                if (w >= R::kW &&
                    !wait_bar(&wempty[t][s], ((w / R::kW) - 1) & 1, a.wait_ns, abort_flag))
                    return false;
                const int it = item_of(t, w / KB), kb = w % KB;
                const int tile = it / a.m_tiles, mt = it % a.m_tiles;
                const int e = weight_slot(a.wslot, a.n_wslots, a.tiles[4 * tile], a.status);
                ptx::mbar_arrive_expect_tx(&wfull[t][s], (uint32_t)win_bytes(FMT));
                ptx::tma_load_3d(wring + (size_t)s * win_bytes(FMT), &tm_w, ((kBlockBytes * kb) & ~15) / 4,
                                 mt * kBM, e, &wfull[t][s]);
                const int pw = w + kPrefetchSteps;
                if (pw < nk) {
                    const int pit = item_of(t, pw / KB), pkb = pw % KB;
                    const int pe = weight_slot(a.wslot, a.n_wslots, a.tiles[4 * (pit / a.m_tiles)], a.status);
                    ptx::tma_prefetch_3d(&tm_w, ((kBlockBytes * pkb) & ~15) / 4,
                                         (pit % a.m_tiles) * kBM, pe);
                }
                return true;
            };
            for (; ok && wc < nk && wc < R::kW - 1; ++wc) ok = issue_w(wc);
            for (int kc = 0; ok && kc < nk; ++kc) {
                const int it = item_of(t, kc / KB), kb = kc % KB;
                const int tile = it / a.m_tiles;
                const int row0 = a.tiles[4 * tile + 1];
                const int nb = (a.tiles[4 * tile + 2] + kBoxRows - 1) / kBoxRows;
                const uint32_t bytes = 2u * nb * kBoxRows * 128u;
                for (int hh = 0; ok && hh < 2; ++hh, ++bc) {
                    const int s = bc % R::kB;
                    if (bc >= R::kB &&
                        !wait_bar(&bempty[t][s], ((bc / R::kB) - 1) & 1, a.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = bring + (size_t)s * kHalfBytes;
                    ptx::mbar_arrive_expect_tx(&bfull[t][s], bytes);
                    for (int c2 = 0; c2 < 2; ++c2)
                        for (int r = 0; r < nb; ++r)
                            ptx::tma_load_2d(st + c2 * kChunkBytes + r * kBoxRows * 128, &tm_h,
                                             (2 * kb + hh) * 128 + 64 * c2, row0 + kBoxRows * r,
                                             &bfull[t][s]);
                }
                if (ok && wc < nk) ok = issue_w(wc++);
            }
            if (!ok) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            s_wissued[t] = wc;
            s_bissued[t] = bc;
        }
    } else if (warp < kFirstDequantWarp) {
        // ---------------- MMA issuer of team t ----------------
        const int t = warp - kFirstIssuerWarp;
        const uint64_t bdesc0 = ptx::sw128_desc(ptx::smem_addr(smem + R::kBOff(t)));
        const uint32_t acc = tmem + kAccCol + 128u * (uint32_t)t;
        int hc = 0;                                     // half steps (fills) of the team
        bool ok = true;
        for (int q = 0; ok && q < team_items(t); ++q) {
            const int it = item_of(t, q);
            const int nb = (a.tiles[4 * (it / a.m_tiles) + 2] + kBoxRows - 1) / kBoxRows;
            const uint32_t idesc = ptx::idesc_f16(kBM, nb * kBoxRows);
            if (q > 0) {
                ok = wait_bar(&accempty[t], (q - 1) & 1, a.wait_ns, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            ptx::tc_fence_after();
            for (int hs = 0; ok && hs < 2 * KB; ++hs, ++hc) {
                const int s = hc % R::kB;
                const int buf = 2 * t + (hc & 1);
                ok = wait_bar(&bfull[t][s], (hc / R::kB) & 1, a.wait_ns, abort_flag);
                ok = ok && wait_bar(&afull[buf], (hc >> 1) & 1, a.wait_ns, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint64_t bd0 = bdesc0 + (uint64_t)((s * kHalfBytes) >> 4);
                const uint32_t a_buf = tmem + (uint32_t)buf * 64u;
#pragma unroll
                for (int i = 0; i < kHalfMmas; ++i) {
                    const int kk = 16 * i;
                    const uint64_t bd = bd0 + (uint64_t)(((kk >> 6) * kChunkBytes + (kk & 63) * 2) >> 4);
                    ptx::mma_f16_ts_elect(acc, a_buf + 8 * i, bd, idesc, hs > 0 || i > 0);
                }
                ptx::mma_commit_elect(&aempty[buf]);
                ptx::mma_commit_elect(&bempty[t][s]);
                __syncwarp();
            }
            if (!ok) break;
            ptx::mma_commit_elect(&accfull[t]);
            __syncwarp();
        }
        if (!ok && lane == 0) {
            set_status(a.status, DS4G_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        ptx::mma_commit_elect(&drain[t]);
        ptx::mbar_wait(&drain[t], 0, a.wait_ns);
        __syncwarp();
    } else if (warp >= kFirstDequantWarp + kDequantWarps) {
        // ---------------- epilogue: both teams' items in the CTA's order ----------------
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            const int t = j & 1, q = j >> 1;
            const int it = item_of(t, q);
            const int tile = it / a.m_tiles, mt = it % a.m_tiles;
            const int row0 = a.tiles[4 * tile + 1], nlen = a.tiles[4 * tile + 2];
            ok = wait_bar(&accfull[t], q & 1, a.wait_ns, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const int m = mt * kBM + row;
            const uint32_t acc = tmem + lane_base + kAccCol + 128u * (uint32_t)t;
            for (int c = 0; 8 * c < nlen; ++c) {
                float o[8];
                ptx::tmem_ld8(acc + 8 * c, o);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int tk = 8 * c + i;
                    if (tk < nlen) {
                        const int pos = row0 + tk;
                        const float sh = exp2i(2 * __ldg(a.eseg + pos) + kHExpOffset);
                        a.yslot[(size_t)pos * a.H + m] = __ldg(a.wseg + pos) * (o[i] * sh);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&accempty[t]);
        }
        if (!ok) {
            if (lane == 0) set_status(a.status, DS4G_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ---------------- dequantizers of team t ----------------
        const int wg = (warp - kFirstDequantWarp) >> 2;
        const int t = wg >> 1, gh = wg & 1;
        const QuarterConst k = quarter_const(0, gh);
        const int row = 32 * (warp & 3) + lane;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t cb_lane = ptx::smem_addr(cbrep) + (uint32_t)(lane & 15) * 8;
        const uint8_t *wring = smem + R::kWOff(t);
        int kc = 0, tf = 0;
        bool ok = true;
        for (int q = 0; ok && q < team_items(t); ++q) {
            for (int kb = 0; ok && kb < KB; ++kb, ++kc) {
                const int ws = kc % R::kW;
                ok = wait_bar(&wfull[t][ws], (kc / R::kW) & 1, a.wait_ns, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint8_t *win = wring + (size_t)ws * win_bytes(FMT) + row * (4 * win_words(FMT));
                for (int hh = 0; ok && hh < 2; ++hh, ++tf) {
                    const int buf = 2 * t + (tf & 1);
                    if (tf >= 2) {
                        ok = wait_bar(&aempty[buf], ((tf >> 1) - 1) & 1, a.wait_ns, abort_flag);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ptx::tc_fence_after();
                    }
                    uint32_t out[32];
                    if (!quarter_values<FMT>(win, kb, hh, k, cb_lane, out))
                        set_status(a.status, DS4G_ERR_RANGE);
                    ptx::tmem_st32(tmem + lane_base + (uint32_t)buf * 64u + 32u * gh, out);
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&afull[buf]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&wempty[t][ws]);
            }
        }
        if (!ok) {
            if (lane == 0) set_status(a.status, DS4G_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    // after an abort: the copies this CTA issued land before it exits
    if (threadIdx.x == 0 && *abort_flag) {
        for (int t = 0; t < 2; ++t) {
            drain_ring(wfull[t], R::kW, s_wissued[t], a.wait_ns);
            drain_ring(bfull[t], R::kB, s_bissued[t], a.wait_ns);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Token exponents: texp[t] = e_t (see token_exponent), one warp per token.
__global__ void __launch_bounds__(256) token_exp_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                        int32_t *__restrict__ texp)
{
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
    float m = 0.0f;
    for (int i = lane; i < H / 8; i += 32) {
        const uint4 r = __ldg(row + i);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(bf16_abs_finite(w[j] & 0xFFFFu), bf16_abs_finite(w[j] >> 16)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) texp[t] = token_exponent(m);
}

// Token tiles of every active segment and the activation gather:
//   tiles[j] = (expert, first segment row, rows <= kNT, 0) for the segments
//   of at least min_tokens rows, in expert order; *n_tiles = count; the
//   shorter non-empty segments' experts in light[0 .. *n_light) (the GEMV
//   kernels take those; min_tokens 0 sends every segment to the tiles);
//   wseg[p] = wts[perm[p]];
//   eseg[p] = texp[perm[p] / k];
//   xseg[p, :] = fp16(x[perm[p] / k, :] * 2^-eseg[p]), for Q2_K with element
//   16b + l of every aligned group of 32 at position 2l + b (perm32), in
//   natural order for the codebook format.  One thread writes 16 consecutive
//   positions.
constexpr int kPrepWarps = DS4G_MAX_EXPERTS / 32;   // tc_prep_kernel: one thread per expert

__global__ void __launch_bounds__(kPrepWarps * 32) tc_prep_kernel(const uint16_t *__restrict__ x, int H, int k,
                                                      int A, const int32_t *__restrict__ perm,
                                                      const int32_t *counts,
                                                      const int32_t *offsets, int E,
                                                      __half *__restrict__ xseg, int32_t *tiles,
                                                      int32_t *n_tiles, int permute32,
                                                      const float *__restrict__ wts,
                                                      float *__restrict__ wseg,
                                                      const int32_t *__restrict__ texp,
                                                      int32_t *__restrict__ eseg, int min_tokens,
                                                      int32_t *__restrict__ light,
                                                      int32_t *__restrict__ n_light)
{
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < A; p += gridDim.x * blockDim.x) {
        wseg[p] = wts[perm[p]];
        eseg[p] = texp[perm[p] / k];
    }
    if (blockIdx.x == 0) {
        // thread e (256 threads, one per expert): its tile count, an exclusive
        // scan over the experts (warp shuffles, then the warp totals) for its
        // first tile, and a ballot compaction of the light experts in id order
        __shared__ int s_wtiles[kPrepWarps], s_wlight[kPrepWarps];
        const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int c = e < E ? counts[e] : 0;
        const int nt = c > 0 && c >= min_tokens ? (c + kNT - 1) / kNT : 0;
        const bool is_light = c > 0 && c < min_tokens;
        int incl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned lb = __ballot_sync(0xffffffffu, is_light);
        if (lane == 31) s_wtiles[warp] = incl;
        if (lane == 0) s_wlight[warp] = __popc(lb);
        __syncthreads();
        int tbase = 0, lbase = 0;
        for (int w = 0; w < warp; ++w) {
            tbase += s_wtiles[w];
            lbase += s_wlight[w];
        }
        if (is_light) light[lbase + __popc(lb & ((1u << lane) - 1u))] = e;
        if (e == kPrepWarps * 32 - 1) {
            *n_tiles = tbase + incl;
            *n_light = lbase + __popc(lb);
        }
        const int o = e < E ? offsets[e] : 0;
        for (int j = 0; j < nt; ++j) {
            int32_t *t = tiles + 4 * (tbase + incl - nt + j);
            t[0] = e;
            t[1] = o + j * kNT;
            t[2] = min(kNT, c - j * kNT);
            t[3] = 0;
        }
    }
    const int per_row = H / 16;
    const int64_t total = (int64_t)A * per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(i / per_row), c = (int)(i % per_row);
        const int t = perm[p] / k;
        const float sx = exp2i(-__ldg(texp + t));
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        // Q2_K: positions 16c .. 16c+15 interleave elements 32(c/2) + 8(c%2) + l'
        // and the same + 16 (l' = 0..7); codebook: elements 16c .. 16c+15
        const int e0 = permute32 ? 32 * (c >> 1) + 8 * (c & 1) : 16 * c;
        const int e1 = permute32 ? e0 + 16 : e0 + 8;
        const uint4 ra = __ldg(src + e0 / 8), rb = __ldg(src + e1 / 8);
        const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
        __half ha[8], hb[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            ha[2 * j] = __float2half_rn(bf16_bits(wa[j] & 0xFFFFu) * sx);
            ha[2 * j + 1] = __float2half_rn(bf16_bits(wa[j] >> 16) * sx);
            hb[2 * j] = __float2half_rn(bf16_bits(wb[j] & 0xFFFFu) * sx);
            hb[2 * j + 1] = __float2half_rn(bf16_bits(wb[j] >> 16) * sx);
        }
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 lo, hi;
            if (permute32) {
                lo = __halves2half2(ha[2 * j], hb[2 * j]);
                hi = __halves2half2(ha[2 * j + 1], hb[2 * j + 1]);
                o[2 * j] = *reinterpret_cast<const uint32_t *>(&lo);
                o[2 * j + 1] = *reinterpret_cast<const uint32_t *>(&hi);
            } else {
                lo = __halves2half2(ha[2 * j], ha[2 * j + 1]);
                hi = __halves2half2(hb[2 * j], hb[2 * j + 1]);
                o[j] = *reinterpret_cast<const uint32_t *>(&lo);
                o[4 + j] = *reinterpret_cast<const uint32_t *>(&hi);
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(xseg + (size_t)p * H + 16 * c);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
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

template <int FMT>
cudaError_t launch_tc_down(const CUtensorMap &w, const CUtensorMap &h, const TcArgs &args, int grid,
                           cudaStream_t s)
{
    const size_t smem = DownRing<FMT>::kBytes + 1024;
    cudaError_t e = cudaFuncSetAttribute(tc_down_kernel<FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    tc_down_kernel<FMT><<<grid, kDownThreads, smem, s>>>(w, h, args);
    return cudaGetLastError();
}

template <int MODE, int FMT>
cudaError_t launch_tc(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b,
                      const TcArgs &args, int grid, cudaStream_t s)
{
    const size_t smem = Ring<MODE, FMT>::kBytes + 1024;
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
// box = box_words x 128 rows x 1 expert, no swizzle, zero fill.
cudaError_t weight_map(CUtensorMap *m, const void *base, int64_t row_bytes, int64_t rows,
                       int64_t expert_stride, int64_t experts, int phases, int box_words)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    // `phases` consecutive rows form one super-row (phases * row_bytes is a
    // multiple of 16); the box covers 128 / phases super-rows
    cuuint64_t dims[3] = {(cuuint64_t)(phases * row_bytes / 4), (cuuint64_t)(rows / phases),
                          (cuuint64_t)experts};
    cuuint64_t strides[2] = {(cuuint64_t)(phases * row_bytes), (cuuint64_t)expert_stride};
    cuuint32_t box[3] = {(cuuint32_t)box_words, (cuuint32_t)(kBM / phases), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool tc_path_supported(const Plan &p, const ds4g_moe_desc *d)
{
    // every format has a tensor-core dequantizer (Q6_K only for W_down)
    const auto fmt_ok = [](int f) {
        return f == DS4G_FMT_Q2K || f == DS4G_FMT_CB2 || f == DS4G_FMT_MXFP4 ||
               f == DS4G_FMT_Q4K || f == DS4G_FMT_Q5K;
    };
    return p.A > 0 && fmt_ok(d->format) && (fmt_ok(d->down_format) || d->down_format == DS4G_FMT_Q6K) &&
           d->gate_up_row_bytes % 16 == 0 && d->down_row_bytes % 16 == 0 && p.H % kBM == 0;
}

int32_t tc_max_tiles(int32_t E, int32_t A) { return E + A / kNT + 1; }

cudaError_t launch_token_exponents(const uint16_t *x, int T, int H, int32_t *texp, cudaStream_t s)
{
    token_exp_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, T, H, texp);
    return cudaGetLastError();
}

cudaError_t launch_tc_prep(const LayerArgs &la, const TcBufs &tb, const DeviceInfo &dev,
                           cudaStream_t s)
{
    cudaError_t e = launch_token_exponents(la.x, la.T, la.H, tb.texp, s);
    if (e != cudaSuccess) return e;
    const int prep_grid = dev.sm_count * 4;
    tc_prep_kernel<<<prep_grid, kPrepWarps * 32, 0, s>>>(la.x, la.H, la.k, la.A, la.perm, la.counts,
                                             la.offsets, la.E, tb.xseg, tb.tiles, tb.n_tiles,
                                             perm32_format(la.gu_format) ? 1 : 0, la.wts, tb.wseg,
                                             tb.texp, tb.eseg, tb.min_tokens, tb.light, tb.n_light);
    return cudaGetLastError();
}

cudaError_t launch_tc_path(const LayerArgs &la, const TcBufs &tb, const DeviceInfo &dev,
                           cudaStream_t s, const cudaEvent_t *ev, uint64_t wait_ns,
                           bool stall)
{
    CUtensorMap m_gate, m_up, m_down, m_x, m_h;
    cudaError_t e;
    const int nw = la.n_wslots;             // experts (or slots) the weight tensors hold
    const int gw = win_words(la.gu_format), dw = win_words(la.dn_format);
    if ((e = weight_map(&m_gate, la.w_gate, la.gu_row, la.I, la.gu_stride, nw, 1, gw)) != cudaSuccess ||
        (e = weight_map(&m_up, la.w_up, la.gu_row, la.I, la.gu_stride, nw, 1, gw)) != cudaSuccess ||
        (e = weight_map(&m_down, la.w_down, la.dn_row, la.H, la.dn_stride, nw, 1, dw)) != cudaSuccess ||
        (e = act_map(&m_x, tb.xseg, la.H, la.A)) != cudaSuccess ||
        (e = act_map(&m_h, tb.hp, la.I_pad, la.A)) != cudaSuccess)
        return e;

    TcArgs a{};
    a.H = la.H;
    a.I_pad = la.I_pad;
    a.tiles = tb.tiles;
    a.n_tiles = tb.n_tiles;
    a.wseg = tb.wseg;
    a.eseg = tb.eseg;
    a.hp = tb.hp;
    a.yslot = la.yslot;
    a.status = tb.status;
    a.wslot = la.wslot;
    a.n_wslots = la.n_wslots;
    a.wait_ns = wait_ns;
    a.stall = stall ? 1 : 0;

    a.K = la.H;
    a.m_tiles = la.I_pad / kBM;
    a.codebook = la.codebook;
    a.h_perm32 = perm32_format(la.dn_format) ? 1 : 0;
    // per-segment split: the light segments' experts on the GEMV kernels
    LayerArgs lg = la;
    lg.active = tb.light;
    lg.n_active = tb.n_light;
    const bool split = tb.min_tokens > 0;
    switch (la.gu_format) {
    case DS4G_FMT_CB2: e = launch_tc<0, DS4G_FMT_CB2>(m_gate, m_up, m_x, a, dev.sm_count, s); break;
    case DS4G_FMT_MXFP4: e = launch_tc<0, DS4G_FMT_MXFP4>(m_gate, m_up, m_x, a, dev.sm_count, s); break;
    case DS4G_FMT_Q4K: e = launch_tc<0, DS4G_FMT_Q4K>(m_gate, m_up, m_x, a, dev.sm_count, s); break;
    case DS4G_FMT_Q5K: e = launch_tc<0, DS4G_FMT_Q5K>(m_gate, m_up, m_x, a, dev.sm_count, s); break;
    default: e = launch_tc<0, DS4G_FMT_Q2K>(m_gate, m_up, m_x, a, dev.sm_count, s); break;
    }
    if (e != cudaSuccess) return e;
    if (split && (e = launch_gemv_gateup(lg, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[2], s)) != cudaSuccess) return e;

    a.K = la.I_pad;
    a.m_tiles = la.H / kBM;
    switch (la.dn_format) {
    case DS4G_FMT_CB2: e = launch_tc_down<DS4G_FMT_CB2>(m_down, m_h, a, dev.sm_count, s); break;
    case DS4G_FMT_MXFP4: e = launch_tc<1, DS4G_FMT_MXFP4>(m_down, m_down, m_h, a, dev.sm_count, s); break;
    case DS4G_FMT_Q4K: e = launch_tc<1, DS4G_FMT_Q4K>(m_down, m_down, m_h, a, dev.sm_count, s); break;
    case DS4G_FMT_Q5K: e = launch_tc<1, DS4G_FMT_Q5K>(m_down, m_down, m_h, a, dev.sm_count, s); break;
    case DS4G_FMT_Q6K: e = launch_tc<1, DS4G_FMT_Q6K>(m_down, m_down, m_h, a, dev.sm_count, s); break;
    default: e = launch_tc<1, DS4G_FMT_Q2K>(m_down, m_down, m_h, a, dev.sm_count, s); break;
    }
    if (e != cudaSuccess) return e;
    if (split && (e = launch_gemv_down(lg, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[3], s)) != cudaSuccess) return e;

    if ((e = launch_combine(la, dev, s)) != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[4], s)) != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ds4g
