// decode.cu -- the decode path for Q2_K experts: small expert segments
// (micro-batched decode, ds4 README mirror, "So, what can I do with this
// software?"), bound by the HBM bytes of the quantized weights.
//
//   gate/up: h[p, n] = SiLU(W_gate[e][n,:] . x_t) * (W_up[e][n,:] . x_t)
//   down:    y[t, m] = sum_{i<k} w[t,i] * (W_down[e_i][m,:] . h[p(t,i), :])
//
// Up to 8 tokens, one persistent kernel runs the whole layer
// (decode_q2k_kernel, below), one CTA per SM; from 9 to 32 tokens the
// tcgen05 kernel further down (decode_tc_kernel) does, with the same routing
// and work claiming.  Every CTA first routes all T tokens itself (top-k, counts, offsets,
// the stable token-by-expert order) into shared memory, so no work item
// waits on global metadata; CTA 0 also writes the routing to the workspace.
// A tiny kernel ahead of it (decode_pre_kernel) resets the claim counters
// and, when the activations do not fit in shared memory, converts them;
// programmatic dependent launch overlaps the two.  A producer warp then
// claims work from two global counters -- first 16-row gate/up tiles
// (expert, rows), then 32-row down items -- and streams each claimed tile
// (runs of 84-byte blocks: the whole tile, pairs of padded gate/up rows, or
// single padded down rows) into a shared-memory ring with
// cp.async.bulk (TMA, no tensor map) completing on mbarriers; a down stage
// also carries the h rows of its experts.  The ring keeps streaming W_down
// right after W_gate/W_up, so HBM does not idle at the phase boundary.
// Twelve consumer warps dequantize in registers straight into mma.sync
// m16n8k16 fragments; each warp owns one (matrix, half) pair and every
// third K block of a tile, and the warps' partial sums meet in shared
// memory.  (Fourteen warps in all, so each thread may use 128 registers.)
//
// Phase order without a grid barrier: a gate/up tile bumps its expert's
// completion counter after its h rows are written (fence, then atomic); the
// producer issues a down tile of expert e only once that counter shows all
// of e's tiles.  Work is claimed dynamically, so a tile that is waited on has
// always been claimed by a CTA that is running; every wait is bounded.
//
// Block-diagonal activation operand.  A Q2_K weight is
// w = d*sc_s*q - dmin*m_s with per-row, per-16-weight-sub-block scales.  One
// MMA takes 16 rows x 16 k-slots of A and 16 k-slots x 8 columns of B; here
// the 8 columns are the 8 sub-blocks of one half super-block: column n of B
// holds x only in the slots that belong to sub-block n (zero elsewhere).  So
// D[row, n] = sum over sub-block n of A*x, and the sub-block scale is applied
// once per 16 weights in the epilogue instead of once per weight.
//
// A fragments without a multiply: a 2-bit quant field is OR-ed into the
// mantissa of fp16 1024 (lop3 with a mask), giving 1024 + q*4^g exactly for
// bit field g.  The constant 1024*sum(x) that this adds to column n is removed
// by starting the accumulator at -1024*X_n (X_n = sum of sub-block n of x),
// so D = 4^g * sum(q*x).  Products are exact in the MMA (11-bit x 11-bit);
// accumulation is fp32.
//
// Activations enter as fp16 (bf16 -> fp16 is exact for 6.1e-5 <= |x| <=
// 65504; smaller magnitudes become fp16 subnormals).  h leaves the gate/up
// phase as fp16 (one rounding, relative 2^-11) with fp32 sub-block sums of
// those fp16 values for the down phase's correction and min terms.  When the
// layer's activations fit, every CTA converts them into its shared memory.
//
// Every mbarrier and counter wait is bounded (globaltimer); on expiry the
// kernel records DS4G_ERR_TIMEOUT in the workspace status word, drains its
// own copies (also bounded) and returns.
#include "ds4g_common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"
#include "topk.cuh"

namespace ds4g {
namespace {

constexpr int kTileM = 16;

// 4-group permutation of activations: element i of an aligned group of 4 is
// stored at position perm4(i), so that elements (i, i+2) are adjacent.
__device__ __forceinline__ int perm4(int n) { return (n & ~3) | ((n & 1) << 1) | ((n >> 1) & 1); }

// 4-bit fields as floats without the integer-conversion pipe: OR into the
// mantissa of 2^23, subtract 2^23 (exact).
__device__ __forceinline__ float nib_lo(uint32_t b)
{
    return __uint_as_float(ptx::lop3_and_or(b, 15u, 0x4B000000u)) - 8388608.0f;
}
__device__ __forceinline__ float nib_hi(uint32_t b) { return nib_lo(b >> 4); }
// The low 4 bits of b as the float 2^23 + v (exact).
__device__ __forceinline__ float nib23(uint32_t b)
{
    return __uint_as_float(ptx::lop3_and_or(b, 15u, 0x4B000000u));
}

__device__ __forceinline__ void set_status(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// One half (128 weights) of one super-block for rows (grp, grp+8) of a tile:
// builds the A fragments of the 8 MMAs.  `blk0`/`blk1`: the block of row grp
// and of row grp+8 in shared memory.
struct HalfA {
    uint32_t a[8][4];
};

// Lane constants of build_half_a: the two bit-field masks and the qs byte
// offset of this lane's 16 weights.
struct LaneA {
    uint32_t m1, m2;
    int off;
};

__device__ __forceinline__ LaneA lane_a(int h, int c)
{
    const uint32_t g1 = (uint32_t)(c >> 1);
    LaneA l;
    l.m1 = 0x00030003u << (2 * g1);          // field g1   -> sub-block c
    l.m2 = 0x00030003u << (2 * (g1 + 2));    // field g1+2 -> sub-block c+4
    l.off = 16 + 32 * h + 16 * (c & 1);
    return l;
}

__device__ __forceinline__ void build_half_a(HalfA &ha, const uint8_t *blk0, const uint8_t *blk1,
                                             const LaneA &la)
{
    const uint32_t m1 = la.m1, m2 = la.m2;
    const int off = la.off;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t r0 = ptx::lds32(blk0 + off + 4 * w);
        const uint32_t r1 = ptx::lds32(blk1 + off + 4 * w);
        const uint32_t r0h = r0 >> 8, r1h = r1 >> 8;
        // MMA t = 2w (bytes 0,2 of the word) and t = 2w+1 (bytes 1,3)
        ha.a[2 * w][0] = ptx::lop3_and_or(r0, m1, 0x64006400u);
        ha.a[2 * w][1] = ptx::lop3_and_or(r1, m1, 0x64006400u);
        ha.a[2 * w][2] = ptx::lop3_and_or(r0, m2, 0x64006400u);
        ha.a[2 * w][3] = ptx::lop3_and_or(r1, m2, 0x64006400u);
        ha.a[2 * w + 1][0] = ptx::lop3_and_or(r0h, m1, 0x64006400u);
        ha.a[2 * w + 1][1] = ptx::lop3_and_or(r1h, m1, 0x64006400u);
        ha.a[2 * w + 1][2] = ptx::lop3_and_or(r0h, m2, 0x64006400u);
        ha.a[2 * w + 1][3] = ptx::lop3_and_or(r1h, m2, 0x64006400u);
    }
}

constexpr int kConsumers = 12;
constexpr int kKPhases = kConsumers / 4;   // warps per (matrix or m-tile, half) pair
constexpr int kProducerWarp = kConsumers;
constexpr int kThreads = (kConsumers + 2) * 32;
// Register budget: with 14 warps at most 4 share an SM sub-partition (16K
// registers), so 128 registers per thread fit; bounds of 512 threads let the
// compiler use them.
constexpr int kLaunchBound = 512;
// named barriers: 1 = consumers only; 2, 3 = reduction buffer 0/1 filled
// (consumers arrive, epilogue warp waits); 4, 5 = buffer 0/1 released
// (epilogue warp arrives, consumers wait)
constexpr int kBarConsumers = 1, kBarJobFull = 2, kBarJobEmpty = 4, kBarConvert = 6;
constexpr int kJobThreads = (kConsumers + 1) * 32;
constexpr int kDownRows = 32;            // rows of H per down item (two MMA tiles)
constexpr int kMaxDownPerStage = 8;
constexpr int kDownPairs = 4;             // (expert, token chunk) pairs per down reduction round
constexpr size_t kSmemBudget = 216 * 1024;     // dynamic shared memory of the decode kernel
constexpr size_t kXStageMax = 48 * 1024;
constexpr int kMaxAssign = kDecodeMaxT * DS4G_MAX_TOPK;     // 256

// Stage tag written by the producer before it arms the stage's barrier:
// [0] kind, [1] item, [2] first active-expert index, [3] experts in the stage,
// [4 + 2j] byte offset of expert j's W_down tile, [5 + 2j] byte offset of its
// h rows (h sums follow them), or -1 when h is read from global memory.
enum { kTagEnd = -1, kTagGateUp = 0, kTagDown = 1 };
constexpr int kTagWords = 4 + 2 * kMaxDownPerStage;

struct DecArgs {
    int H, I, I_pad, E, k, T, A, score;
    int H_blocks, I_blocks;
    const uint8_t *w_gate, *w_up, *w_down;
    int64_t gu_row, dn_row, gu_stride, dn_stride;
    const int32_t *wslot;  // [E] weight slot of each expert, or null (slot = expert)
    int n_wslots;
    int gu_pitch, dn_pitch;   // row pitch of the tiles in shared memory (padded against bank conflicts)
    const float *logits;   // [T][E]
    const uint16_t *x;     // [T][H] bf16
    const __half *xp;      // [T][H] converted by decode_pre_kernel (x_smem == 0)
    const float *xs;       // [T][H/16]
    const int32_t *texp;   // [T] token exponents written by decode_pre_kernel (x_smem == 0)
    __half *hp;            // [A][I_pad]
    float *hs;             // [A][I_pad/16]
    float *y;              // [T][H]
    int32_t *ids, *counts, *offsets, *perm;   // routing outputs (CTA 0)
    float *wts;
    int32_t *status;
    int32_t *sync;         // [0] gate/up claim, [1] down claim, [4 + e] h values done of expert e
    uint64_t wait_ns;
    int stages;
    uint32_t stage_bytes;
    int x_smem;            // activations converted into shared memory
    int stall;             // debug: the producer issues nothing (tests the bounded waits)
};

// Routing of the call in shared memory.
struct RouteSmem {
    int32_t ids[kMaxAssign];
    float wts[kMaxAssign];
    int32_t perm[kMaxAssign];      // segment position -> assignment
    int32_t slot[kMaxAssign];      // assignment -> segment position
    int32_t cnt[DS4G_MAX_EXPERTS];
    int32_t off[DS4G_MAX_EXPERTS + 1];
    int32_t act[DS4G_MAX_EXPERTS];
    int32_t n_act;
};

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void named_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void consumer_sync() { named_sync(kBarConsumers, kConsumers * 32); }

// One epilogue job: the consumers' partial sums of one token chunk of one
// gate/up tile sit in reduction buffer `rb`; the epilogue warp finishes it
// (SiLU * up, the h stores, and publishing them to the down phase).
enum { kJobStop = 0, kJobGateUp = 1 };
struct Job {
    int kind, e, mt, seg0, c0, nt, item, last;
};

// Bounded wait for a global counter to reach `target` (acquire, gpu scope).
__device__ __forceinline__ bool wait_counter(const int32_t *p, int target, uint64_t limit_ns)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        __nanosleep(64);
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// h of the gate/up phase is written by other CTAs of this kernel: read it at
// L2 (ld.global.cg), never through a possibly stale L1 line.
__device__ __forceinline__ uint4 ld_cg4(const void *p) { return __ldcg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ float2 ld_cg2f(const float *p) { return __ldcg(reinterpret_cast<const float2 *>(p)); }

// The 8 MMAs of one half for one activation vector.  `xh`: the half's 128
// activations (fp16, 4-group permuted); `xs`: its 8 sub-block sums.
// SHARED: both in shared memory; lanes whose B registers are zero read the
// 32-byte zero buffer `zero` instead, so no selects are needed.  Otherwise
// global memory written by other CTAs of this kernel.  Returns D (rows grp,
// grp+8 x columns 2c, 2c+1) = 4^c * sum_{sub-block} q*x.
template <bool SHARED>
__device__ __forceinline__ void half_mma_v(const HalfA &ha, const __half *xh, const float *xs,
                                           const __half *zero, int grp, int c, float (&d)[4],
                                           float &x0, float &x1)
{
    const float2 xx = SHARED ? *reinterpret_cast<const float2 *>(xs + 2 * c) : ld_cg2f(xs + 2 * c);
    x0 = xx.x;
    x1 = xx.y;
    d[0] = -1024.0f * x0;
    d[1] = -1024.0f * x1;
    d[2] = d[0];
    d[3] = d[1];
    const bool act = (grp & 3) == c, lo = grp < 4;
    uint32_t b0[8], b1[8];
    if (SHARED) {
        const uint4 *p0 = reinterpret_cast<const uint4 *>(act && lo ? xh + 16 * grp : zero);
        const uint4 *p1 = reinterpret_cast<const uint4 *>(act && !lo ? xh + 16 * grp : zero);
        const uint4 u0 = p0[0], u1 = p0[1], v0 = p1[0], v1 = p1[1];
        b0[0] = u0.x; b0[1] = u0.y; b0[2] = u0.z; b0[3] = u0.w;
        b0[4] = u1.x; b0[5] = u1.y; b0[6] = u1.z; b0[7] = u1.w;
        b1[0] = v0.x; b1[1] = v0.y; b1[2] = v0.z; b1[3] = v0.w;
        b1[4] = v1.x; b1[5] = v1.y; b1[6] = v1.z; b1[7] = v1.w;
    } else {
        uint32_t bv[8];
        if (act) {
            const uint4 u0 = ld_cg4(xh + 16 * grp), u1 = ld_cg4(xh + 16 * grp + 8);
            bv[0] = u0.x; bv[1] = u0.y; bv[2] = u0.z; bv[3] = u0.w;
            bv[4] = u1.x; bv[5] = u1.y; bv[6] = u1.z; bv[7] = u1.w;
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) bv[t] = 0u;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            b0[t] = lo ? bv[t] : 0u;
            b1[t] = lo ? 0u : bv[t];
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) ptx::mma_16816(d, ha.a[t], b0[t], b1[t], d);
}

// One (K block, half) unit of one 16-row tile for up to NT activation
// vectors: accumulates d * (scale terms) - dmin * (min terms) into part.
// `blk0`: block kb of row grp of the tile in shared memory; `xk`/`sk`: the
// K block's activations / sub-block sums; `off[j]`: element offset of
// vector j's activations (its sums start at off[j] / 16).
template <int NT, bool SHARED>
__device__ __forceinline__ void tile_unit(const uint8_t *blk0, int64_t row_bytes, int h, int grp,
                                          int c, const LaneA &la, float inv4c, const __half *xk,
                                          const float *sk, const __half *zero,
                                          const uint32_t (&off)[NT], int nt, float (&part)[NT][2])
{
    const uint8_t *blk1 = blk0 + 8 * row_bytes;
    const uint32_t dd0 = ptx::lds32(blk0 + 80), dd1 = ptx::lds32(blk1 + 80);
    HalfA ha;
    build_half_a(ha, blk0, blk1, la);
    const uint32_t sb0 = *reinterpret_cast<const uint16_t *>(blk0 + 8 * h + 2 * c);
    const uint32_t sb1 = *reinterpret_cast<const uint16_t *>(blk1 + 8 * h + 2 * c);
    // d*sc and dmin*m per sub-block (columns 2c, 2c+1), rows grp and grp+8
    const float d0 = half_bits(dd0 & 0xFFFFu) * inv4c, dm0 = half_bits(dd0 >> 16);
    const float d1 = half_bits(dd1 & 0xFFFFu) * inv4c, dm1 = half_bits(dd1 >> 16);
    const float s00 = d0 * nib_lo(sb0), s01 = d0 * nib_lo(sb0 >> 8);
    const float s10 = d1 * nib_lo(sb1), s11 = d1 * nib_lo(sb1 >> 8);
    const float m00 = dm0 * nib_hi(sb0), m01 = dm0 * nib_hi(sb0 >> 8);
    const float m10 = dm1 * nib_hi(sb1), m11 = dm1 * nib_hi(sb1 >> 8);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < nt) {
            float d[4], x0, x1;
            half_mma_v<SHARED>(ha, xk + off[j] + 128 * h, sk + (off[j] >> 4) + 8 * h, zero, grp, c,
                               d, x0, x1);
            part[j][0] += s00 * d[0] + s01 * d[1] - (m00 * x0 + m01 * x1);
            part[j][1] += s10 * d[2] + s11 * d[3] - (m10 * x0 + m11 * x1);
        }
    }
}

// tile_unit with every operand in shared memory, addressed by 32-bit
// shared-window addresses: `blk0` (block kb of row grp), `xk`/`sk` (the K
// block's activations / sums).  off[j]: element offset of vector j's
// activations (its sums start at off[j] / 16).
//
// Shared-memory traffic is kept to about 17 wavefronts per unit:
//  * lanes with odd c read their qs words rotated by two words, so the two
//    16-byte halves of a row's 32-byte qs chunk land in different banks; the
//    activation operand of those sub-blocks is loaded with the same rotation,
//    so every MMA still pairs each weight with its activation;
//  * b0/b1 are the caller's registers, zero in every lane that holds no
//    diagonal entry: only the 8 lanes on the diagonal load (predicated), the
//    others keep their zeros across units;
//  * the 4-bit scales and mins are read from the scale bytes with ALU
//    operations instead of a table: (2^23 + v) as a float, times s, minus
//    2^23 * s, is v * s exactly in one fma.
template <int NT>
__device__ __forceinline__ void tile_unit_s(uint32_t blk0, uint32_t pitch, int h, int grp, int c,
                                            const LaneA &la, float inv4c, uint32_t xk, uint32_t sk,
                                            const uint32_t (&off)[NT], int nt, uint32_t (&b0)[8],
                                            uint32_t (&b1)[8], float (&part)[NT][2])
{
    const uint32_t blk1 = blk0 + 8 * pitch;
    const uint32_t dd0 = ptx::ld_s32(blk0 + 80), dd1 = ptx::ld_s32(blk1 + 80);
    const uint32_t rot = (uint32_t)(c & 1) * 8u;
    HalfA ha;
    {
        const uint32_t m1 = la.m1, m2 = la.m2;
        const uint32_t q0 = blk0 + la.off, q1 = blk1 + la.off;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t o = (4u * w + rot) & 15u;
            const uint32_t r0 = ptx::ld_s32(q0 + o), r1 = ptx::ld_s32(q1 + o);
            const uint32_t r0h = r0 >> 8, r1h = r1 >> 8;
            ha.a[2 * w][0] = ptx::lop3_and_or(r0, m1, 0x64006400u);
            ha.a[2 * w][1] = ptx::lop3_and_or(r1, m1, 0x64006400u);
            ha.a[2 * w][2] = ptx::lop3_and_or(r0, m2, 0x64006400u);
            ha.a[2 * w][3] = ptx::lop3_and_or(r1, m2, 0x64006400u);
            ha.a[2 * w + 1][0] = ptx::lop3_and_or(r0h, m1, 0x64006400u);
            ha.a[2 * w + 1][1] = ptx::lop3_and_or(r1h, m1, 0x64006400u);
            ha.a[2 * w + 1][2] = ptx::lop3_and_or(r0h, m2, 0x64006400u);
            ha.a[2 * w + 1][3] = ptx::lop3_and_or(r1h, m2, 0x64006400u);
        }
    }
    const uint32_t sb0 = ptx::ld_s16(blk0 + 8 * h + 2 * c), sb1 = ptx::ld_s16(blk1 + 8 * h + 2 * c);
    const float d0 = half_bits(dd0 & 0xFFFFu) * inv4c, dm0 = half_bits(dd0 >> 16);
    const float d1 = half_bits(dd1 & 0xFFFFu) * inv4c, dm1 = half_bits(dd1 >> 16);
    const float nd0 = -8388608.0f * d0, ndm0 = -8388608.0f * dm0;
    const float nd1 = -8388608.0f * d1, ndm1 = -8388608.0f * dm1;
    const float s00 = fmaf(nib23(sb0), d0, nd0), s01 = fmaf(nib23(sb0 >> 8), d0, nd0);
    const float m00 = fmaf(nib23(sb0 >> 4), dm0, ndm0), m01 = fmaf(nib23(sb0 >> 12), dm0, ndm0);
    const float s10 = fmaf(nib23(sb1), d1, nd1), s11 = fmaf(nib23(sb1 >> 8), d1, nd1);
    const float m10 = fmaf(nib23(sb1 >> 4), dm1, ndm1), m11 = fmaf(nib23(sb1 >> 12), dm1, ndm1);
    const uint32_t ld_lo = (grp & 3) == c && grp < 4, ld_hi = (grp & 3) == c && grp >= 4;
    const uint32_t sw = (uint32_t)(c & 1) * 16u;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        if (j < nt) {
            const uint32_t xa = xk + 2 * (off[j] + 128 * h + 16 * grp);
            const float2 xx = ptx::ld_s64f(sk + 4 * ((off[j] >> 4) + 8 * h + 2 * c));
            ptx::ld_s128_if(ld_lo, xa + sw, b0);
            ptx::ld_s128_if(ld_lo, xa + (sw ^ 16u), b0 + 4);
            ptx::ld_s128_if(ld_hi, xa + sw, b1);
            ptx::ld_s128_if(ld_hi, xa + (sw ^ 16u), b1 + 4);
            // two accumulator chains (even and odd MMAs) halve the dependent latency
            float de[4] = {-1024.0f * xx.x, -1024.0f * xx.y, -1024.0f * xx.x, -1024.0f * xx.y};
            float dq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int t = 0; t < 8; t += 2) {
                ptx::mma_16816(de, ha.a[t], b0[t], b1[t], de);
                ptx::mma_16816(dq, ha.a[t + 1], b0[t + 1], b1[t + 1], dq);
            }
            float p = part[j][0], r = part[j][1];
            p = fmaf(s00, de[0] + dq[0], p); p = fmaf(s01, de[1] + dq[1], p);
            p = fmaf(-m00, xx.x, p); p = fmaf(-m01, xx.y, p);
            r = fmaf(s10, de[2] + dq[2], r); r = fmaf(s11, de[3] + dq[3], r);
            r = fmaf(-m10, xx.x, r); r = fmaf(-m11, xx.y, r);
            part[j][0] = p;
            part[j][1] = r;
        }
    }
}

// Quad-reduces this warp's partial sums into red[warp][j][16] (the caller
// reads red after consumer_sync).
template <int NT>
__device__ __forceinline__ void store_partials(float *red, int warp, int grp, int c,
                                               float (&part)[NT][2])
{
    float *rw = red + (size_t)warp * NT * kTileM;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float v = part[j][r];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (c == 0) rw[j * kTileM + grp + 8 * r] = v;
        }
}

// Routing of all T tokens by the whole CTA into shared memory (every CTA
// computes the same result); CTA 0 writes it to the workspace.
__device__ void route_into_smem(const DecArgs &a, RouteSmem &r)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = blockDim.x >> 5;
    const int A = a.A;
    for (int t = warp; t < a.T; t += nw)
        topk_warp(a.logits + (size_t)t * a.E, a.E, a.k, a.score, r.ids + t * a.k, r.wts + t * a.k);
    for (int e = tid; e < DS4G_MAX_EXPERTS; e += blockDim.x) r.cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < A; i += blockDim.x) atomicAdd(&r.cnt[r.ids[i]], 1);
    __syncthreads();
    if (warp == 0) {
        // exclusive scan of the counts (8 experts per lane) and the active list
        int c[kMaxPerLane], sum = 0;
#pragma unroll
        for (int j = 0; j < kMaxPerLane; ++j) {
            const int e = lane * kMaxPerLane + j;
            c[j] = e < a.E ? r.cnt[e] : 0;
            sum += c[j];
        }
        int incl = sum, nact = 0;
#pragma unroll
        for (int j = 0; j < kMaxPerLane; ++j) nact += c[j] > 0;
        int nincl = nact;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            const int w = __shfl_up_sync(0xffffffffu, nincl, o);
            if (lane >= o) { incl += v; nincl += w; }
        }
        int run = incl - sum, arun = nincl - nact;
#pragma unroll
        for (int j = 0; j < kMaxPerLane; ++j) {
            const int e = lane * kMaxPerLane + j;
            if (e < a.E) {
                r.off[e] = run;
                if (c[j] > 0) r.act[arun++] = e;
            }
            run += c[j];
        }
        if (lane == 31) {
            r.off[a.E] = incl;
            r.n_act = nincl;
        }
    }
    __syncthreads();
    // stable placement: rank of assignment i among the earlier ones of its expert
    for (int i = tid; i < A; i += blockDim.x) {
        const int e = r.ids[i];
        int rank = 0;
        for (int q = 0; q < i; ++q) rank += r.ids[q] == e;
        const int pos = r.off[e] + rank;
        r.perm[pos] = i;
        r.slot[i] = pos;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int i = tid; i < A; i += blockDim.x) {
            a.ids[i] = r.ids[i];
            a.wts[i] = r.wts[i];
            a.perm[i] = r.perm[i];
        }
        for (int e = tid; e < a.E; e += blockDim.x) a.counts[e] = r.cnt[e];
        if (tid == 0) a.offsets[a.E] = r.off[a.E];
        for (int e = tid; e < a.E; e += blockDim.x) a.offsets[e] = r.off[e];
    }
}

constexpr int kWarpRouteT = 4;   // T at or below which one warp routes (T*k <= 32)

// Routing of up to 32 assignments by one warp (the producer warp) into
// shared memory: top-k per token, then counts, offsets, the stable
// token-by-expert order and the active list from warp votes.  Only the
// entries of active experts are written.  In CTA 0 the warp also writes the
// routing to the workspace.
__device__ void route_warp(const DecArgs &a, RouteSmem &r)
{
    const int lane = threadIdx.x & 31;
    for (int t = 0; t < a.T; ++t)
        topk_warp(a.logits + (size_t)t * a.E, a.E, a.k, a.score, r.ids + t * a.k, r.wts + t * a.k);
    __syncwarp();
    const bool valid = lane < a.A;
    const int e = valid ? r.ids[lane] : 0x1FF;               // invalid lanes sort last
    // lanes whose expert id is smaller than this lane's (`less`) or equal
    // (`peers`), one ballot per bit of the 9-bit key, most significant first
    unsigned less = 0u, peers = 0xffffffffu;
#pragma unroll
    for (int b = 8; b >= 0; --b) {
        const unsigned bit = (unsigned)(e >> b) & 1u;
        const unsigned ones = __ballot_sync(0xffffffffu, bit);
        if (bit) less |= peers & ~ones;
        peers &= bit ? ones : ~ones;
    }
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = valid && rank == 0;
    const unsigned lm = __ballot_sync(0xffffffffu, leader);
    const int off = __popc(less);              // invalid keys are larger than every valid one
    const int aidx = __popc(less & lm);
    if (valid) {
        r.perm[off + rank] = lane;
        r.slot[lane] = off + rank;
    }
    if (leader) {
        r.cnt[e] = __popc(peers);
        r.off[e] = off;
        r.act[aidx] = e;
    }
    if (lane == 0) r.n_act = __popc(lm);
    __syncwarp();
    if (blockIdx.x == 0) {
        if (valid) {
            a.ids[lane] = r.ids[lane];
            a.wts[lane] = r.wts[lane];
            a.perm[lane] = r.perm[lane];
        }
        int run = 0;
        for (int e0 = 0; e0 < a.E; e0 += 32) {
            const int me = e0 + lane;
            int cnt = 0;
            for (int i = 0; i < 32; ++i) cnt += __shfl_sync(0xffffffffu, e, i) == me;
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (me < a.E) {
                a.counts[me] = cnt;
                a.offsets[me] = run + incl - cnt;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) a.offsets[a.E] = run;
    }
}

// x (bf16) -> fp16 x * 2^-e_t in the (0, 2, 1, 3) order per 4, plus fp32
// sums of 16, for groups of 4 g0, g0 + stride, ... below n_groups (all
// threads of the CTA or a grid stride).  `texp`: e_t of each token (H
// elements per token).
__device__ __forceinline__ void convert_x(const uint16_t *x, __half *xp, float *xs, size_t g0,
                                          size_t n_groups, size_t stride, int H, const int32_t *texp)
{
    // one group of 4 per lane; lanes 4j..4j+3 of a warp form a sub-block
    for (size_t g = g0; g < n_groups; g += stride) {
        const float sx = exp2i(-texp[(4 * g) / H]);
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x) + g);
        const __half h0 = __float2half_rn(bf16_bits(raw.x & 0xFFFFu) * sx);
        const __half h1 = __float2half_rn(bf16_bits(raw.x >> 16) * sx);
        const __half h2 = __float2half_rn(bf16_bits(raw.y & 0xFFFFu) * sx);
        const __half h3 = __float2half_rn(bf16_bits(raw.y >> 16) * sx);
        __half2 *o = reinterpret_cast<__half2 *>(xp + 4 * g);
        o[0] = __halves2half2(h0, h2);
        o[1] = __halves2half2(h1, h3);
        float v = __half2float(h0) + __half2float(h1) + __half2float(h2) + __half2float(h3);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        if ((g & 3) == 0) xs[g >> 2] = v;
    }
}

// Largest finite |x| of token t's H elements over the threads of a block
// (every thread gets the result; `red` is 32 floats of shared memory).
__device__ __forceinline__ float token_max_block(const uint16_t *x, int t, int H, float *red)
{
    const uint32_t *row = reinterpret_cast<const uint32_t *>(x + (size_t)t * H);
    float m = 0.0f;
    for (int i = threadIdx.x; i < H / 2; i += blockDim.x) {
        const uint32_t w = __ldg(row + i);
        m = fmaxf(m, fmaxf(bf16_abs_finite(w & 0xFFFFu), bf16_abs_finite(w >> 16)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float r = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, red[w]);
    return r;
}

// Resets the status word and the decode kernel's counters; when the
// activations do not fit in the decode kernel's shared memory, computes
// every token's exponent (texp) and converts the activations (one block per
// token at a time).
__global__ void __launch_bounds__(256) decode_pre_kernel(int32_t *status, int32_t *sync, int n_sync,
                                                         const uint16_t *x, __half *xp, float *xs,
                                                         int T, int H, int32_t *texp)
{
    __shared__ float red[32];
    __shared__ int32_t s_e[1];
    ptx::grid_dep_launch();
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) *status = DS4G_OK;
        for (int i = threadIdx.x; i < n_sync; i += blockDim.x) sync[i] = 0;
    }
    if (!x) return;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const float m = token_max_block(x, t, H, red);
        if (threadIdx.x == 0) {
            s_e[0] = token_exponent(m);
            texp[t] = s_e[0];
        }
        __syncthreads();
        const size_t q = (size_t)H / 4;
        convert_x(x + (size_t)t * H, xp + (size_t)t * H, xs + (size_t)t * (H / 16), threadIdx.x, q,
                  blockDim.x, H, s_e);
        __syncthreads();
    }
}

// Exponents of the T tokens (s_e) from x, by `nthr` threads of the CTA with
// index i (consecutive within each warp); `sync` separates the phases (a
// named barrier over those threads, or __syncthreads).  s_m: T ints of
// shared memory for the maxima (float bits, monotone for non-negative values).
template <typename Sync>
__device__ __forceinline__ void token_exponents_cta(const uint16_t *x, int T, int H, int i,
                                                    int nthr, int *s_m, int32_t *s_e, Sync sync)
{
    for (int t = i; t < T; t += nthr) s_m[t] = 0;
    sync();
    for (int t = 0; t < T; ++t) {
        const uint32_t *row = reinterpret_cast<const uint32_t *>(x + (size_t)t * H);
        float m = 0.0f;
        for (int j = i; j < H / 2; j += nthr) {
            const uint32_t w = __ldg(row + j);
            m = fmaxf(m, fmaxf(bf16_abs_finite(w & 0xFFFFu), bf16_abs_finite(w >> 16)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((i & 31) == 0 && m > 0.0f) atomicMax(s_m + t, __float_as_int(m));
    }
    sync();
    for (int t = i; t < T; t += nthr) s_e[t] = token_exponent(__int_as_float(s_m[t]));
    sync();
}

template <int NT>
__global__ void __launch_bounds__(kLaunchBound, 1) decode_q2k_kernel(DecArgs a)
{
    // one vector: the launcher guarantees that x and every expert's h rows
    // sit in shared memory, so the global-memory unit paths are compiled out
    constexpr bool kSmemOnly = NT == 1;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ RouteSmem rs;
    __shared__ __align__(16) __half zero[16];
    __shared__ int s_pabort, s_cabort, s_consumed, s_issued;
    __shared__ Job jobs[2];
    __shared__ int32_t s_e[kDecodeMaxT];     // token exponents
    __shared__ int s_m[kDecodeMaxT];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 2, c = lane & 3;
    const uint32_t gu_tile = (uint32_t)(kTileM * a.gu_row);
    const uint32_t dn_tile = (uint32_t)(kDownRows * a.dn_row);
    const uint32_t h_row = (uint32_t)a.I_pad * 2, hs_row = (uint32_t)(a.I_pad / 16) * 4;
    uint8_t *ring = smem;
    uint8_t *p = smem + (size_t)a.stages * a.stage_bytes;
    const size_t x_bytes = a.x_smem ? (size_t)a.T * a.H * 2 : 0;
    const size_t xs_bytes = a.x_smem ? (size_t)a.T * (a.H / 16) * 4 : 0;
    __half *x_s = reinterpret_cast<__half *>(p);
    float *xs_s = reinterpret_cast<float *>(p + x_bytes);
    float *red = reinterpret_cast<float *>(p + x_bytes + xs_bytes);       // [2][16][NT][16] gate/up
    float *redd = red + 2 * kConsumers * NT * kTileM;                     // [kDownPairs][16][NT][16] down
    float *obuf = redd + kDownPairs * kConsumers * NT * kTileM;           // [A][32]
    int *tags = reinterpret_cast<int *>(obuf + (size_t)a.A * kDownRows);  // [stages][kTagWords]
    uint64_t *bars = reinterpret_cast<uint64_t *>(tags + kTagWords * a.stages);
    uint64_t *full = bars, *empty = bars + a.stages;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kConsumers);
        }
        ptx::fence_mbar_init();
        s_pabort = 0;
        s_cabort = 0;
        s_consumed = 0;
        s_issued = 0;
    }
    if (tid < 16) zero[tid] = __float2half_rn(0.0f);
    if (a.T <= kWarpRouteT && a.A <= 32) {
        // the producer warp routes while the other warps convert x (neither
        // needs the barriers or tables set up above until the barrier below)
        if (warp == kProducerWarp) {
            route_warp(a, rs);
        } else if (a.x_smem) {
            const int t2 = tid < kProducerWarp * 32 ? tid : tid - 32;
            const int nthr = blockDim.x - 32;
            token_exponents_cta(a.x, a.T, a.H, t2, nthr, s_m, s_e,
                                [&] { named_sync(kBarConvert, nthr); });
            convert_x(a.x, x_s, xs_s, t2, (size_t)a.T * (a.H / 4), nthr, a.H, s_e);
        }
        __syncthreads();
    } else {
        if (a.x_smem) {
            token_exponents_cta(a.x, a.T, a.H, tid, blockDim.x, s_m, s_e, [] { __syncthreads(); });
            convert_x(a.x, x_s, xs_s, tid, (size_t)a.T * (a.H / 4), blockDim.x, a.H, s_e);
        }
        route_into_smem(a, rs);   // ends with __syncthreads
    }

    // the counters are reset (and, without x_smem, the activations converted
    // and the token exponents written) by the kernel ahead of this one
    ptx::grid_dep_wait();
    if (!a.x_smem) {
        if (tid < a.T) s_e[tid] = a.texp[tid];
        __syncthreads();
    }

    const int n_act = rs.n_act;
    const int tiles = a.I / kTileM;
    const int gu_items = n_act * tiles;
    const int dn_items = a.H / kDownRows;
    int32_t *const claim_gu = a.sync, *const claim_dn = a.sync + 1, *const done = a.sync + 4;

    if (warp == kProducerWarp) {
        // ---------------- producer ----------------
        if (lane == 0 && !a.stall) {
            int q = 0;
            bool ok = true;
            // claims a ring slot: waits for it to be empty; false on abort
            auto slot = [&](int &s) -> bool {
                s = q % a.stages;
                if (q >= a.stages &&
                    !ptx::mbar_wait(&empty[s], ((q / a.stages) - 1) & 1, a.wait_ns)) {
                    set_status(a.status, DS4G_ERR_TIMEOUT);
                    s_pabort = 1;
                    return false;
                }
                return !*(volatile int *)&s_cabort;
            };
            // every item comes from the counter, so an item that a down item
            // waits for has always been claimed by a CTA that is running
            while (ok) {
                const int it = atomicAdd(claim_gu, 1);
                if (it >= gu_items) break;
                int s;
                if (!(ok = slot(s))) break;
                const int e = rs.act[it / tiles], mt = it % tiles;
                int *tg = tags + kTagWords * s;
                tg[0] = kTagGateUp;
                tg[1] = it;
                uint8_t *st = ring + (size_t)s * a.stage_bytes;
                const int we = weight_slot(a.wslot, a.n_wslots, e, a.status);
                const uint8_t *g = a.w_gate + (size_t)we * a.gu_stride + (size_t)mt * gu_tile;
                const uint8_t *u = a.w_up + (size_t)we * a.gu_stride + (size_t)mt * gu_tile;
                ptx::mbar_arrive_expect_tx(&full[s], 2 * gu_tile);
                if (a.gu_pitch == a.gu_row) {
                    ptx::bulk_g2s(st, g, gu_tile, &full[s]);
                    ptx::bulk_g2s(st + gu_tile, u, gu_tile, &full[s]);
                } else {
                    // padded layout: pairs of rows, each pair one copy (see gu_pair)
                    const size_t pp = 2 * (size_t)a.gu_pitch - 16;
                    for (int r = 0; r < kTileM; r += 2) {
                        ptx::bulk_g2s(st + (size_t)(r >> 1) * pp, g + (size_t)r * a.gu_row,
                                      2 * (uint32_t)a.gu_row, &full[s]);
                        ptx::bulk_g2s(st + (size_t)(kTileM / 2 + (r >> 1)) * pp, u + (size_t)r * a.gu_row,
                                      2 * (uint32_t)a.gu_row, &full[s]);
                    }
                }
                s_issued = ++q;
            }
            while (ok) {
                const int it = atomicAdd(claim_dn, 1);
                if (it >= dn_items) break;
                int j = 0;
                while (ok && j < n_act) {
                    int s;
                    if (!(ok = slot(s))) break;
                    int *tg = tags + kTagWords * s;
                    uint8_t *st = ring + (size_t)s * a.stage_bytes;
                    // pack experts j, j+1, ... with their h rows while they fit
                    const uint32_t dn_smem = (uint32_t)(kDownRows * a.dn_pitch);
                    uint32_t used = 0, bytes = 0;
                    int cnt = 0;
                    const int j0 = j;
                    while (j < n_act && cnt < kMaxDownPerStage) {
                        const int e = rs.act[j];
                        const int n_e = rs.cnt[e];
                        const uint32_t hb = (uint32_t)n_e * (h_row + hs_row);
                        const bool h_in = used + dn_smem + hb <= a.stage_bytes;
                        // the one-vector kernel reads h from shared memory
                        // only: an expert whose h rows no longer fit starts
                        // the next stage (the launcher checked that a W_down
                        // tile and its h rows fit one stage)
                        if (kSmemOnly && !h_in && cnt > 0) break;
                        const uint32_t need = dn_smem + (h_in ? hb : 0);
                        if (cnt > 0 && used + need > a.stage_bytes) break;
                        if (!wait_counter(done + e, a.I * n_e, a.wait_ns)) {
                            set_status(a.status, DS4G_ERR_TIMEOUT);
                            s_pabort = 1;
                            ok = false;
                            break;
                        }
                        tg[4 + 2 * cnt] = (int)used;
                        tg[5 + 2 * cnt] = h_in ? (int)(used + dn_smem) : -1;
                        used += need;
                        ++cnt;
                        ++j;
                    }
                    if (!ok) break;
                    tg[0] = kTagDown;
                    tg[1] = it;
                    tg[2] = j0;
                    tg[3] = cnt;
                    // h was written by other CTAs (generic proxy); the copies
                    // below read it through the async proxy
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    for (int i = 0; i < cnt; ++i)
                        bytes += dn_tile + (tg[5 + 2 * i] >= 0 ? (uint32_t)rs.cnt[rs.act[j0 + i]] * (h_row + hs_row) : 0u);
                    ptx::mbar_arrive_expect_tx(&full[s], bytes);
                    for (int i = 0; i < cnt; ++i) {
                        const int e = rs.act[j0 + i];
                        const int we = weight_slot(a.wslot, a.n_wslots, e, a.status);
                        const uint8_t *src = a.w_down + (size_t)we * a.dn_stride + (size_t)it * dn_tile;
                        if (a.dn_pitch == a.dn_row)
                            ptx::bulk_g2s(st + tg[4 + 2 * i], src, dn_tile, &full[s]);
                        else
                            for (int r = 0; r < kDownRows; ++r)
                                ptx::bulk_g2s(st + tg[4 + 2 * i] + (size_t)r * a.dn_pitch,
                                              src + (size_t)r * a.dn_row, (uint32_t)a.dn_row, &full[s]);
                        if (tg[5 + 2 * i] >= 0) {
                            const int n_e = rs.cnt[e], seg0 = rs.off[e];
                            uint8_t *hd = st + tg[5 + 2 * i];
                            ptx::bulk_g2s(hd, a.hp + (size_t)seg0 * a.I_pad, n_e * h_row, &full[s]);
                            ptx::bulk_g2s(hd + (size_t)n_e * h_row,
                                          a.hs + (size_t)seg0 * (a.I_pad / 16), n_e * hs_row,
                                          &full[s]);
                        }
                    }
                    s_issued = ++q;
                }
            }
            if (ok) {
                int s;
                if (slot(s)) {
                    tags[kTagWords * s] = kTagEnd;
                    ptx::mbar_arrive(&full[s]);
                }
            }
        }
    } else if (warp < kConsumers) {
        // ---------------- consumers ----------------
        const float inv4c = 1.0f / (float)(1 << (2 * c));
        // each consumer warp owns one (matrix or m-tile, half) pair and every
        // kKPhases-th K block: warp = 4 * wk + 2 * wm + wh, K blocks kb = wk (mod kKPhases)
        const int wm = (warp >> 1) & 1, wh = warp & 1, wk = warp >> 2;
        const LaneA la_ = lane_a(wh, c);
        const uint32_t x_s_a = ptx::smem_addr(x_s), xs_s_a = ptx::smem_addr(xs_s);
        // activation operand registers: zero except in the lanes on the block
        // diagonal, which reload them per unit (see tile_unit_s)
        uint32_t bz0[8], bz1[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) bz0[t] = bz1[t] = 0u;
        int rb = 0, uses0 = 0, uses1 = 0;
        // hands the partial sums in `part` to the epilogue warp as job `jb`
        auto emit = [&](const Job &jb, float (&part)[NT][2]) {
            int &uses = rb ? uses1 : uses0;
            if (uses > 0) named_sync(kBarJobEmpty + rb, kJobThreads);
            store_partials<NT>(red + rb * kConsumers * NT * kTileM, warp, grp, c, part);
            if (tid == 0) jobs[rb] = jb;
            named_arrive(kBarJobFull + rb, kJobThreads);
            ++uses;
            rb ^= 1;
        };
        for (int q = 0; !*(volatile int *)&s_cabort; ++q) {
            const int s = q % a.stages;
            if (!ptx::mbar_wait(&full[s], (q / a.stages) & 1, a.wait_ns)) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                s_cabort = 1;
            }
            consumer_sync();
            if (*(volatile int *)&s_cabort) break;
            const int *tg = tags + kTagWords * s;
            const int kind = tg[0];
            if (kind == kTagEnd) break;
            const uint8_t *st = ring + (size_t)s * a.stage_bytes;
            if (kind == kTagGateUp) {
                const int it = tg[1];
                const int e = rs.act[it / tiles], mt = it % tiles;
                const int seg0 = rs.off[e], seg_n = rs.cnt[e];
                // padded tiles hold row pairs back to back with 16 bytes after each
                // pair: row r at (r / 2) * pp + (r % 2) * row_bytes, so row r + 8 is
                // 4 pairs on, i.e. an effective pitch of pp / 2 for the unit
                const bool paired = a.gu_pitch != a.gu_row;
                const size_t pp = 2 * (size_t)a.gu_pitch - 16;
                const uint32_t gu_step = paired ? (uint32_t)(pp / 2) : (uint32_t)a.gu_pitch;
                const uint8_t *mat = paired ? st + (size_t)wm * (kTileM / 2) * pp + (size_t)(grp >> 1) * pp +
                                                  (size_t)(grp & 1) * a.gu_row
                                            : st + (size_t)wm * kTileM * a.gu_pitch + (size_t)grp * a.gu_pitch;
                for (int c0 = 0; c0 < seg_n; c0 += NT) {
                    const int nt = min(NT, seg_n - c0);
                    uint32_t off[NT];
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        off[j] = (uint32_t)(rs.perm[seg0 + c0 + (j < nt ? j : 0)] / a.k) * a.H;
                    float part[NT][2];
#pragma unroll
                    for (int j = 0; j < NT; ++j) part[j][0] = part[j][1] = 0.0f;
                    if (kSmemOnly || a.x_smem) {
                        const uint32_t mat_s = ptx::smem_addr(mat);
                        for (int kb = wk; kb < a.H_blocks; kb += kKPhases)
                            tile_unit_s<NT>(mat_s + kb * kQ2KBytes, gu_step, wh, grp, c, la_,
                                            inv4c, x_s_a + kb * kQK * 2, xs_s_a + kb * 64, off, nt,
                                            bz0, bz1, part);
                    } else {
                        for (int kb = wk; kb < a.H_blocks; kb += kKPhases)
                            tile_unit<NT, false>(mat + kb * kQ2KBytes, gu_step, wh, grp, c, la_, inv4c,
                                                 a.xp + kb * kQK, a.xs + kb * 16, zero, off, nt, part);
                    }
                    emit(Job{kJobGateUp, e, mt, seg0, c0, nt, it, 0}, part);
                }
            } else {
                const int it = tg[1], j0 = tg[2], cnt = tg[3];
                // The stage's (expert, token chunk) pairs, in rounds of up to
                // kDownPairs.  Inside a round the (pair, K block) units are
                // dealt to the four K-phase warps of each (m-tile, half) in
                // turn, so every warp gets the same number of units; each warp
                // leaves one partial sum per pair, and one barrier per round
                // precedes the reduction into obuf.
                int rj = 0, rc = 0;                  // first pair of the round
                while (rj < cnt) {
                    int np = 0, qj = rj, qc = rc;
                    for (; np < kDownPairs && qj < cnt; ++np) {
                        const int e = rs.act[j0 + qj];
                        const int seg0 = rs.off[e], seg_n = rs.cnt[e];
                        const int nt = min(NT, seg_n - qc);
                        const uint8_t *mat = st + tg[4 + 2 * qj] + (size_t)(wm * kTileM + grp) * a.dn_pitch;
                        const int hoff = tg[5 + 2 * qj];
                        float part[NT][2];
#pragma unroll
                        for (int j = 0; j < NT; ++j) part[j][0] = part[j][1] = 0.0f;
                        const int kb0 = ((wk - np * a.I_blocks) % kKPhases + kKPhases) % kKPhases;
                        if (kSmemOnly || hoff >= 0) {
                            uint32_t off[NT];
#pragma unroll
                            for (int j = 0; j < NT; ++j) off[j] = (uint32_t)(qc + (j < nt ? j : 0)) * a.I_pad;
                            const uint32_t mat_s = ptx::smem_addr(mat);
                            const uint32_t h_a = ptx::smem_addr(st + hoff);
                            const uint32_t hs_a = h_a + (uint32_t)seg_n * h_row;
                            for (int kb = kb0; kb < a.I_blocks; kb += kKPhases)
                                tile_unit_s<NT>(mat_s + kb * kQ2KBytes, (uint32_t)a.dn_pitch, wh, grp, c,
                                                la_, inv4c, h_a + kb * kQK * 2, hs_a + kb * 64, off, nt,
                                                bz0, bz1, part);
                        } else {
                            uint32_t off[NT];
#pragma unroll
                            for (int j = 0; j < NT; ++j)
                                off[j] = (uint32_t)(seg0 + qc + (j < nt ? j : 0)) * a.I_pad;
                            for (int kb = kb0; kb < a.I_blocks; kb += kKPhases)
                                tile_unit<NT, false>(mat + kb * kQ2KBytes, a.dn_pitch, wh, grp, c, la_, inv4c,
                                                     a.hp + kb * kQK, a.hs + kb * 16, zero, off, nt, part);
                        }
                        store_partials<NT>(redd + (size_t)np * kConsumers * NT * kTileM, warp, grp, c, part);
                        qc += NT;
                        if (qc >= seg_n) { ++qj; qc = 0; }
                    }
                    consumer_sync();
                    // the down partial sums are finished here, by the consumers:
                    // thread i -> pair i / (NT * 32), vector, row
                    for (int i = tid; i < np * NT * kDownRows; i += kConsumers * 32) {
                        const int pq = i / (NT * kDownRows), rem = i % (NT * kDownRows);
                        const int j = rem / kDownRows, row = rem % kDownRows;
                        int pj = rj, pc = rc;                  // walk to pair pq
                        for (int w = 0; w < pq; ++w) {
                            pc += NT;
                            if (pc >= rs.cnt[rs.act[j0 + pj]]) { ++pj; pc = 0; }
                        }
                        const int e = rs.act[j0 + pj];
                        if (pc + j < rs.cnt[e]) {
                            const int mtl = row >> 4, r16 = row & 15;
                            const float *rbuf = redd + (size_t)pq * kConsumers * NT * kTileM;
                            // warps with (warp >> 1) & 1 == mtl hold rows mtl*16 .. +15
                            float o = 0.0f;
#pragma unroll
                            for (int w = 0; w < kConsumers; ++w)
                                if (((w >> 1) & 1) == mtl) o += rbuf[((size_t)w * NT + j) * kTileM + r16];
                            obuf[(size_t)(rs.off[e] + pc + j) * kDownRows + row] = o;
                        }
                    }
                    rj = qj;
                    rc = qc;
                    if (rj < cnt) consumer_sync();       // redd is reused by the next round
                }
                if (j0 + cnt == n_act) {
                    // every expert of this item is in obuf: weighted combine in slot order
                    consumer_sync();
                    for (int i = tid; i < a.T * kDownRows; i += kConsumers * 32) {
                        const int t = i / kDownRows, row = i % kDownRows;
                        float acc = 0.0f;
                        for (int sl = 0; sl < a.k; ++sl) {
                            const int asg = t * a.k + sl;
                            acc += rs.wts[asg] * obuf[(size_t)rs.slot[asg] * kDownRows + row];
                        }
                        a.y[(size_t)t * a.H + (size_t)it * kDownRows + row] =
                            acc * exp2i(2 * s_e[t] + kHExpOffset);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty[s]);
            if (tid == 0) s_consumed = q + 1;
        }
        // tell the epilogue warp to stop
        {
            int &uses = rb ? uses1 : uses0;
            if (uses > 0) named_sync(kBarJobEmpty + rb, kJobThreads);
            if (tid == 0) jobs[rb].kind = kJobStop;
            named_arrive(kBarJobFull + rb, kJobThreads);
        }
    } else {
        // ---------------- epilogue warp ----------------
        for (int rb = 0;; rb ^= 1) {
            named_sync(kBarJobFull + rb, kJobThreads);
            const Job jb = jobs[rb];
            if (jb.kind == kJobStop) break;
            const float *rbuf = red + rb * kConsumers * NT * kTileM;
            if (jb.kind == kJobGateUp) {
                const int tiles_e = tiles;
                for (int base = 0; base < jb.nt * kTileM; base += 32) {
                    const int i = base + lane;
                    const bool valid = i < jb.nt * kTileM;
                    const int row = i & 15, j = valid ? i >> 4 : 0;
                    float g = 0.0f, uu = 0.0f;
                    // warps with (warp >> 1) & 1 == 0 hold gate, the others up
#pragma unroll
                    for (int w = 0; w < kConsumers; ++w) {
                        const float v = rbuf[((size_t)w * NT + j) * kTileM + row];
                        if ((w >> 1) & 1) uu += v; else g += v;
                    }
                    const int pos = jb.seg0 + jb.c0 + j;
                    // undo the token's activation scale; h leaves scaled by 2^-f
                    const int e = s_e[rs.perm[pos] / a.k];
                    const float sx = exp2i(e);
                    const __half hv = __float2half_rn(silu_mul(g * sx, uu * sx) *
                                                      exp2i(-(2 * e + kHExpOffset)));
                    const int n = jb.mt * kTileM + row;
                    float hsum = valid ? __half2float(hv) : 0.0f;
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) hsum += __shfl_xor_sync(0xffffffffu, hsum, o);
                    if (valid) {
                        a.hp[(size_t)pos * a.I_pad + perm4(n)] = hv;
                        if (row == 0) a.hs[(size_t)pos * (a.I_pad / 16) + jb.mt] = hsum;
                        // rows inter .. I_pad-1 of h (the down projection's padded K) are 0
                        if (jb.mt == tiles_e - 1)
                            for (int n2 = a.I + row; n2 < a.I_pad; n2 += kTileM) {
                                a.hp[(size_t)pos * a.I_pad + n2] = __float2half_rn(0.0f);
                                if ((n2 & 15) == 0) a.hs[(size_t)pos * (a.I_pad / 16) + n2 / 16] = 0.0f;
                            }
                    }
                }
                // publish: every value of h counts once toward its expert's total
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(done + jb.e, jb.nt * kTileM);
            }
            named_arrive(kBarJobEmpty + rb, kJobThreads);
        }
    }
    __syncthreads();
    // after an abort: the copies this CTA issued land before it exits
    if (tid == kProducerWarp * 32 && (s_pabort || s_cabort)) {
        for (int q = s_consumed; q < s_issued; ++q) {
            const int s = q % a.stages;
            if (!ptx::mbar_wait(&full[s], (q / a.stages) & 1, a.wait_ns)) break;
        }
    }
}

// ===========================================================================
// tcgen05 decode kernel (decode_tc_kernel)
//
// The block-diagonal trick of the mma.sync kernel above, on the 5th
// generation tensor core, for 9..32 tokens (where the mma.sync kernel's
// 8-column operand would be re-run per chunk of tokens).  Per 128-row tile
// and 256-wide K block: the dequantizing warps store the raw fields
// (1024 + q * 4^g, exact fp16, lop3 only) of their row to tensor memory as
// the MMA's A operand; B, in shared memory, is block-diagonal over the 16
// sub-blocks: row (t, s) of B holds activation vector t only in the 16
// k-slots of sub-block s.  D (tensor memory, fp32) then holds per row one
// value per (vector, sub-block), and the same warps apply
//   w . x = sum_s d*sc_s*4^-g (D_s - 1024*X_s) - dmin*m_s*X_s
// in a short per-block epilogue.  The tensor core does the 16-term sums, so
// the CUDA cores spend about one instruction per weight.
//
// Work items, claimed from global counters by the producer warp:
//   gate/up  (token chunk of <= 4 vectors of one expert, 128 rows of I,
//             K half when the layer is small): both matrices, h = SiLU(g)*u;
//             the CTA that finishes the second K half of a tile combines the
//             halves;
//   down     (token chunk, 128 rows of H): y_slot[p, m] = w_p * o; the CTA
//             that completes the last chunk of an m-tile combines y in slot
//             order.
// A down item waits (bounded) until its expert's h is complete.  Warps: 0 TMA
// producer (3-D tensor maps over 112-byte block windows; rows that are not a
// multiple of 16 bytes use several row phases), 1 MMA issuer, 2..9 two
// dequantizing warpgroups that are also the epilogue, which lags the MMAs by
// one K block.
// ===========================================================================
namespace tcd {

constexpr int kBM = 128;
constexpr int kNtMax = 4;                 // activation vectors per item
constexpr int kWinBytes = 112;            // 16-byte aligned window of one block row
constexpr int kAq = kWinBytes * kBM;      // one matrix's windows of 128 rows
constexpr int kChunk = 16 * kNtMax * 128; // one 64-wide K chunk of the diagonal operand
constexpr int kBDiag = 4 * kChunk;
constexpr int kOffB = 2 * kAq;            // 28672, 1024-aligned
constexpr int kOffXc = kOffB + kBDiag;    // compact fp16 activations of the block
constexpr int kOffXs = kOffXc + kNtMax * 512;   // their sub-block sums
constexpr uint32_t kStage = 64 * 1024;
constexpr int kStages = 3;
constexpr int kDq = 8;                    // dequantizing warps (two warpgroups)
constexpr int kThreads = (2 + kDq) * 32;
constexpr uint32_t kTmemCols = 512, kDCol = 256;
constexpr int kMaxPairs = 1024;           // K-split tile pairs
constexpr int kBarWG = 1, kBarWG0 = 2;    // named barriers: both warpgroups / warpgroup 0

enum { kItemGateUp = 0, kItemDown = 1, kItemEnd = 2 };

struct Args {
    int H, I, I_pad, E, k, T, A, score;
    int H_blocks, I_blocks;
    int P_gu, P_dn;                 // row phases of the weight windows
    int64_t gu_row, dn_row;
    const int32_t *wslot;   // [E] weight slot of each expert, or null
    int n_wslots;
    int ks;                         // K split of gate/up tiles (1 or 2)
    const float *logits;
    const uint16_t *x;
    const __half *xp;               // [T][H] fp16 (4-group permuted)
    const float *xs;                // [T][H/16]
    const int32_t *texp;            // [T] token exponents (decode_pre_kernel)
    __half *hp;                     // [A][I_pad]
    float *hs;                      // [A][I_pad/16]
    float *yslot;                   // [A][H]
    float *gpart;                   // [pairs][2 halves][2 matrices][kNtMax][128]
    float *y;
    int32_t *ids, *counts, *offsets, *perm;
    float *wts;
    int32_t *status;
    int32_t *sync;                  // [0] gate/up claim, [1] down claim, [4 + e] h done,
                                    // [4 + E + mt] y tiles done, [4 + E + H/128 + i] pair halves
    uint64_t wait_ns;
    int stall;
};

struct Chunk {
    int e, pos0, nt;
};

// Raw fields of half HALF of the block at word SH of `win`: 64 packed fp16
// pairs (1024 + q * 4^g), stored to tensor memory at taddr.
template <int SH, int HALF>
__device__ __forceinline__ void raw_store(const uint32_t (&win)[24], uint32_t taddr)
{
    const uint32_t *w = win + SH;
    uint32_t out[64];
#pragma unroll
    for (int wd = 0; wd < 8; ++wd) {
        const uint32_t qw = w[4 + 8 * HALF + wd], qh = qw >> 8;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint32_t mask = 0x00030003u << (2 * g);
            out[16 * g + 2 * wd] = ptx::lop3_and_or(qw, mask, 0x64006400u);
            out[16 * g + 2 * wd + 1] = ptx::lop3_and_or(qh, mask, 0x64006400u);
        }
    }
    ptx::tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(&out[0]));
    ptx::tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&out[32]));
}

__device__ __forceinline__ void raw_store_sh(const uint32_t (&win)[24], int sh, int half,
                                             uint32_t taddr)
{
    switch (sh * 2 + half) {
    case 0: raw_store<0, 0>(win, taddr); break;
    case 1: raw_store<0, 1>(win, taddr); break;
    case 2: raw_store<1, 0>(win, taddr); break;
    case 3: raw_store<1, 1>(win, taddr); break;
    case 4: raw_store<2, 0>(win, taddr); break;
    case 5: raw_store<2, 1>(win, taddr); break;
    case 6: raw_store<3, 0>(win, taddr); break;
    default: raw_store<3, 1>(win, taddr); break;
    }
}

// The 5 words of the block that the epilogue needs (scales 0..3, d|dmin).
__device__ __forceinline__ void keep_scales(const uint32_t (&win)[24], int sh, uint32_t (&sc)[5])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v = win[i];
        v = sh == 1 ? win[i + 1] : v;
        v = sh == 2 ? win[i + 2] : v;
        v = sh == 3 ? win[i + 3] : v;
        sc[i] = v;
    }
    uint32_t v = win[20];
    v = sh == 1 ? win[21] : v;
    v = sh == 2 ? win[22] : v;
    v = sh == 3 ? win[23] : v;
    sc[4] = v;
}

// Adds sub-blocks s0 .. s0+NS-1 of one 256-wide block to acc[t], t < nt:
// D from tensor memory (columns 16t + s), sums X from shared memory.
template <int NS>
__device__ __forceinline__ void block_epilogue(uint32_t dcol, int s0, const uint32_t (&sc)[5],
                                               const float2 *lut, const float *xsum, int nt,
                                               float (&acc)[kNtMax])
{
    const float d = half_bits(sc[4] & 0xFFFFu), dmin = half_bits(sc[4] >> 16);
    float cA[NS], cX[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        const int s = s0 + i;
        const uint32_t b = (sc[s >> 2] >> (8 * (s & 3))) & 0xFFu;
        const float2 f = lut[b];
        const int g = (s & 7) >> 1;
        cA[i] = d * f.x * (g == 0 ? 1.0f : g == 1 ? 0.25f : g == 2 ? 0.0625f : 0.015625f);
        cX[i] = -fmaf(1024.0f, cA[i], dmin * f.y);
    }
#pragma unroll
    for (int t = 0; t < kNtMax; ++t) {
        if (t < nt) {
            float v[16];
            if (NS == 16) {
                ptx::tmem_ld16(dcol + 16 * t, v);
            } else {
                float v8[8];
                ptx::tmem_ld8(dcol + 16 * t + s0, v8);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = v8[i];
            }
            ptx::tmem_ld_wait();
            float a = acc[t];
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                a = fmaf(cA[i], v[i], a);
                a = fmaf(cX[i], xsum[16 * t + s0 + i], a);
            }
            acc[t] = a;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_gate,
                     const __grid_constant__ CUtensorMap tm_up,
                     const __grid_constant__ CUtensorMap tm_down, const Args a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    __shared__ RouteSmem rs;
    __shared__ int32_t s_e[kDecodeMaxT];     // token exponents
    __shared__ Chunk chunks[kMaxAssign];
    __shared__ int s_nchunks;
    __shared__ __align__(8) float2 sc_lut[256];
    __shared__ float xch[kNtMax][kBM];        // warpgroup 1 -> warpgroup 0 hand-off
    __shared__ float hsm[kNtMax][kBM];        // h of the tile (for the sub-block sums)
    __shared__ int tags[kStages][2];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], afull[2], aempty[2];
    __shared__ __align__(8) uint64_t dfull[2], dempty[2], drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_issued, s_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort_flag = &s_abort;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kDq);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&afull[b], kDq);
            ptx::mbar_init(&aempty[b], 1);
            ptx::mbar_init(&dfull[b], 1);
            ptx::mbar_init(&dempty[b], kDq);
        }
        ptx::mbar_init(&drain, 1);
        ptx::fence_mbar_init();
        s_abort = 0;
        s_issued = 0;
    }
    if (tid < 256) sc_lut[tid] = make_float2((float)(tid & 15), (float)(tid >> 4));
    // zero the diagonal operand of every stage once; items only rewrite the
    // diagonal entries
    for (int i = tid; i < kStages * kBDiag / 16; i += blockDim.x) {
        const int s = i / (kBDiag / 16), o = i % (kBDiag / 16);
        reinterpret_cast<uint4 *>(smem + (size_t)s * kStage + kOffB)[o] = make_uint4(0, 0, 0, 0);
    }
    if (warp == 1) {
        ptx::tmem_alloc(&s_tmem, kTmemCols);
        ptx::tmem_relinquish();
    }
    // routing: one warp for small batches, the whole CTA otherwise
    DecArgs ra{};
    ra.E = a.E; ra.k = a.k; ra.T = a.T; ra.A = a.A; ra.score = a.score; ra.logits = a.logits;
    ra.ids = a.ids; ra.wts = a.wts; ra.counts = a.counts; ra.offsets = a.offsets; ra.perm = a.perm;
    __syncthreads();
    if (a.T <= kWarpRouteT && a.A <= 32) {
        if (warp == 0) route_warp(ra, rs);
        __syncthreads();
    } else {
        route_into_smem(ra, rs);
    }
    if (warp == 0) {
        // token chunks of <= kNtMax vectors per active expert
        int run = 0;
        for (int j0 = 0; j0 < rs.n_act; j0 += 32) {
            const int j = j0 + lane;
            const int e = j < rs.n_act ? rs.act[j] : 0;
            const int n = j < rs.n_act ? (rs.cnt[e] + kNtMax - 1) / kNtMax : 0;
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            for (int c = 0; c < n; ++c) {
                Chunk ch;
                ch.e = e;
                ch.pos0 = rs.off[e] + c * kNtMax;
                ch.nt = min(kNtMax, rs.cnt[e] - c * kNtMax);
                chunks[run + incl - n + c] = ch;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_nchunks = run;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::grid_dep_wait();        // counters reset, activations converted, exponents written
    if (threadIdx.x < a.T) s_e[threadIdx.x] = a.texp[threadIdx.x];
    __syncthreads();
    const uint32_t tmem = s_tmem;

    const int n_chunks = s_nchunks;
    const int mt_gu = a.I_pad / kBM, mt_dn = a.H / kBM;
    const int n_gu = n_chunks * mt_gu * a.ks, n_dn = n_chunks * mt_dn;
    const int kb_gu = a.H_blocks / a.ks, kb_dn = a.I_blocks;
    int32_t *const claim_gu = a.sync, *const claim_dn = a.sync + 1, *const done = a.sync + 4;
    int32_t *const tiles_done = a.sync + 4 + a.E, *const pairs = tiles_done + mt_dn;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0 && !a.stall) {
            ptx::prefetch_tmap(&tm_gate);
            ptx::prefetch_tmap(&tm_up);
            ptx::prefetch_tmap(&tm_down);
            int sc = 0;
            bool ok = true;
            auto slot = [&](int &s) -> bool {
                s = sc % kStages;
                if (sc >= kStages &&
                    !ptx::mbar_wait_or_abort(&empty[s], ((sc / kStages) - 1) & 1, a.wait_ns,
                                             abort_flag)) {
                    set_status(a.status, DS4G_ERR_TIMEOUT);
                    *abort_flag = 1;
                    return false;
                }
                return true;
            };
            for (int phase = 0; ok && phase < 2; ++phase) {
                while (ok) {
                    const int it = atomicAdd(phase == 0 ? claim_gu : claim_dn, 1);
                    if (it >= (phase == 0 ? n_gu : n_dn)) break;
                    int ch, mt, kh = 0;
                    if (phase == 0) {
                        ch = it / (mt_gu * a.ks);
                        const int rem = it % (mt_gu * a.ks);
                        mt = rem / a.ks;
                        kh = rem % a.ks;
                    } else {
                        ch = it / mt_dn;
                        mt = it % mt_dn;
                    }
                    const Chunk c = chunks[ch];
                    if (phase == 1) {
                        if (!wait_counter(done + c.e, a.I_pad * rs.cnt[c.e], a.wait_ns)) {
                            set_status(a.status, DS4G_ERR_TIMEOUT);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        // h was written by other CTAs (generic proxy); the
                        // copies below read it through the async proxy
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                    const int P = phase == 0 ? a.P_gu : a.P_dn;
                    const int64_t row = phase == 0 ? a.gu_row : a.dn_row;
                    const int nkb = phase == 0 ? kb_gu : kb_dn;
                    const int nmat = phase == 0 ? 2 : 1;
                    const int we = weight_slot(a.wslot, a.n_wslots, c.e, a.status);
                    const uint32_t bytes = (uint32_t)(nmat * kAq + c.nt * (512 + 64));
                    for (int j = 0; ok && j < nkb; ++j, ++sc) {
                        const int kb = kh * nkb + j;
                        int s;
                        if (!(ok = slot(s))) break;
                        tags[s][0] = phase;
                        tags[s][1] = it;
                        uint8_t *st = smem + (size_t)s * kStage;
                        ptx::mbar_arrive_expect_tx(&full[s], bytes);
                        for (int p = 0; p < P; ++p) {
                            const int xw = (int)(((p * row + kQ2KBytes * kb) & ~15ll) / 4);
                            uint8_t *dst = st + p * (kBM / P) * kWinBytes;
                            if (phase == 0) {
                                ptx::tma_load_3d(dst, &tm_gate, xw, mt * (kBM / P), we, &full[s]);
                                ptx::tma_load_3d(dst + kAq, &tm_up, xw, mt * (kBM / P), we, &full[s]);
                            } else {
                                ptx::tma_load_3d(dst, &tm_down, xw, mt * (kBM / P), we, &full[s]);
                            }
                        }
                        for (int t = 0; t < c.nt; ++t) {
                            const __half *src;
                            const float *ssrc;
                            if (phase == 0) {
                                const int tok = rs.perm[c.pos0 + t] / a.k;
                                src = a.xp + (size_t)tok * a.H + (size_t)kb * kQK;
                                ssrc = a.xs + (size_t)tok * (a.H / 16) + (size_t)kb * 16;
                            } else {
                                const int pos = c.pos0 + t;
                                src = a.hp + (size_t)pos * a.I_pad + (size_t)kb * kQK;
                                ssrc = a.hs + (size_t)pos * (a.I_pad / 16) + (size_t)kb * 16;
                            }
                            ptx::bulk_g2s(st + kOffXc + t * 512, src, 512, &full[s]);
                            ptx::bulk_g2s(st + kOffXs + t * 64, ssrc, 64, &full[s]);
                        }
                        s_issued = sc + 1;
                    }
                }
            }
            int s;
            if (ok && slot(s)) {
                tags[s][0] = kItemEnd;
                ptx::mbar_arrive(&full[s]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int sc = 0, fc = 0, dc = 0;
            bool ok = true;
            while (ok) {
                const int s = sc % kStages;
                if (!ptx::mbar_wait_or_abort(&full[s], (sc / kStages) & 1, a.wait_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                const int kind = tags[s][0];
                if (kind == kItemEnd) break;
                const int it = tags[s][1];
                const Chunk c = chunks[kind == kItemGateUp ? it / (mt_gu * a.ks) : it / mt_dn];
                const uint32_t idesc = ptx::idesc_f16(kBM, 16 * c.nt);
                const int db = dc & 1;
                if (dc >= 2 && !ptx::mbar_wait_or_abort(&dempty[db], ((dc >> 1) - 1) & 1, a.wait_ns,
                                                        abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t b_base = ptx::smem_addr(smem + (size_t)s * kStage + kOffB);
                const uint32_t dcol = tmem + kDCol + 128u * db;
                const int fills = kind == kItemGateUp ? 2 : 1;
                for (int h = 0; ok && h < fills; ++h, ++fc) {
                    const int fb = fc & 1;
                    if (!ptx::mbar_wait_or_abort(&afull[fb], (fc >> 1) & 1, a.wait_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t abuf = tmem + 128u * fb;
                    if (kind == kItemGateUp) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int kk = 128 * h + 16 * i;
                            const uint64_t bd =
                                ptx::sw128_desc(b_base + (kk >> 6) * kChunk + (kk & 63) * 2);
                            const bool acc = !(h == 0 && i == 0);
                            ptx::mma_f16_ts(dcol, abuf + 8 * i, bd, idesc, acc);
                            ptx::mma_f16_ts(dcol + 64, abuf + 64 + 8 * i, bd, idesc, acc);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int kk = 16 * i;
                            const uint64_t bd =
                                ptx::sw128_desc(b_base + (kk >> 6) * kChunk + (kk & 63) * 2);
                            ptx::mma_f16_ts(dcol, abuf + 8 * i, bd, idesc, i > 0);
                        }
                    }
                    ptx::mma_commit(&aempty[fb]);
                }
                if (!ok) break;
                ptx::mma_commit(&dfull[db]);
                ++dc;
                ++sc;
            }
            if (!ok) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            ptx::mma_commit(&drain);
            ptx::mbar_wait(&drain, 0, a.wait_ns);
        }
    } else {
        // ---------------- dequantizers / epilogue ----------------
        const int wg = (warp - 2) >> 2;                 // 0: gate (or K half 0), 1: up (half 1)
        const int ell = 32 * (warp & 3) + lane;         // tensor-memory lane = A row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int wtid = tid - 64 - 128 * wg;            // 0..127 inside the warpgroup
        uint32_t dfull_phase[2] = {0, 0};
        int sc = 0, fc = 0, dc = 0;
        float acc[kNtMax];
        // the epilogue of one block: its D buffer, scales and stage (the
        // stage still holds the block's activation sums)
        uint32_t pscw[5] = {0, 0, 0, 0, 0};
        int pss = 0, pdb = 0;
        auto block_done = [&](bool gu_, const uint32_t (&sc5)[5], int stg, int db, int nt,
                              float (&ac)[kNtMax]) {
            if (!ptx::mbar_wait_or_abort(&dfull[db], dfull_phase[db], a.wait_ns, abort_flag)) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            dfull_phase[db] ^= 1;
            ptx::tc_fence_after();
            const float *xsum = reinterpret_cast<const float *>(smem + (size_t)stg * kStage + kOffXs);
            const uint32_t dcol = tmem + lane_base + kDCol + 128u * db;
            if (gu_)
                block_epilogue<16>(dcol + 64u * wg, 0, sc5, sc_lut, xsum, nt, ac);
            else
                block_epilogue<8>(dcol, 8 * wg, sc5, sc_lut, xsum, nt, ac);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&dempty[db]);
                ptx::mbar_arrive(&empty[stg]);
            }
        };
        while (true) {
            const int s = sc % kStages;
            if (!ptx::mbar_wait_or_abort(&full[s], (sc / kStages) & 1, a.wait_ns, abort_flag)) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every abort decision is taken here, by both warpgroups alike
            named_sync(kBarWG, kDq * 32);
            if (*abort_flag) break;
            const int kind = tags[s][0];
            if (kind == kItemEnd) break;
            const int it = tags[s][1];
            const bool gu = kind == kItemGateUp;
            int ch, mt, kh = 0;
            if (gu) {
                ch = it / (mt_gu * a.ks);
                const int rem = it % (mt_gu * a.ks);
                mt = rem / a.ks;
                kh = rem % a.ks;
            } else {
                ch = it / mt_dn;
                mt = it % mt_dn;
            }
            const Chunk c = chunks[ch];
            const int P = gu ? a.P_gu : a.P_dn;
            const int64_t row = gu ? a.gu_row : a.dn_row;
            const int nkb = gu ? kb_gu : kb_dn;
            const int p = ell / (kBM / P);                 // row phase of this lane
            const int wrow = (ell % (kBM / P)) * P + p;    // weight row inside the tile
#pragma unroll
            for (int t = 0; t < kNtMax; ++t) acc[t] = 0.0f;
            for (int j = 0; j < nkb; ++j, ++sc) {
                const int ss = sc % kStages;
                if (j > 0) {
                    if (!ptx::mbar_wait_or_abort(&full[ss], (sc / kStages) & 1, a.wait_ns, abort_flag)) {
                        set_status(a.status, DS4G_ERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                }
                const int kb = kh * nkb + j;
                uint8_t *st = smem + (size_t)ss * kStage;
                // warpgroup 0 scatters the block's activations onto the diagonal
                if (wg == 0) {
                    const uint32_t bb = ptx::smem_addr(st + kOffB), xc = ptx::smem_addr(st + kOffXc);
                    const int kk = 2 * wtid, sb = kk >> 4, ck = kk >> 6, u = (kk & 63) >> 3;
                    for (int t = 0; t < c.nt; ++t) {
                        const int r = 16 * t + sb;
                        const uint32_t v = ptx::ld_s32(xc + t * 512 + 4 * wtid);
                        ptx::sts32(bb + ck * kChunk + r * 128 + ((u ^ (r & 7)) << 4) + (kk & 7) * 2, v);
                    }
                    ptx::fence_proxy_async_smem();
                }
                // this lane's 112-byte window of its matrix
                const uint8_t *wn = st + (gu ? wg * kAq : 0) + ell * kWinBytes;
                uint32_t win[24];
#pragma unroll
                for (int v = 0; v < 6; ++v) {
                    const uint4 q = reinterpret_cast<const uint4 *>(wn)[v];
                    win[4 * v] = q.x; win[4 * v + 1] = q.y; win[4 * v + 2] = q.z; win[4 * v + 3] = q.w;
                }
                const int sh = (int)(((p * row + kQ2KBytes * kb) & 15) >> 2);
                uint32_t scw[5];
                keep_scales(win, sh, scw);
                const int fills = gu ? 2 : 1;
                for (int h = 0; h < fills; ++h, ++fc) {
                    const int fb = fc & 1;
                    if (fc >= 2 &&
                        !ptx::mbar_wait_or_abort(&aempty[fb], ((fc >> 1) - 1) & 1, a.wait_ns, abort_flag)) {
                        set_status(a.status, DS4G_ERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ptx::tc_fence_after();
                    const int half = gu ? h : wg;
                    raw_store_sh(win, sh, half, tmem + lane_base + 128u * fb + 64u * wg);
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&afull[fb]);
                }
                // epilogue of the previous block, while the tensor core works on this one
                if (j > 0) block_done(gu, pscw, pss, pdb, c.nt, acc);
#pragma unroll
                for (int i = 0; i < 5; ++i) pscw[i] = scw[i];
                pss = ss;
                pdb = dc & 1;
                ++dc;
            }
            block_done(gu, pscw, pss, pdb, c.nt, acc);
            // ---- item epilogue ----
            if (gu) {
                const int pair = ch * mt_gu + mt;
                bool have = true;
                if (a.ks == 2) {
                    // both warpgroups park their half-K partial sums; the
                    // second half to finish combines them (fixed order)
                    float *gp = a.gpart + ((size_t)(pair * 2 + kh) * 2 + wg) * kNtMax * kBM;
                    for (int t = 0; t < c.nt; ++t) gp[t * kBM + wrow] = acc[t];
                    __threadfence();
                    named_sync(kBarWG, kDq * 32);
                    if (wtid == 0 && wg == 0) s_flag = atomicAdd(pairs + pair, 1);
                    named_sync(kBarWG, kDq * 32);
                    have = s_flag == 1;
                    if (have) {
                        __threadfence();
                        const float *g0 = a.gpart + ((size_t)(pair * 2 + 0) * 2 + wg) * kNtMax * kBM;
                        const float *g1 = a.gpart + ((size_t)(pair * 2 + 1) * 2 + wg) * kNtMax * kBM;
                        for (int t = 0; t < c.nt; ++t)
                            acc[t] = __ldcg(g0 + t * kBM + wrow) + __ldcg(g1 + t * kBM + wrow);
                    }
                }
                if (have) {
                    if (wg == 1)
                        for (int t = 0; t < c.nt; ++t) xch[t][wrow] = acc[t];
                    named_sync(kBarWG, kDq * 32);
                    if (wg == 0) {
                        const int n = mt * kBM + wrow;
                        for (int t = 0; t < c.nt; ++t) {
                            // undo the token's activation scale; h leaves scaled by 2^-f
                            const int e = s_e[rs.perm[c.pos0 + t] / a.k];
                            const float sx = exp2i(e);
                            const __half hv = __float2half_rn(
                                silu_mul(acc[t] * sx, xch[t][wrow] * sx) * exp2i(-(2 * e + kHExpOffset)));
                            a.hp[(size_t)(c.pos0 + t) * a.I_pad + perm4(n)] = hv;
                            hsm[t][wrow] = __half2float(hv);
                        }
                        named_sync(kBarWG0, 128);
                        if (wtid < 8 * c.nt) {
                            const int t = wtid >> 3, sb = wtid & 7;
                            float sum = 0.0f;
                            for (int r = 0; r < 16; ++r) sum += hsm[t][16 * sb + r];
                            a.hs[(size_t)(c.pos0 + t) * (a.I_pad / 16) + mt * 8 + sb] = sum;
                        }
                        // publish: h and its sums of this tile are visible
                        __threadfence();
                        named_sync(kBarWG0, 128);
                        if (wtid == 0) atomicAdd(done + c.e, kBM * c.nt);
                    }
                }
            } else {
                if (wg == 1)
                    for (int t = 0; t < c.nt; ++t) xch[t][wrow] = acc[t];
                named_sync(kBarWG, kDq * 32);
                if (wg == 0) {
                    const int m = mt * kBM + wrow;
                    for (int t = 0; t < c.nt; ++t) {
                        const int pos = c.pos0 + t;
                        const float sh = exp2i(2 * s_e[rs.perm[pos] / a.k] + kHExpOffset);
                        a.yslot[(size_t)pos * a.H + m] =
                            rs.wts[rs.perm[pos]] * ((acc[t] + xch[t][wrow]) * sh);
                    }
                    __threadfence();
                    named_sync(kBarWG0, 128);
                    if (wtid == 0) s_flag = atomicAdd(tiles_done + mt, c.nt) + c.nt == a.A;
                }
                named_sync(kBarWG, kDq * 32);
                if (s_flag) {
                    // every assignment of these rows is in y_slot: combine in slot order
                    __threadfence();
                    const int i0 = wg * 128 + wtid;
                    for (int i = i0; i < a.T * kBM; i += 256) {
                        const int t = i / kBM, m = mt * kBM + i % kBM;
                        float yv = 0.0f;
                        for (int sl = 0; sl < a.k; ++sl)
                            yv += __ldcg(a.yslot + (size_t)rs.slot[t * a.k + sl] * a.H + m);
                        a.y[(size_t)t * a.H + m] = yv;
                    }
                }
                named_sync(kBarWG, kDq * 32);
            }
        }
    }

    __syncthreads();
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

}  // namespace tcd


// Row pitch of a weight tile in shared memory.  Lane groups read rows grp
// and grp+8 (grp = 0..7) at the same column: a pitch of a multiple of 32
// bytes would put several groups on one bank, so such rows get 16 bytes of
// padding (copied row by row; only possible for rows of a multiple of 16
// bytes, the others are copied whole).
int64_t smem_pitch(int64_t row_bytes)
{
    if (row_bytes % 16 == 0 && (row_bytes / 4) % 8 == 0) return row_bytes + 16;
    return row_bytes;
}

size_t fixed_smem(const DecArgs &a, int nt)
{
    const size_t x = a.x_smem ? (size_t)a.T * a.H * 2 + (size_t)a.T * (a.H / 16) * 4 : 0;
    return x + (size_t)(2 + kDownPairs) * kConsumers * nt * kTileM * 4 + (size_t)a.A * kDownRows * 4 +
           4 * (size_t)kTagWords * a.stages + 8 * (2 * (size_t)a.stages);
}

template <int NT>
cudaError_t launch_nt(DecArgs a, const DeviceInfo &dev, cudaStream_t s, const cudaEvent_t *ev)
{
    const size_t gu = (size_t)2 * kTileM * a.gu_pitch, dn = (size_t)kDownRows * a.dn_pitch;
    a.stage_bytes = (uint32_t)((std::max(gu, dn) + 127) / 128 * 128);
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_q2k_kernel<NT>);
    if (e != cudaSuccess) return e;
    const size_t budget = std::min(kSmemBudget, (size_t)dev.max_smem_optin - fa.sharedSizeBytes - 256);
    a.stages = 8;
    while (a.stages > 2 && (size_t)a.stages * a.stage_bytes + fixed_smem(a, NT) > budget) --a.stages;
    if ((size_t)a.stages * a.stage_bytes + fixed_smem(a, NT) > budget) return cudaErrorInvalidValue;
    const size_t smem = (size_t)a.stages * a.stage_bytes + fixed_smem(a, NT);
    e = cudaFuncSetAttribute(decode_q2k_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(dev.sm_count);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_q2k_kernel<NT>, a);
    if (e != cudaSuccess) return e;
    // one kernel covers the whole layer: the gate/up, down and combine marks coincide
    if (ev) {
        for (int i = 2; i <= 4; ++i)
            if ((e = record_phase(ev[i], s)) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

// Row phases that make a super-row a multiple of 16 bytes.
int row_phases(int64_t row_bytes)
{
    int64_t g = 16;
    while (row_bytes % g) g >>= 1;
    return (int)(16 / g);
}

cudaError_t launch_decode_tc(const LayerArgs &la, const DecodeBufs &db, const DeviceInfo &dev,
                             cudaStream_t s, const cudaEvent_t *events, uint64_t wait_ns, bool stall)
{
    tcd::Args a{};
    a.H = la.H;
    a.I = la.I;
    a.I_pad = la.I_pad;
    a.E = la.E;
    a.k = la.k;
    a.T = la.T;
    a.A = la.A;
    a.score = db.score;
    a.H_blocks = la.H / kQK;
    a.I_blocks = la.I_pad / kQK;
    a.P_gu = row_phases(la.gu_row);
    a.P_dn = row_phases(la.dn_row);
    a.gu_row = la.gu_row;
    a.dn_row = la.dn_row;
    // split the gate/up tiles over K when there are too few of them to
    // occupy every SM (single-token decode)
    const int mt_gu = la.I_pad / tcd::kBM;
    const int est_chunks = std::min(la.A, la.E);
    a.ks = (est_chunks * mt_gu < 2 * dev.sm_count && a.H_blocks % 2 == 0 &&
            la.A * mt_gu <= tcd::kMaxPairs)
               ? 2
               : 1;
    a.logits = db.logits;
    a.x = la.x;
    a.xp = db.xp;
    a.xs = db.xs;
    a.texp = db.texp;
    a.hp = db.hp;
    a.hs = db.hs;
    a.yslot = la.yslot;
    a.gpart = db.gpart;
    a.y = la.y;
    a.ids = db.ids;
    a.wts = const_cast<float *>(la.wts);
    a.counts = const_cast<int32_t *>(la.counts);
    a.offsets = const_cast<int32_t *>(la.offsets);
    a.perm = const_cast<int32_t *>(la.perm);
    a.status = db.status;
    a.sync = db.sync;
    a.wait_ns = wait_ns;
    a.stall = stall ? 1 : 0;
    a.wslot = la.wslot;
    a.n_wslots = la.n_wslots;

    CUtensorMap m_gate, m_up, m_down;
    cudaError_t e;
    if ((e = weight_map(&m_gate, la.w_gate, la.gu_row, la.I, la.gu_stride, la.n_wslots, a.P_gu)) != cudaSuccess ||
        (e = weight_map(&m_up, la.w_up, la.gu_row, la.I, la.gu_stride, la.n_wslots, a.P_gu)) != cudaSuccess ||
        (e = weight_map(&m_down, la.w_down, la.dn_row, la.H, la.dn_stride, la.n_wslots, a.P_dn)) != cudaSuccess)
        return e;

    // counters and status reset, activations to fp16 (the kernel copies them
    // into its pipeline by TMA)
    decode_pre_kernel<<<a.T, 256, 0, s>>>(db.status, db.sync, decode_sync_words(la.E, la.H), la.x,
                                          const_cast<__half *>(db.xp), const_cast<float *>(db.xs),
                                          a.T, a.H, db.texp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (events && (e = record_phase(events[1], s)) != cudaSuccess) return e;

    const size_t smem = (size_t)tcd::kStages * tcd::kStage + 1024;
    if ((e = cudaFuncSetAttribute(tcd::decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(dev.sm_count);
    cfg.blockDim = dim3(tcd::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, tcd::decode_tc_kernel, m_gate, m_up, m_down, a)) != cudaSuccess)
        return e;
    if (events)
        for (int i = 2; i <= 4; ++i)
            if ((e = record_phase(events[i], s)) != cudaSuccess) return e;
    return cudaGetLastError();
}

bool decode_path_supported(const Plan &p, const ds4g_moe_desc *d)
{
    if (d->format != DS4G_FMT_Q2K || d->down_format != DS4G_FMT_Q2K || p.T > kDecodeMaxT ||
        p.I % kTileM != 0 ||
        p.H % kDownRows != 0)
        return false;
    if (p.T > kDecodePreferT) return p.H % tcd::kBM == 0;      // tcgen05 decode kernel
    // two ring stages and the fixed buffers must fit in shared memory
    const size_t gu = (size_t)2 * kTileM * smem_pitch(d->gate_up_row_bytes);
    const size_t dn = (size_t)kDownRows * smem_pitch(d->down_row_bytes);
    const size_t stage = (std::max(gu, dn) + 127) / 128 * 128;
    const size_t fixed = (size_t)(2 + kDownPairs) * kConsumers * 4 * kTileM * 4 +
                         (size_t)p.A * kDownRows * 4 + 1024;
    return 2 * stage + fixed <= kSmemBudget;
}

cudaError_t launch_decode_path(const LayerArgs &la, const DecodeBufs &db, const DeviceInfo &dev,
                               cudaStream_t s, const cudaEvent_t *events, uint64_t wait_ns,
                               bool stall)
{
    // up to kDecodePreferT vectors the mma.sync kernel has the shorter
    // dependency chain; above that the tcgen05 kernel's lower instruction
    // count per weight wins
    if (la.T > kDecodePreferT) return launch_decode_tc(la, db, dev, s, events, wait_ns, stall);
    DecArgs a{};
    a.H = la.H;
    a.I = la.I;
    a.I_pad = la.I_pad;
    a.E = la.E;
    a.k = la.k;
    a.T = la.T;
    a.A = la.A;
    a.score = db.score;
    a.H_blocks = la.H / kQK;
    a.I_blocks = la.I_pad / kQK;
    a.w_gate = la.w_gate;
    a.w_up = la.w_up;
    a.w_down = la.w_down;
    a.gu_row = la.gu_row;
    a.dn_row = la.dn_row;
    a.gu_stride = la.gu_stride;
    a.dn_stride = la.dn_stride;
    a.wslot = la.wslot;
    a.n_wslots = la.n_wslots;
    a.gu_pitch = (int)smem_pitch(la.gu_row);
    a.dn_pitch = (int)smem_pitch(la.dn_row);
    a.logits = db.logits;
    a.x = la.x;
    a.xp = db.xp;
    a.xs = db.xs;
    a.texp = db.texp;
    a.hp = db.hp;
    a.hs = db.hs;
    a.y = la.y;
    a.ids = db.ids;
    a.wts = const_cast<float *>(la.wts);
    a.counts = const_cast<int32_t *>(la.counts);
    a.offsets = const_cast<int32_t *>(la.offsets);
    a.perm = const_cast<int32_t *>(la.perm);
    a.status = db.status;
    a.sync = db.sync;
    a.wait_ns = wait_ns;
    a.stall = stall ? 1 : 0;
    const size_t xb = (size_t)a.T * a.H * 2 + (size_t)a.T * (a.H / 16) * 4;
    a.x_smem = xb <= kXStageMax ? 1 : 0;

    // counters and status reset; activation conversion when it does not fit
    const int pre_grid = a.x_smem ? 1 : a.T;
    decode_pre_kernel<<<pre_grid, 256, 0, s>>>(db.status, db.sync, decode_sync_words(a.E, a.H),
                                               a.x_smem ? nullptr : la.x,
                                               const_cast<__half *>(db.xp),
                                               const_cast<float *>(db.xs), a.T, a.H, db.texp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (events && (e = record_phase(events[1], s)) != cudaSuccess) return e;

    // token chunk per pass: segments longer than 4 run in several chunks
    // the one-vector kernel reads x and h from shared memory only
    const size_t dn_stage = (size_t)kDownRows * a.dn_pitch + (size_t)a.I_pad * 2 + (size_t)(a.I_pad / 16) * 4;
    const size_t gu_stage = (size_t)2 * kTileM * a.gu_pitch;
    if (la.T <= 1 && a.x_smem && dn_stage <= std::max(gu_stage, (size_t)kDownRows * a.dn_pitch))
        return launch_nt<1>(a, dev, s, events);
    if (la.T <= 2) return launch_nt<2>(a, dev, s, events);   // also T = 1 otherwise
    return launch_nt<4>(a, dev, s, events);
}

}  // namespace ds4g
