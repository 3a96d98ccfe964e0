// decode.cu -- the decode path for Q2_K experts: small expert segments
// (micro-batched decode, ds4 README mirror, "So, what can I do with this
// software?"), bound by the HBM bytes of the quantized weights.
//
//   gateup kernel: h[p, n] = SiLU(W_gate[e][n,:] . x_t) * (W_up[e][n,:] . x_t)
//   down kernel:   y[t, m] = sum_{i<k} w[t,i] * (W_down[e_i][m,:] . h[p(t,i), :])
//
// Both kernels are persistent (one CTA per SM).  A producer warp streams
// 16-row (gate/up) or 32-row (down) weight tiles -- contiguous runs of
// 84-byte blocks -- into a shared-memory ring with cp.async.bulk (TMA, no
// tensor map) completing on mbarriers; eight consumer warps dequantize in
// registers straight into mma.sync m16n8k16 fragments.
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
// kernel as fp16 (one rounding, relative 2^-11) with fp32 sub-block sums of
// those fp16 values for the down kernel's correction and min terms.
//
// Kernel chaining: routing -> gateup -> down by programmatic dependent launch.
// The down kernel's producer starts streaming W_down (which does not depend
// on h) before griddepcontrol.wait; its consumers wait.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel records
// DS4G_ERR_TIMEOUT in the workspace status word, drains its own copies (also
// bounded) and returns.
#include "ds4g_common.cuh"
#include "ptx.cuh"

namespace ds4g {
namespace {

constexpr int kTileM = 16;
constexpr int kConsumers = 8;
constexpr int kThreads = (kConsumers + 1) * 32;

// 4-group permutation of activations: element i of an aligned group of 4 is
// stored at position perm4(i), so that elements (i, i+2) are adjacent.
__device__ __forceinline__ int perm4(int n) { return (n & ~3) | ((n & 1) << 1) | ((n >> 1) & 1); }

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ float nib_lo(uint32_t b) { return (float)(b & 15u); }
__device__ __forceinline__ float nib_hi(uint32_t b) { return (float)((b >> 4) & 15u); }

struct Ring {
    uint64_t *full;
    uint64_t *empty;
    uint8_t *data;
    int stages;
    uint32_t stage_bytes;
    __device__ uint8_t *stage(int s) const { return data + (size_t)s * stage_bytes; }
};

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

__device__ __forceinline__ void build_half_a(HalfA &ha, const uint8_t *blk0, const uint8_t *blk1,
                                             int h, int c)
{
    const uint32_t g1 = (uint32_t)(c >> 1);
    const uint32_t m1 = 0x00030003u << (2 * g1);          // field g1   -> sub-block c
    const uint32_t m2 = 0x00030003u << (2 * (g1 + 2));    // field g1+2 -> sub-block c+4
    const int off = 16 + 32 * h + 16 * (c & 1);
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

// The 8 MMAs of one half for one activation vector.  `xh`: the half's 128
// activations (fp16, 4-group permuted) in global memory; `xs`: the 8
// sub-block sums.  Returns D (rows grp, grp+8 x columns 2c, 2c+1) =
// 4^c * sum_{sub-block} q*x.
__device__ __forceinline__ void half_mma(const HalfA &ha, const __half *xh, const float *xs,
                                         int grp, int c, float (&d)[4], float &x0, float &x1)
{
    const float2 xx = *reinterpret_cast<const float2 *>(xs + 2 * c);
    x0 = xx.x;
    x1 = xx.y;
    d[0] = -1024.0f * x0;
    d[1] = -1024.0f * x1;
    d[2] = d[0];
    d[3] = d[1];
    uint32_t bv[8];
    const bool act = (grp & 3) == c;
    if (act) {
        // coherent loads: h is written by the previous grid of the chain
        const uint4 *p = reinterpret_cast<const uint4 *>(xh + 16 * grp);
        uint4 u0 = p[0], u1 = p[1];
        bv[0] = u0.x; bv[1] = u0.y; bv[2] = u0.z; bv[3] = u0.w;
        bv[4] = u1.x; bv[5] = u1.y; bv[6] = u1.z; bv[7] = u1.w;
    } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) bv[t] = 0u;
    }
    const bool lo = grp < 4;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t b0 = lo ? bv[t] : 0u;
        const uint32_t b1 = lo ? 0u : bv[t];
        ptx::mma_16816(d, ha.a[t], b0, b1, d);
    }
}

struct DecArgs {
    int H, I, I_pad, E, k, T, A;
    int H_blocks, I_blocks;
    const uint8_t *w_gate, *w_up, *w_down;
    int64_t gu_row, dn_row, gu_stride, dn_stride;
    const float *wts;
    const int32_t *offsets, *perm, *slot_pos, *active, *n_active;
    const __half *xp;   // [T][H]
    const float *xs;    // [T][H/16]
    __half *hp;         // [A][I_pad]
    float *hs;          // [A][I_pad/16]
    float *y;           // [T][H]
    int32_t *status;
    uint64_t wait_ns;
    int stages;
    int stall;          // debug: the producer issues nothing (tests the bounded waits)
};

// ---------------------------------------------------------------------------
// gate/up
// ---------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) gateup_q2k_kernel(DecArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 2, c = lane & 3;
    const uint32_t tile_bytes = (uint32_t)(kTileM * a.gu_row);
    Ring ring;
    ring.stages = a.stages;
    ring.stage_bytes = (2 * tile_bytes + 127) / 128 * 128;
    ring.data = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)ring.stages * ring.stage_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + kConsumers * 2 * NT * kTileM);
    ring.full = bars;
    ring.empty = bars + ring.stages;
    // s_pabort: set by the producer; s_cabort: set by consumers only between
    // their wait and the consumer barrier that follows it, and read by all
    // consumers right after that barrier, so every consumer warp takes the
    // same branch (a bar.sync cannot time out).
    __shared__ int s_pabort, s_cabort, s_consumed, s_issued;

    if (tid == 0) {
        for (int s = 0; s < ring.stages; ++s) {
            ptx::mbar_init(&ring.full[s], 1);
            ptx::mbar_init(&ring.empty[s], kConsumers);
        }
        ptx::fence_mbar_init();
        s_pabort = 0;
        s_cabort = 0;
        s_consumed = 0;
        s_issued = 0;
    }
    __syncthreads();

    ptx::grid_dep_wait();          // routing and the activation prep are complete
    ptx::grid_dep_launch();        // let the down kernel start streaming W_down

    const int tiles = a.I / kTileM;
    const int n_items = *a.n_active * tiles;
    const int first = (int)((int64_t)blockIdx.x * n_items / gridDim.x);
    const int last = (int)((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);
    const int mine = last - first;

    if (warp == kConsumers) {
        // ---------------- producer ----------------
        if (lane == 0 && !a.stall) {
            for (int li = 0; li < mine; ++li) {
                const int s = li % ring.stages;
                if (li >= ring.stages &&
                    !ptx::mbar_wait(&ring.empty[s], ((li / ring.stages) - 1) & 1, a.wait_ns)) {
                    set_status(a.status, DS4G_ERR_TIMEOUT);
                    s_pabort = 1;
                    break;
                }
                if (*(volatile int *)&s_cabort) break;
                const int item = first + li;
                const int e = a.active[item / tiles];
                const int mt = item % tiles;
                const uint8_t *g = a.w_gate + (size_t)e * a.gu_stride + (size_t)mt * tile_bytes;
                const uint8_t *u = a.w_up + (size_t)e * a.gu_stride + (size_t)mt * tile_bytes;
                ptx::mbar_arrive_expect_tx(&ring.full[s], 2 * tile_bytes);
                ptx::bulk_g2s(ring.stage(s), g, tile_bytes, &ring.full[s]);
                ptx::bulk_g2s(ring.stage(s) + tile_bytes, u, tile_bytes, &ring.full[s]);
                s_issued = li + 1;
            }
        }
    } else {
        // ---------------- consumers ----------------
        const float inv4c = 1.0f / (float)(1 << (2 * c));
        for (int li = 0; li < mine; ++li) {
            const int s = li % ring.stages;
            if (!ptx::mbar_wait(&ring.full[s], (li / ring.stages) & 1, a.wait_ns)) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                s_cabort = 1;
            }
            consumer_sync();
            if (*(volatile int *)&s_cabort) break;
            const int item = first + li;
            const int e = a.active[item / tiles];
            const int mt = item % tiles;
            const int seg0 = a.offsets[e], seg_n = a.offsets[e + 1] - seg0;
            const uint8_t *st = ring.stage(s);
            for (int c0 = 0; c0 < seg_n; c0 += NT) {
                const int nt = min(NT, seg_n - c0);
                int tok[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) tok[j] = a.perm[seg0 + c0 + (j < nt ? j : 0)] / a.k;
                float part[2][NT][2];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int j = 0; j < NT; ++j) part[m][j][0] = part[m][j][1] = 0.0f;
                for (int kb = warp; kb < a.H_blocks; kb += kConsumers) {
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const uint8_t *b0 = st + m * tile_bytes + (size_t)grp * a.gu_row + kb * kQ2KBytes;
                        const uint8_t *b1 = b0 + 8 * a.gu_row;
                        const uint32_t dd0 = ptx::lds32(b0 + 80), dd1 = ptx::lds32(b1 + 80);
                        float S[NT][2], M[NT][2];
#pragma unroll
                        for (int j = 0; j < NT; ++j) S[j][0] = S[j][1] = M[j][0] = M[j][1] = 0.0f;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            HalfA ha;
                            build_half_a(ha, b0, b1, h, c);
                            const uint32_t sb0 = *reinterpret_cast<const uint16_t *>(b0 + 8 * h + 2 * c);
                            const uint32_t sb1 = *reinterpret_cast<const uint16_t *>(b1 + 8 * h + 2 * c);
                            const float sc00 = nib_lo(sb0), sc01 = nib_lo(sb0 >> 8);
                            const float mn00 = nib_hi(sb0), mn01 = nib_hi(sb0 >> 8);
                            const float sc10 = nib_lo(sb1), sc11 = nib_lo(sb1 >> 8);
                            const float mn10 = nib_hi(sb1), mn11 = nib_hi(sb1 >> 8);
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                if (j < nt) {
                                    const __half *xh = a.xp + (size_t)tok[j] * a.H + kb * kQK + 128 * h;
                                    const float *xsh = a.xs + (size_t)tok[j] * (a.H / 16) + kb * 16 + 8 * h;
                                    float d[4], x0, x1;
                                    half_mma(ha, xh, xsh, grp, c, d, x0, x1);
                                    S[j][0] += sc00 * d[0] + sc01 * d[1];
                                    S[j][1] += sc10 * d[2] + sc11 * d[3];
                                    M[j][0] += mn00 * x0 + mn01 * x1;
                                    M[j][1] += mn10 * x0 + mn11 * x1;
                                }
                            }
                        }
                        const float d0 = half_bits(dd0 & 0xFFFFu) * inv4c, dm0 = half_bits(dd0 >> 16);
                        const float d1 = half_bits(dd1 & 0xFFFFu) * inv4c, dm1 = half_bits(dd1 >> 16);
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            part[m][j][0] += d0 * S[j][0] - dm0 * M[j][0];
                            part[m][j][1] += d1 * S[j][1] - dm1 * M[j][1];
                        }
                    }
                }
                // reduce over the quad (sub-block owners), then over warps
                float *rw = red + (size_t)warp * 2 * NT * kTileM;
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            float v = part[m][j][r];
                            v += __shfl_xor_sync(0xffffffffu, v, 1);
                            v += __shfl_xor_sync(0xffffffffu, v, 2);
                            if (c == 0) rw[(m * NT + j) * kTileM + grp + 8 * r] = v;
                        }
                consumer_sync();
                if (tid < nt * kTileM) {
                    const int row = tid & 15, j = tid >> 4;
                    float g = 0.0f, u = 0.0f;
                    for (int w = 0; w < kConsumers; ++w) {
                        g += red[((size_t)w * 2 * NT + j) * kTileM + row];
                        u += red[((size_t)w * 2 * NT + NT + j) * kTileM + row];
                    }
                    const __half hv = __float2half_rn(silu_mul(g, u));
                    const int pos = seg0 + c0 + j;
                    const int n = mt * kTileM + row;
                    a.hp[(size_t)pos * a.I_pad + perm4(n)] = hv;
                    float hsum = __half2float(hv);
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) hsum += __shfl_xor_sync(0x0000ffffu << (16 * ((tid >> 4) & 1)), hsum, off);
                    if (row == 0) a.hs[(size_t)pos * (a.I_pad / 16) + mt] = hsum;
                }
                consumer_sync();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ring.empty[s]);
            if (tid == 0) s_consumed = li + 1;
        }
    }
    __syncthreads();
    const bool aborted = s_pabort || s_cabort;
    // drain copies that were issued but not consumed (only after an abort)
    if (tid == kConsumers * 32 && aborted) {
        for (int li = s_consumed; li < s_issued; ++li) {
            const int s = li % ring.stages;
            if (!ptx::mbar_wait(&ring.full[s], (li / ring.stages) & 1, a.wait_ns)) break;
        }
    }
    // zero h rows inter..I_pad-1 (padding of the down projection's K)
    const int pad_tiles = (a.I_pad - a.I) / kTileM;
    if (pad_tiles > 0 && !aborted) {
        const int n_act = *a.n_active;
        for (int j = blockIdx.x; j < n_act; j += gridDim.x) {
            const int e = a.active[j];
            const int seg0 = a.offsets[e], seg_n = a.offsets[e + 1] - seg0;
            for (int i = tid; i < seg_n * (a.I_pad - a.I); i += blockDim.x) {
                const int pos = seg0 + i / (a.I_pad - a.I), n = a.I + i % (a.I_pad - a.I);
                a.hp[(size_t)pos * a.I_pad + n] = __float2half_rn(0.0f);
                if ((n & 15) == 0) a.hs[(size_t)pos * (a.I_pad / 16) + n / 16] = 0.0f;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// down + weighted combine
// ---------------------------------------------------------------------------
constexpr int kDownRows = 32;   // two MMA tiles per work item

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) down_q2k_kernel(DecArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = lane >> 2, c = lane & 3;
    const uint32_t tile_bytes = (uint32_t)(kDownRows * a.dn_row);
    Ring ring;
    ring.stages = a.stages;
    ring.stage_bytes = (tile_bytes + 127) / 128 * 128;
    ring.data = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)ring.stages * ring.stage_bytes);
    float *obuf = red + kConsumers * NT * kTileM;                   // [A][32]
    uint64_t *bars = reinterpret_cast<uint64_t *>(obuf + (size_t)a.A * kDownRows);
    ring.full = bars;
    ring.empty = bars + ring.stages;
    __shared__ int s_pabort, s_cabort, s_consumed, s_issued;   // as in the gate/up kernel

    if (tid == 0) {
        for (int s = 0; s < ring.stages; ++s) {
            ptx::mbar_init(&ring.full[s], 1);
            ptx::mbar_init(&ring.empty[s], kConsumers);
        }
        ptx::fence_mbar_init();
        s_pabort = 0;
        s_cabort = 0;
        s_consumed = 0;
        s_issued = 0;
    }
    __syncthreads();

    // Routing finished before the gate/up kernel let this grid launch, so the
    // expert list is final; h is not (consumers wait for it below).
    const int n_act = *a.n_active;
    const int n_items = a.H / kDownRows;
    const int first = (int)((int64_t)blockIdx.x * n_items / gridDim.x);
    const int last = (int)((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);
    const int total = (last - first) * n_act;     // (item, expert) stages

    if (warp == kConsumers) {
        if (lane == 0 && !a.stall) {
            for (int q = 0; q < total; ++q) {
                const int s = q % ring.stages;
                if (q >= ring.stages &&
                    !ptx::mbar_wait(&ring.empty[s], ((q / ring.stages) - 1) & 1, a.wait_ns)) {
                    set_status(a.status, DS4G_ERR_TIMEOUT);
                    s_pabort = 1;
                    break;
                }
                if (*(volatile int *)&s_cabort) break;
                const int item = first + q / n_act;
                const int e = a.active[q % n_act];
                const uint8_t *src = a.w_down + (size_t)e * a.dn_stride + (size_t)item * tile_bytes;
                ptx::mbar_arrive_expect_tx(&ring.full[s], tile_bytes);
                ptx::bulk_g2s(ring.stage(s), src, tile_bytes, &ring.full[s]);
                s_issued = q + 1;
            }
        }
    } else {
        ptx::grid_dep_wait();      // h from the gate/up kernel
        const int mtile = warp >> 2, kw = warp & 3;
        const float inv4c = 1.0f / (float)(1 << (2 * c));
        for (int q = 0; q < total; ++q) {
            const int s = q % ring.stages;
            if (!ptx::mbar_wait(&ring.full[s], (q / ring.stages) & 1, a.wait_ns)) {
                set_status(a.status, DS4G_ERR_TIMEOUT);
                s_cabort = 1;
            }
            consumer_sync();
            if (*(volatile int *)&s_cabort) break;
            const int item = first + q / n_act;
            const int jx = q % n_act;
            const int e = a.active[jx];
            const int seg0 = a.offsets[e], seg_n = a.offsets[e + 1] - seg0;
            const uint8_t *st = ring.stage(s) + (size_t)mtile * kTileM * a.dn_row;
            for (int c0 = 0; c0 < seg_n; c0 += NT) {
                const int nt = min(NT, seg_n - c0);
                float part[NT][2];
#pragma unroll
                for (int j = 0; j < NT; ++j) part[j][0] = part[j][1] = 0.0f;
                for (int kb = kw; kb < a.I_blocks; kb += 4) {
                    const uint8_t *b0 = st + (size_t)grp * a.dn_row + kb * kQ2KBytes;
                    const uint8_t *b1 = b0 + 8 * a.dn_row;
                    const uint32_t dd0 = ptx::lds32(b0 + 80), dd1 = ptx::lds32(b1 + 80);
                    float S[NT][2], M[NT][2];
#pragma unroll
                    for (int j = 0; j < NT; ++j) S[j][0] = S[j][1] = M[j][0] = M[j][1] = 0.0f;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        HalfA ha;
                        build_half_a(ha, b0, b1, h, c);
                        const uint32_t sb0 = *reinterpret_cast<const uint16_t *>(b0 + 8 * h + 2 * c);
                        const uint32_t sb1 = *reinterpret_cast<const uint16_t *>(b1 + 8 * h + 2 * c);
                        const float sc00 = nib_lo(sb0), sc01 = nib_lo(sb0 >> 8);
                        const float mn00 = nib_hi(sb0), mn01 = nib_hi(sb0 >> 8);
                        const float sc10 = nib_lo(sb1), sc11 = nib_lo(sb1 >> 8);
                        const float mn10 = nib_hi(sb1), mn11 = nib_hi(sb1 >> 8);
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            if (j < nt) {
                                const int pos = seg0 + c0 + j;
                                const __half *hh = a.hp + (size_t)pos * a.I_pad + kb * kQK + 128 * h;
                                const float *hsh = a.hs + (size_t)pos * (a.I_pad / 16) + kb * 16 + 8 * h;
                                float d[4], x0, x1;
                                half_mma(ha, hh, hsh, grp, c, d, x0, x1);
                                S[j][0] += sc00 * d[0] + sc01 * d[1];
                                S[j][1] += sc10 * d[2] + sc11 * d[3];
                                M[j][0] += mn00 * x0 + mn01 * x1;
                                M[j][1] += mn10 * x0 + mn11 * x1;
                            }
                        }
                    }
                    const float d0 = half_bits(dd0 & 0xFFFFu) * inv4c, dm0 = half_bits(dd0 >> 16);
                    const float d1 = half_bits(dd1 & 0xFFFFu) * inv4c, dm1 = half_bits(dd1 >> 16);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        part[j][0] += d0 * S[j][0] - dm0 * M[j][0];
                        part[j][1] += d1 * S[j][1] - dm1 * M[j][1];
                    }
                }
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
                consumer_sync();
                if (tid < nt * kDownRows) {
                    const int row = tid & 31, j = tid >> 5;
                    const int mt = row >> 4, r16 = row & 15;
                    float o = 0.0f;
                    for (int w = 0; w < 4; ++w) o += red[((size_t)(4 * mt + w) * NT + j) * kTileM + r16];
                    obuf[(size_t)(seg0 + c0 + j) * kDownRows + row] = o;
                }
                consumer_sync();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&ring.empty[s]);
            if (tid == 0) s_consumed = q + 1;
            // after the item's last expert: weighted combine in slot order
            if (jx == n_act - 1) {
                consumer_sync();
                for (int i = tid; i < a.T * kDownRows; i += kConsumers * 32) {
                    const int t = i / kDownRows, row = i % kDownRows;
                    float acc = 0.0f;
                    for (int sl = 0; sl < a.k; ++sl) {
                        const int asg = t * a.k + sl;
                        acc += a.wts[asg] * obuf[(size_t)a.slot_pos[asg] * kDownRows + row];
                    }
                    a.y[(size_t)t * a.H + (size_t)item * kDownRows + row] = acc;
                }
                consumer_sync();
            }
        }
    }
    __syncthreads();
    if (tid == kConsumers * 32 && (s_pabort || s_cabort)) {
        for (int q = s_consumed; q < s_issued; ++q) {
            const int s = q % ring.stages;
            if (!ptx::mbar_wait(&ring.full[s], (q / ring.stages) & 1, a.wait_ns)) break;
        }
    }
}

size_t gateup_smem(const DecArgs &a, int nt)
{
    const size_t stage = ((size_t)2 * kTileM * a.gu_row + 127) / 128 * 128;
    return stage * a.stages + (size_t)kConsumers * 2 * nt * kTileM * 4 + 2 * a.stages * 8;
}

size_t down_smem(const DecArgs &a, int nt)
{
    const size_t stage = ((size_t)kDownRows * a.dn_row + 127) / 128 * 128;
    return stage * a.stages + (size_t)kConsumers * nt * kTileM * 4 + (size_t)a.A * kDownRows * 4 +
           2 * a.stages * 8;
}

template <typename K>
cudaError_t launch_pdl(K kernel, int grid, size_t smem, cudaStream_t s, const DecArgs &a)
{
    // the opt-in limit covers static + dynamic shared memory, so ask for the
    // dynamic bytes this launch needs
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Shared memory per SM is split so that a gate/up CTA and a down CTA can be
// resident together (the down CTA streams W_down while gate/up computes).
constexpr size_t kGateUpBudget = 132 * 1024;
constexpr size_t kDownBudget = 90 * 1024;


template <int NT>
cudaError_t launch_nt(DecArgs a, const DeviceInfo &dev, cudaStream_t s, const cudaEvent_t *ev)
{
    const size_t budget = (size_t)dev.max_smem_optin - 1024;   // static shared memory
    a.stages = 4;
    while (a.stages > 2 && gateup_smem(a, NT) > kGateUpBudget) --a.stages;
    if (gateup_smem(a, NT) > budget) return cudaErrorInvalidValue;
    const int gu_items = min(a.E, a.A) * (a.I / kTileM);
    int grid = min(dev.sm_count, gu_items);
    cudaError_t e = launch_pdl(gateup_q2k_kernel<NT>, grid, gateup_smem(a, NT), s, a);
    if (e != cudaSuccess) return e;
    if (ev && (e = record_phase(ev[2], s)) != cudaSuccess) return e;
    DecArgs b = a;
    b.stages = 6;
    while (b.stages > 2 && down_smem(b, NT) > kDownBudget) --b.stages;
    if (down_smem(b, NT) > budget) return cudaErrorInvalidValue;
    grid = min(dev.sm_count, a.H / kDownRows);
    e = launch_pdl(down_q2k_kernel<NT>, grid, down_smem(b, NT), s, b);
    if (e != cudaSuccess) return e;
    if (ev) {
        if ((e = record_phase(ev[3], s)) != cudaSuccess) return e;
        if ((e = record_phase(ev[4], s)) != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

bool decode_path_supported(const Plan &p, const ds4g_moe_desc *d)
{
    if (d->format != DS4G_FMT_Q2K || p.T > kDecodeMaxT || p.I % kTileM != 0 ||
        p.H % kDownRows != 0)
        return false;
    // two ring stages of each kernel must fit in shared memory
    const size_t gu = 2 * (((size_t)2 * kTileM * d->gate_up_row_bytes + 127) / 128 * 128);
    const size_t dn = 2 * (((size_t)kDownRows * d->down_row_bytes + 127) / 128 * 128) +
                      (size_t)p.A * kDownRows * 4;
    return gu + 16 * 1024 <= 200 * 1024 && dn + 16 * 1024 <= 200 * 1024;
}

cudaError_t launch_decode_path(const LayerArgs &la, const DecodeBufs &db, const DeviceInfo &dev,
                               cudaStream_t s, const cudaEvent_t *events, uint64_t wait_ns,
                               bool stall)
{
    DecArgs a{};
    a.H = la.H;
    a.I = la.I;
    a.I_pad = la.I_pad;
    a.E = la.E;
    a.k = la.k;
    a.T = la.T;
    a.A = la.A;
    a.H_blocks = la.H / kQK;
    a.I_blocks = la.I_pad / kQK;
    a.w_gate = la.w_gate;
    a.w_up = la.w_up;
    a.w_down = la.w_down;
    a.gu_row = la.gu_row;
    a.dn_row = la.dn_row;
    a.gu_stride = la.gu_stride;
    a.dn_stride = la.dn_stride;
    a.wts = la.wts;
    a.offsets = la.offsets;
    a.perm = la.perm;
    a.slot_pos = la.slot_pos;
    a.active = la.active;
    a.n_active = la.n_active;
    a.xp = db.xp;
    a.xs = db.xs;
    a.hp = db.hp;
    a.hs = db.hs;
    a.y = la.y;
    a.status = db.status;
    a.wait_ns = wait_ns;
    a.stall = stall ? 1 : 0;
    if (la.T <= 1) return launch_nt<1>(a, dev, s, events);
    if (la.T <= 2) return launch_nt<2>(a, dev, s, events);
    if (la.T <= 4) return launch_nt<4>(a, dev, s, events);
    return launch_nt<8>(a, dev, s, events);
}

}  // namespace ds4g
