// ds4g_common.cuh -- internal declarations shared by the libds4g translation
// units (device helpers, workspace plan, kernel launchers).  Not installed.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/ds4g.h"

namespace ds4g {

constexpr int kQK = 256;         // weights per super-block
constexpr int kQ2KBytes = 84;    // Q2_K super-block
constexpr int kCB2Bytes = 70;    // codebook-2-bit super-block
constexpr int kQ4KBytes = 144;   // Q4_K super-block
constexpr int kQ5KBytes = 176;   // Q5_K super-block
constexpr int kQ6KBytes = 210;   // Q6_K super-block
constexpr int kMXFP4Bytes = 136; // eight 17-byte MXFP4 blocks (256 weights)

// The weight slot of expert e: e itself, or wslot[e] when the weight
// tensors hold a set of resident slots (an expert cache).  An entry outside
// 0 .. n_slots-1 is recorded as DS4G_ERR_INVALID in the status word and
// replaced by slot 0, so no weight access leaves the tensors.
__device__ __forceinline__ int weight_slot(const int32_t *wslot, int n_slots, int e,
                                           int32_t *status)
{
    if (!wslot) return e;
    const int s = __ldg(wslot + e);
    if (s >= 0 && s < n_slots) return s;
    if (status) atomicCAS(status, 0, (int32_t)DS4G_ERR_INVALID);
    return 0;
}

// Super-block bytes of a ds4g_format (0 for an unknown one).
__host__ __device__ constexpr int block_bytes_of(int fmt)
{
    return fmt == DS4G_FMT_Q2K ? kQ2KBytes
         : fmt == DS4G_FMT_CB2 ? kCB2Bytes
         : fmt == DS4G_FMT_Q4K ? kQ4KBytes
         : fmt == DS4G_FMT_Q5K ? kQ5KBytes
         : fmt == DS4G_FMT_Q6K ? kQ6KBytes
         : fmt == DS4G_FMT_MXFP4 ? kMXFP4Bytes
         : 0;
}

// ---------------------------------------------------------------------------
// Workspace plan: byte offsets of every scratch array inside the caller's
// workspace (each 256-byte aligned).  A = T * k assignments.
// ---------------------------------------------------------------------------
struct Plan {
    int32_t T, H, I, E, k, A;
    int32_t I_pad;          // inter rounded up to a multiple of 256 (down K)
    int32_t H_blocks;       // hidden / 256
    int32_t I_blocks;       // I_pad / 256
    int32_t gu_block_bytes; // super-block bytes of W_gate, W_up
    int32_t dn_block_bytes; // super-block bytes of W_down
    size_t ids, wts, counts, offsets, perm, slot_pos, active, meta;
    size_t status;          // int32 device status word (DS4G_OK or DS4G_ERR_TIMEOUT)
    size_t sync;            // [decode_sync_words] int32 counters of the decode kernels
    size_t gpart;           // K-split partial sums (decode)
    size_t xp, xs;          // [T x H] fp16 activations (4-group permuted), [T x H/16] sums
    size_t hp, hs;          // [A x I_pad] fp16 h (4-group permuted), [A x I_pad/16] sums
    size_t hbuf;            // [A x I_pad] fp32: SiLU(g)*u per assignment (segment order)
    size_t yslot;           // [A x H] fp32: w * o per assignment (segment order)
    size_t xseg;            // [A x H] fp16: activations in segment order (tensor-core path)
    size_t tiles;           // [tc_max_tiles x 4] int32 token tiles (tensor-core path)
    size_t wseg;            // [A] fp32 routing weight per segment row (tensor-core path)
    size_t texp;            // [T] int32 activation exponent of each token (see token_exponent)
    size_t eseg;            // [A] int32 activation exponent of each segment row (tensor-core path)
    size_t light;           // [E] int32 experts whose segments take the GEMV kernels (split calls)
    size_t x_stage;         // [T x H] bf16 (host entry point)
    size_t l_stage;         // [T x E] fp32 (host entry point)
    size_t y_stage;         // [T x H] fp32 (host entry point)
    size_t total;
};

// meta words (int32) at Plan::meta
enum { kMetaActive = 0, kMetaTiles = 1, kMetaLight = 2, kMetaWords = 64 };

// Validation + plan.  Returns DS4G_OK or the first error found.
ds4g_status make_plan(const ds4g_moe_desc *d, int32_t T, Plan *p);

// Per-device cached properties.
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
};
ds4g_status device_info(DeviceInfo *out);
// DS4G_OK for cudaSuccess, else DS4G_ERR_CUDA (remembering the CUDA error for
// ds4g_last_cuda_error).
ds4g_status status_from_cuda(cudaError_t e);

// ---------------------------------------------------------------------------
// Kernel launchers (all asynchronous on `s`; return cudaGetLastError()).
// ---------------------------------------------------------------------------
// Routing; optionally (x != nullptr) also the activation prep of the decode
// path: xp = fp16(x) in 4-group permuted order, xs = fp32 sums of 16.
// Writes *status = DS4G_OK first (status nullable) and zeroes sync[0 .. n_sync).
cudaError_t launch_route(const float *logits, int T, int E, int k, int score,
                         int32_t *ids, float *wts, int32_t *counts, int32_t *offsets,
                         int32_t *perm, int32_t *slot_pos, int32_t *active,
                         int32_t *n_active, const uint16_t *x, int H, __half *xp, float *xs,
                         int32_t *status, int32_t *sync, int n_sync, cudaStream_t s);

cudaError_t launch_q2k_dequant(const uint8_t *blocks, int64_t n_blocks, void *out, int dtype,
                               cudaStream_t s);
cudaError_t launch_cb2_dequant(const uint8_t *blocks, int64_t n_blocks, const int8_t *cb,
                               void *out, int dtype, cudaStream_t s);
// Q4_K / Q5_K / Q6_K / MXFP4 (fmt) super-blocks to fp32 / fp16 / bf16.
cudaError_t launch_kquant_dequant(int fmt, const uint8_t *blocks, int64_t n_blocks, void *out,
                                  int dtype, cudaStream_t s);

struct LayerArgs {
    int H, I, I_pad, E, k, A, T;
    int gu_format, dn_format;  // block formats of W_gate / W_up and of W_down
    const uint8_t *w_gate, *w_up, *w_down;
    int64_t gu_row, dn_row, gu_stride, dn_stride;
    const int32_t *wslot;      // [E] weight slot of each expert, or null (slot = expert)
    int n_wslots;              // slots the weight tensors hold (E when wslot is null)
    int32_t *status;           // device status word
    const int8_t *codebook;
    const uint16_t *x;         // [T x H] bf16
    const float *wts;          // [A] routing weights (assignment order)
    const int32_t *counts, *offsets, *perm, *slot_pos, *active, *n_active;
    float *hbuf;               // [A x I_pad]
    float *yslot;              // [A x H]
    float *y;                  // [T x H]
};

// Launches gate/up, down and combine.  `events` (nullable): events[2..4]
// are recorded after each of the three kernels.
cudaError_t launch_gemv_path(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s,
                             const cudaEvent_t *events);
int32_t gemv_path_launches(const Plan &p);
// y[t] = sum_i yslot[slot_pos[t*k+i]] in slot order (one launch).
cudaError_t launch_combine(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s);
// The GEMV gate/up and down kernels alone, over the experts a.active[0 ..
// *a.n_active) (the per-segment split runs them on the light segments).
cudaError_t launch_gemv_gateup(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s);
cudaError_t launch_gemv_down(const LayerArgs &a, const DeviceInfo &dev, cudaStream_t s);

// Records `ev` on `s`; inside a stream capture the record becomes an
// external event node, so that it is recorded again at every replay.
inline cudaError_t record_phase(cudaEvent_t ev, cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(
        ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault);
}

// T at or below which routing runs as one single-CTA launch.
constexpr int kRouteSmallT = 64;

// Decode path (decode.cu): T <= kDecodeMaxT, Q2_K, inter % 16 == 0.  Two
// launches: a reset/conversion kernel and one persistent layer kernel that
// routes by itself -- the mma.sync kernel up to kDecodePreferT tokens, the
// tcgen05 kernel above (events[1] after the first, events[2..4] after the
// second).
constexpr int kDecodeMaxT = 32;
constexpr int kDecodePreferT = 8;       // mma.sync decode kernel up to here, tcgen05 above
struct DecodeBufs {
    const float *logits;    // [T x E]
    int32_t *ids;           // routing outputs of the call (the kernel routes by itself)
    int score;
    const __half *xp;       // [T x H] fp16 activations when they do not fit on chip
    const float *xs;
    __half *hp;
    float *hs;
    int32_t *status;
    int32_t *sync;          // [decode_sync_words] claim and completion counters
    float *gpart;           // K-split partial sums of the tensor-core decode kernel
    int32_t *texp;          // [T] token exponents (written when the activations are converted ahead)
};
constexpr int kSyncWords = 4;
constexpr int kDecodeMaxPairs = 1024;
// Counter words of the decode kernels: claims, per-expert h completion,
// per-128-row y tiles, K-split tile pairs.
inline int decode_sync_words(int E, int H) { return kSyncWords + E + H / 128 + kDecodeMaxPairs; }
// Bytes of K-split partial sums: per (token chunk, 128-row tile) pair, two
// K halves x two matrices x 4 vectors x 128 rows of fp32.
inline size_t decode_gpart_bytes(int A, int I_pad)
{
    const size_t pairs = (size_t)std::min(A * (I_pad / 128), kDecodeMaxPairs);
    return pairs * 2 * 2 * 4 * 128 * 4;
}
bool decode_path_supported(const Plan &p, const ds4g_moe_desc *d);
cudaError_t launch_decode_path(const LayerArgs &a, const DecodeBufs &b, const DeviceInfo &dev,
                               cudaStream_t s, const cudaEvent_t *events, uint64_t wait_ns,
                               bool stall);

// Tensor-core path (tc.cu): Q2_K, rows a multiple of 16 bytes.
constexpr int kTcTileTokens = 128;      // tokens per tensor-core work item at most
struct TcBufs {
    __half *xseg;          // [A x H] fp16
    __half *hp;            // [A x I_pad] fp16
    int32_t *tiles;        // [tc_max_tiles x 4]
    int32_t *n_tiles;
    int32_t *status;
    float *wseg;           // [A] routing weight of each segment row
    int32_t *texp;         // [T] activation exponent of each token
    int32_t *eseg;         // [A] activation exponent of each segment row
    int32_t *light;        // [E] experts routed to the GEMV kernels (split calls)
    int32_t *n_light;
    int min_tokens;        // segments with fewer tokens take the GEMV kernels (0: none)
};
bool tc_path_supported(const Plan &p, const ds4g_moe_desc *d);
int32_t tc_max_tiles(int32_t E, int32_t A);
// Token tiles and the activation gather (one launch), then gate/up, down and
// the combine (events[2..4] recorded after each, when given).
cudaError_t launch_tc_prep(const LayerArgs &a, const TcBufs &b, const DeviceInfo &dev,
                           cudaStream_t s);
cudaError_t launch_tc_path(const LayerArgs &a, const TcBufs &b, const DeviceInfo &dev,
                           cudaStream_t s, const cudaEvent_t *events, uint64_t wait_ns,
                           bool stall);
constexpr int32_t kTcPathLaunches = 5;  // token exponents, prep, gate/up, down, combine
constexpr int32_t kSplitLaunches = 2;   // GEMV gate/up and down of a per-segment split

// Bounded device waits: default limit, and the short limit used with
// DS4G_DEBUG_STALL.
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kStallWaitNs = 2000000ull;

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float half_bits(uint32_t bits16)
{
    return __half2float(__ushort_as_half((unsigned short)bits16));
}

__device__ __forceinline__ float bf16_bits(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g / (1.0f + expf(-g)) * u;
}

// ---------------------------------------------------------------------------
// Per-token power-of-two scaling of the fp16 operands.  The tensor-core and
// decode kernels multiply in fp16, whose range (6.1e-5 .. 65504 at full
// precision) is narrower than bf16's.  Token t's activations enter as
// x * 2^-e_t with e_t chosen so that the largest finite |x| of the token lands
// in [2^10, 2^11); the gate and up accumulators are multiplied back by 2^e_t
// in fp32, SiLU(g)*u is formed in fp32 and stored as h * 2^-f_t with
// f_t = 2 e_t + 14 (h grows like x^2), and the down projection's result is
// multiplied back by 2^f_t.  Every scaling is by a power of two, so it is
// exact wherever no value leaves the normal range.  e_t is clamped to
// [-40, 40]; a token without a nonzero finite value gets 0.
// ---------------------------------------------------------------------------
constexpr int kExpTarget = 10;
constexpr int kExpMin = -40, kExpMax = 40;
constexpr int kHExpOffset = 14;

// e_t from the token's largest finite |x| (non-negative, finite).
__device__ __forceinline__ int token_exponent(float max_abs)
{
    if (!(max_abs > 0.0f)) return 0;                 // no nonzero finite value
    const int e = ((int)((__float_as_uint(max_abs) >> 23) & 0xFF) - 127) - kExpTarget;
    return e < kExpMin ? kExpMin : (e > kExpMax ? kExpMax : e);
}

// 2^e as a float for -126 <= e <= 127.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// |x| of a bf16 value as float when finite, else 0 (for token maxima).
__device__ __forceinline__ float bf16_abs_finite(uint32_t bits16)
{
    const uint32_t a = (bits16 & 0x7FFFu) << 16;
    return a < 0x7F800000u ? __uint_as_float(a) : 0.0f;
}

// texp[t] = e_t for t < T (one warp per token; x [T x H] bf16).
cudaError_t launch_token_exponents(const uint16_t *x, int T, int H, int32_t *texp, cudaStream_t s);

}  // namespace ds4g
