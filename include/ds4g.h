/*
 * ds4g.h -- C ABI of libds4g: the routed mixture-of-experts expert layer over
 * low-bit quantized expert weights (2-bit in the shipping mix; also the
 * routed Q4_K / Q5_K / Q6_K and MXFP4 formats), as hand-written CUDA kernels
 * for the NVIDIA B300 (sm_103a).
 *
 * What the layer is.  The ds4 README (codehub.bot mirror, section "Model
 * Weights") states that only the routed MoE experts are quantized -- up/gate
 * and down -- at 2 bits (IQ2_XXS for up/gate, Q2_K for down in the shipping
 * mix), that these experts are the majority of the model's bytes, and that
 * the GGUF quant layouts are those of llama.cpp (same page, section
 * "Acknowledgements to llama.cpp and GGML").  The same page ("So, what can I
 * do with this software?") names micro-batched decode and prefill on CUDA.
 * For one layer call over T tokens this library computes:
 *
 *   1. top-k routing over the router logits (ds4g_route_topk);
 *   2. per-expert token counts, segment offsets and the token-by-expert
 *      permutation;
 *   3. for every (token t, slot i), expert e = ids[t,i]:
 *        g = W_gate[e] x_t,  u = W_up[e] x_t,  h = SiLU(g) * u,
 *        o = W_down[e] h;
 *   4. y_t = sum_{i<k} w[t,i] * o_{t,i}, summed in slot order.
 *
 * Formats (256-weight super-blocks, little-endian fp16 scalars):
 *   Q2_K, 84 bytes:  scales[16] (low nibble = scale sc_s, high nibble = min
 *     m_s of 16-weight sub-block s), qs[64] (2-bit quants), d, dmin.
 *     Weight j: h = j/128, g = (j%128)/32, l = j%32,
 *     q = (qs[32h + l] >> 2g) & 3, s = j/16,
 *     w_j = d * (sc_s & 15) * q - dmin * (sc_s >> 4).
 *   Codebook-2-bit ("CB2", IQ2_XXS-style), 70 bytes: idx[32] (codebook row
 *     of weights 8o..8o+7), sgn[32] (bit b set: weight 8o+b negated), sc[4]
 *     (4-bit scale of 32-weight group G in nibble G&1 of byte G>>1, low
 *     nibble first), d.  w_j = d * s_{j/32} * cb[idx[j/8]][j%8] * (+-1);
 *     cb is a 256 x 8 int8 codebook.
 *   A matrix [N rows x K] is N rows of ceil(K/256) blocks; row n starts at
 *   n * row_bytes; weights at columns >= K are ignored.
 *
 * Conventions for every entry point.
 *   - Memory: every array argument is a DEVICE pointer owned by the caller,
 *     except where an entry point says "host".  The library allocates no
 *     device memory; scratch lives in the caller's workspace.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Work is enqueued on it; no entry point synchronizes
 *     except ds4g_moe_forward_host, which says so.
 *   - Errors: a status is returned synchronously.  Arguments are validated on
 *     the host before any launch; a rejected call launches nothing and leaves
 *     every output untouched.  Launch failures map to DS4G_ERR_CUDA.
 *     Faults inside a kernel surface at the caller's next synchronization.
 *   - Threads: calls on distinct streams with distinct workspaces may run
 *     concurrently.  The only library state is a per-device property cache.
 *   - Determinism: identical inputs give bit-identical outputs; no result
 *     depends on floating-point atomics or on launch timing.
 */
#ifndef DS4G_H
#define DS4G_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DS4G_ABI_VERSION 3

/* Symbols of the shared library (built with hidden default visibility). */
#if defined(__GNUC__)
#define DS4G_API __attribute__((visibility("default")))
#else
#define DS4G_API
#endif

typedef enum ds4g_status {
    DS4G_OK = 0,
    DS4G_ERR_INVALID = 1,      /* null pointer, negative size, bad enum, k > E ... */
    DS4G_ERR_SHAPE = 2,        /* a dimension outside the supported range         */
    DS4G_ERR_LAYOUT = 3,       /* misaligned pointer or unusable row/expert stride */
    DS4G_ERR_WORKSPACE = 4,    /* workspace pointer misaligned or too small        */
    DS4G_ERR_UNSUPPORTED = 5,  /* a forced path that cannot run on these inputs    */
    DS4G_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed      */
    DS4G_ERR_TIMEOUT = 7,      /* a bounded device-side wait expired (device status) */
    DS4G_ERR_RANGE = 8         /* device status: an MXFP4 block scale outside
                                  2^-23 .. 2^13 met on the tensor-core kernels,
                                  whose fp16 operands then rounded weights     */
} ds4g_status;

typedef enum ds4g_score {
    DS4G_SCORE_SOFTMAX = 0,    /* w_i = exp(l_i - l_max) / sum_j exp(l_j - l_max)  */
    DS4G_SCORE_SIGMOID = 1     /* w_i = sigma(l_i) / sum_j sigma(l_j)              */
} ds4g_score;

typedef enum ds4g_format {
    DS4G_FMT_Q2K = 0,          /* 84-byte Q2_K super-blocks                         */
    DS4G_FMT_CB2 = 1,          /* 70-byte codebook-2-bit super-blocks               */
    DS4G_FMT_Q4K = 2,          /* 144-byte Q4_K super-blocks (gate/up or down)      */
    DS4G_FMT_Q5K = 3,          /* 176-byte Q5_K super-blocks (gate/up or down)      */
    DS4G_FMT_Q6K = 4,          /* 210-byte Q6_K super-blocks (down only)            */
    DS4G_FMT_MXFP4 = 5         /* MXFP4: 17-byte blocks of 32 weights (gate/up, down),
                                  counted in 136-byte units of 256 weights          */
} ds4g_format;

typedef enum ds4g_dtype {
    DS4G_F32 = 0,
    DS4G_F16 = 1,
    DS4G_BF16 = 2
} ds4g_dtype;

/* ds4g_moe_desc.flags */
enum {
    DS4G_FORCE_GEMV = 1,       /* every expert segment on the decode (GEMV) kernels   */
    DS4G_FORCE_TC = 2,         /* every expert segment on the tensor-core kernels     */
    DS4G_DEBUG_STALL = 256     /* test hook: the copy producers of the decode and
                                  tensor-core kernels issue nothing, so their
                                  consumers' bounded waits (2 ms in this mode)
                                  expire and the workspace status word reads
                                  DS4G_ERR_TIMEOUT; y is garbage                    */
};

/* Limits checked by the entry points. */
#define DS4G_MAX_EXPERTS 256
#define DS4G_MAX_TOPK 8
#define DS4G_MAX_TOKENS 65536
#define DS4G_MAX_HIDDEN 32768
#define DS4G_MAX_INTER 32768

/*
 * One routed-MoE layer.  Weight tensors are expert-major: expert e of W_gate
 * starts at w_gate + e * gate_up_expert_stride (bytes), and so on.
 *   W_gate[e], W_up[e]: [inter rows x hidden], quantized along hidden.
 *   W_down[e]:          [hidden rows x inter], quantized along inter
 *                       (ceil(inter/256) blocks per row; columns >= inter
 *                       are padding and are ignored).
 * Requirements (else DS4G_ERR_SHAPE / DS4G_ERR_LAYOUT):
 *   hidden % 256 == 0, 256 <= hidden <= DS4G_MAX_HIDDEN;
 *   1 <= inter <= DS4G_MAX_INTER; 1 <= n_experts <= 256;
 *   1 <= top_k <= min(8, n_experts);
 *   row_bytes >= ceil(K/256) * block_bytes and a multiple of 4 (Q2_K,
 *   Q4_K, Q5_K, MXFP4) or 2 (codebook, Q6_K);
 *   expert strides >= rows * row_bytes and multiples of 16;
 *   w_gate, w_up, w_down 16-byte aligned;
 *   DS4G_FORCE_TC additionally needs row_bytes % 16 == 0.
 * tc_min_tokens: the per-segment split of calls that take the tensor-core
 * kernels.  0 (the default): every expert segment runs on them.  N > 0:
 * segments of fewer than N tokens run on the GEMV kernels instead, in the
 * same call (the tensor-core kernels take the others; both write the same
 * per-assignment buffer, summed in slot order as usual).  Calls that take
 * the decode or GEMV kernels as a whole ignore it (see "Path" under
 * ds4g_moe_forward).
 * format / down_format: the block format of W_gate and W_up / of W_down.
 * The shipping mix of the ds4 weights is DS4G_FMT_CB2 / DS4G_FMT_Q2K
 * (IQ2_XXS up/gate, Q2_K down: ds4 README mirror, "Model Weights").  Set
 * both; the codebook is required when either is DS4G_FMT_CB2.  The routed
 * higher-bit formats of the same page ("Model Weights": gate/up in Q2_K,
 * Q4_K or Q5_K, down in Q2_K, Q4_K, Q5_K or Q6_K) are accepted with those
 * roles: format in {Q2K, CB2, Q4K, Q5K, MXFP4}, down_format in {Q2K, CB2,
 * Q4K, Q5K, Q6K, MXFP4} (else DS4G_ERR_INVALID).  MXFP4 is the ds4f-mxfp4
 * routed-expert format of the same page.  Every format has a tensor-core
 * dequantizer (see "Path" under ds4g_moe_forward).  MXFP4 weights become
 * exact fp16 operands there while every block scale
 * 2^(e-127) of the call's experts lies in 2^-23 .. 2^13 (any trained weight:
 * |w| from 2^-24 to 49152); a scale outside it (bar e = 255, NaN) on a
 * block with a nonzero code rounds those weights and sets the workspace
 * status word to DS4G_ERR_RANGE (the
 * GEMV kernels, DS4G_FORCE_GEMV, compute such layers in fp32).  Row
 * alignment: rows of Q2_K, Q4_K, Q5_K and MXFP4
 * a multiple of 4 bytes, of codebook and Q6_K blocks a multiple of 2; rows
 * count ceil(K/256) units of the format's bytes per 256 weights.
 * n_slots / expert_slot: where each expert's weights are.  n_slots == 0
 * (expert_slot NULL): expert e's matrices are slot e of the weight tensors.
 * n_slots > 0: the weight tensors hold n_slots expert slots (same row bytes
 * and expert strides) and expert_slot [n_experts] int32 (device, 4-byte
 * aligned) gives the slot of each expert; only the experts a call routes to
 * need a valid slot (0 .. n_slots-1).  A routed expert whose entry is out of
 * range has its weights read from slot 0 instead and the workspace status
 * word reads DS4G_ERR_INVALID (see ds4g_moe_device_status); y is then not
 * valid.  This is how ds4g_expert_cache below runs layers whose experts
 * live in host memory.
 */
typedef struct ds4g_moe_desc {
    int32_t hidden;
    int32_t inter;
    int32_t n_experts;
    int32_t top_k;
    int32_t score;             /* ds4g_score  */
    int32_t format;            /* ds4g_format of W_gate and W_up */
    int32_t flags;
    int32_t tc_min_tokens;
    int32_t down_format;       /* ds4g_format of W_down                          */
    int32_t n_slots;           /* 0, or the expert slots the weight tensors hold */
    const void *w_gate;
    const void *w_up;
    const void *w_down;
    int64_t gate_up_row_bytes;
    int64_t down_row_bytes;
    int64_t gate_up_expert_stride;
    int64_t down_expert_stride;
    const int8_t *codebook;    /* [256 x 8] int8, device; when a matrix is CB2  */
    const int32_t *expert_slot;/* [n_experts] int32, device; when n_slots > 0    */
} ds4g_moe_desc;

/*
 * ds4g_route_topk -- steps 1 and 2 alone.  Passage: the routed experts of
 * the layer (ds4 README mirror, "Model Weights"); the selection order and
 * tie rule are this library's definition (the pages state none).
 *   logits  [T x E] fp32, row-major.
 *   ids     [T x k] int32 out: per token the k largest logits' expert ids in
 *           rank order: larger logit first, equal logits -> lower id first,
 *           a NaN logit ranks as -infinity.
 *   weights [T x k] fp32 out: softmax over the k selected logits, or sigmoid
 *           of each selected logit divided by their sum (`score`).
 *   counts  [E] int32 out (nullable): assignments per expert.
 *   offsets [E+1] int32 out (nullable): exclusive prefix sum of counts.
 *   perm    [T*k] int32 out (nullable): assignment indices a = t*k + i grouped
 *           by expert (segment e = perm[offsets[e] .. offsets[e+1]-1]),
 *           ascending t inside each segment.
 * Errors: DS4G_ERR_INVALID (null ids/weights/logits, T < 0, E < 1, E > 256,
 * k < 1, k > min(8, E), bad score); DS4G_ERR_SHAPE (T > DS4G_MAX_TOKENS);
 * DS4G_ERR_CUDA.  T == 0 is a no-op (counts/offsets still written as zero).
 */
DS4G_API ds4g_status ds4g_route_topk(const float *logits, int32_t T, int32_t E, int32_t k,
                            int32_t score, int32_t *ids, float *weights,
                            int32_t *counts, int32_t *offsets, int32_t *perm,
                            void *stream);

/*
 * ds4g_q2k_dequant -- passage: Q2_K routed experts (ds4 README mirror,
 * "Model Weights") in the GGUF layout kept from llama.cpp (same page,
 * "Acknowledgements to llama.cpp and GGML").
 * n_blocks consecutive Q2_K super-blocks (84 bytes each,
 * `blocks` 4-byte aligned) to n_blocks * 256 values of out_dtype in `out`
 * (16-byte aligned).  fp32 output is exactly the block definition above
 * (both products are exact; one rounding in the subtraction); fp16 / bf16
 * output is that fp32 value rounded to nearest even.
 * Errors: DS4G_ERR_INVALID (null pointer, n_blocks < 0, bad dtype);
 * DS4G_ERR_LAYOUT (alignment); DS4G_ERR_CUDA.  n_blocks == 0 is a no-op.
 */
DS4G_API ds4g_status ds4g_q2k_dequant(const void *blocks, int64_t n_blocks, void *out,
                             int32_t out_dtype, void *stream);

/*
 * ds4g_q4k_dequant / ds4g_q5k_dequant / ds4g_q6k_dequant -- passage: the
 * routed expert formats Q4_K, Q5_K (gate/up and down) and Q6_K (down) (ds4
 * README mirror, "Model Weights") in the GGUF K-quant layouts kept from
 * llama.cpp (same page, "Acknowledgements to llama.cpp and GGML"):
 *   Q4_K, 144 bytes: d, dmin (fp16), 12 bytes of packed 6-bit scales and
 *         mins of eight 32-weight sub-blocks, 128 bytes of 4-bit quants;
 *         w = d * sc_s * q - dmin * m_s;
 *   Q5_K, 176 bytes: as Q4_K plus 32 bytes of fifth bits (bit s of byte l
 *         for weight 32s + l) before the low nibbles;
 *   Q6_K, 210 bytes: 128 bytes of low nibbles, 64 bytes of top two bits,
 *         16 int8 scales of 16-weight sub-blocks, d (fp16);
 *         w = d * scale * (q6 - 32).
 * n_blocks consecutive super-blocks (`blocks` 4-byte aligned for Q4_K /
 * Q5_K, 2-byte aligned for Q6_K) to n_blocks * 256 values of out_dtype in
 * `out` (16-byte aligned).  fp32 output is exactly the definition (every
 * product is exact in fp32; Q4_K / Q5_K round once, in the subtraction);
 * fp16 / bf16 output is that value rounded to nearest even.
 * Errors as ds4g_q2k_dequant.
 */
DS4G_API ds4g_status ds4g_q4k_dequant(const void *blocks, int64_t n_blocks, void *out,
                             int32_t out_dtype, void *stream);
DS4G_API ds4g_status ds4g_q5k_dequant(const void *blocks, int64_t n_blocks, void *out,
                             int32_t out_dtype, void *stream);
DS4G_API ds4g_status ds4g_q6k_dequant(const void *blocks, int64_t n_blocks, void *out,
                             int32_t out_dtype, void *stream);

/*
 * ds4g_mxfp4_dequant -- passage: MXFP4 routed experts (ds4 README mirror,
 * "Model Weights": the ds4f-mxfp4 download keeps DeepSeek's released MXFP4
 * routed-expert weights), read as OCP microscaling FP4 in its GGUF block:
 * 17 bytes per 32 weights, byte 0 an E8M0 scale e (2^(e-127); 255 is NaN),
 * bytes 1..16 the E2M1 codes (weight i in the low nibble of byte 1 + i,
 * weight i + 16 in its high nibble; bit 3 the sign, bits 0..2 the
 * magnitude 0, 0.5, 1, 1.5, 2, 3, 4, 6); w = 2^(e-127) * value.
 * n_blocks counts units of eight blocks (136 bytes, 256 weights); `blocks`
 * is 4-byte aligned, `out` 16-byte aligned.  fp32 output is
 * exactly the definition (a power of two times a 3-bit value: exact unless
 * outside fp32's range); fp16 / bf16 output is it rounded to nearest even.
 * Errors as ds4g_q2k_dequant.
 */
DS4G_API ds4g_status ds4g_mxfp4_dequant(const void *blocks, int64_t n_blocks, void *out,
                               int32_t out_dtype, void *stream);

/*
 * ds4g_cb2_dequant -- passage: the IQ2_XXS half of the IQ2_XXS / Q2_K expert
 * mix (DwarfStar 4 on aiany.app, "What Sets It Apart"; ds4 README mirror,
 * "Model Weights"), as the codebook-2-bit stand-in described at the top.
 * n_blocks consecutive codebook-2-bit super-blocks (70
 * bytes each, `blocks` 2-byte aligned) with a [256 x 8] int8 device codebook
 * to n_blocks * 256 values of out_dtype (16-byte aligned).  fp32 output is
 * exact; fp16 / bf16 output is the fp32 value rounded to nearest even.
 * Errors as ds4g_q2k_dequant, plus DS4G_ERR_INVALID for a null codebook.
 */
DS4G_API ds4g_status ds4g_cb2_dequant(const void *blocks, int64_t n_blocks, const int8_t *codebook,
                             void *out, int32_t out_dtype, void *stream);

/*
 * ds4g_moe_workspace_bytes -- no counterpart on the pages (sizing helper of
 * ds4g_moe_forward).  Bytes of device workspace ds4g_moe_forward
 * (and ds4g_moe_forward_host) need for this layer and T tokens; 0 when the
 * descriptor or T is invalid.  The workspace must be 256-byte aligned.
 */
DS4G_API size_t ds4g_moe_workspace_bytes(const ds4g_moe_desc *desc, int32_t T);

/*
 * ds4g_moe_forward -- the whole layer, steps 1-4.  Passage: the routed-MoE
 * experts run micro-batched in decode and prefill on CUDA (ds4 README mirror,
 * "So, what can I do with this software?" and "Model Weights").
 *   x       [T x hidden] bf16 (uint16 bits), 16-byte aligned.
 *   logits  [T x n_experts] fp32, 4-byte aligned.
 *   y       [T x hidden] fp32 out, 16-byte aligned; overwritten.
 *   workspace / ws_bytes: device scratch of at least
 *           ds4g_moe_workspace_bytes(desc, T) bytes, 256-byte aligned.  After
 *           the call it holds the routing of this call (see
 *           ds4g_moe_routing_view).
 * Path (one per call): layers whose row_bytes are multiples of 16 (any
 * formats; Q6_K W_down rows: inter padded to a multiple of 2048; MXFP4: an
 * even number of 136-byte units) run the tensor-core kernels, except Q2_K
 * layers with inter % 16 == 0 at T <= 3, which run the decode kernels.  Q2_K
 * layers that the tensor-core kernels cannot take run the decode kernels up
 * to T = 32 (mma.sync up to 8 vectors, tcgen05 from 9 to 32, the latter with
 * hidden % 128 == 0).  All others run the GEMV kernels.  DS4G_FORCE_TC forces the tensor-core kernels
 * and DS4G_FORCE_GEMV rules them out.
 * Errors: DS4G_ERR_INVALID, DS4G_ERR_SHAPE, DS4G_ERR_LAYOUT,
 * DS4G_ERR_WORKSPACE, DS4G_ERR_UNSUPPORTED (a forced path that cannot run),
 * DS4G_ERR_CUDA.  T == 0 is a no-op.
 */
DS4G_API ds4g_status ds4g_moe_forward(const ds4g_moe_desc *desc, const uint16_t *x,
                             const float *logits, int32_t T, float *y,
                             void *workspace, size_t ws_bytes, void *stream);

/*
 * ds4g_moe_forward_host -- no counterpart on the pages (a convenience for
 * callers whose activations live in host memory).
 * ds4g_moe_forward with HOST activations, logits
 * and output (weights stay on the device, in desc).  Copies x and logits to
 * the workspace, runs the layer, copies y back and synchronizes `stream`
 * before returning.  Host buffers should be pinned (cudaHostAlloc) for full
 * copy bandwidth; pageable memory works but is slower.
 * Errors: as ds4g_moe_forward.
 */
DS4G_API ds4g_status ds4g_moe_forward_host(const ds4g_moe_desc *desc, const uint16_t *x_host,
                                  const float *logits_host, int32_t T, float *y_host,
                                  void *workspace, size_t ws_bytes, void *stream);

/*
 * ds4g_moe_routing_view -- no counterpart on the pages (exposes steps 1-2 of
 * the last ds4g_moe_forward for checking).  Device pointers, inside a workspace last used by
 * ds4g_moe_forward(desc, ..., T, ...), to that call's routing results:
 * ids [T x k] int32, weights [T x k] fp32, counts [E] int32,
 * offsets [E+1] int32, perm [T*k] int32 (same meaning as ds4g_route_topk).
 * Any output pointer may be NULL.  Pure host arithmetic; launches nothing.
 * Errors: DS4G_ERR_INVALID, DS4G_ERR_WORKSPACE.
 */
DS4G_API ds4g_status ds4g_moe_routing_view(const ds4g_moe_desc *desc, int32_t T, void *workspace,
                                  size_t ws_bytes, int32_t **ids, float **weights,
                                  int32_t **counts, int32_t **offsets, int32_t **perm);

/*
 * ds4g_moe_forward_phased -- no counterpart on the pages (measurement aid).
 * ds4g_moe_forward that also records caller-created
 * CUDA events (cudaEvent_t, passed as void*) on `stream` at the phase
 * boundaries, for per-kernel timing:
 *   events[0] before routing,          events[1] after routing,
 *   events[2] after gate/up + SiLU,    events[3] after the down projection,
 *   events[4] after the weighted combine.
 * n_events must be 5.  Errors: as ds4g_moe_forward, plus DS4G_ERR_INVALID
 * for a null or short event array.
 */
DS4G_API ds4g_status ds4g_moe_forward_phased(const ds4g_moe_desc *desc, const uint16_t *x,
                                             const float *logits, int32_t T, float *y,
                                             void *workspace, size_t ws_bytes, void *stream,
                                             void *const *events, int32_t n_events);

/*
 * ds4g_moe_forward_launches -- no counterpart on the pages (measurement
 * aid).  Number of kernel launches one
 * ds4g_moe_forward(desc, ..., T, ...) call enqueues (0 for an invalid
 * descriptor or T == 0).  Pure host arithmetic.
 */
DS4G_API int32_t ds4g_moe_forward_launches(const ds4g_moe_desc *desc, int32_t T);

/*
 * ds4g_moe_device_status -- no counterpart on the pages (failure detection
 * of this library).  The device status word of the last
 * ds4g_moe_forward on this workspace (the first problem a kernel recorded):
 * DS4G_OK; DS4G_ERR_TIMEOUT when a bounded wait inside a kernel expired (the
 * kernel then returned early and y is not valid); DS4G_ERR_INVALID when a
 * routed expert's slot map entry was out of range (y not valid);
 * DS4G_ERR_RANGE when an MXFP4 block scale beyond fp16 was rounded on the
 * tensor-core kernels (y computed, those weights inexact).  Synchronizes
 * `stream`.  Errors: DS4G_ERR_INVALID, DS4G_ERR_WORKSPACE, DS4G_ERR_CUDA.
 */
DS4G_API ds4g_status ds4g_moe_device_status(const ds4g_moe_desc *desc, int32_t T,
                                            const void *workspace, size_t ws_bytes,
                                            int32_t *status_out, void *stream);

/*
 * ds4g_moe_forward_noalloc -- ds4g_moe_forward for callers that cannot
 * allocate device memory, so cannot hand the library a workspace: a plugin
 * inside a host runtime that owns every device allocation and gives its
 * plugins no allocator, or a serving loop that must not call cudaMalloc
 * (which can synchronize the device) once it is running.  This entry point
 * has no counterpart on the pages; it is a convenience of this library.
 *
 * Scratch comes from one static device array of DS4G_NOALLOC_SCRATCH_BYTES
 * per GPU, held by every GPU that loads the library until the process exits.
 * Calls whose workspace (ds4g_moe_workspace_bytes(desc, T)) would exceed it
 * return DS4G_ERR_WORKSPACE before launching anything; 32 MiB covers decode
 * up to T = 32 tokens at hidden 7168 / inter 2048 / 256 experts / top-8
 * (a 23.5 MiB workspace).
 * x, logits, y: as ds4g_moe_forward (device pointers owned by the caller).
 *
 * The first call on a device looks up the array's device address (a CUDA
 * runtime query, no allocation); make that first call before any stream
 * capture.  No call allocates or frees device memory.  Every call on a GPU
 * shares the one array and leaves its contents behind; the kernels write
 * every scratch value they later read (the status word is reset by the first
 * kernel of each call), so nothing needs clearing between calls.  Calls that
 * overlap on the same GPU (other streams, other host threads) race on the
 * array: serialize them.  ds4g_moe_routing_view and ds4g_moe_device_status do
 * not apply to this entry point; ds4g_moe_noalloc_status reads its status
 * word.  The array's address is looked up once per device and kept for the
 * life of the process: after a cudaDeviceReset it is stale, so a process
 * that resets a device must not call this entry point on it again.
 * Errors: as ds4g_moe_forward.
 */
#define DS4G_NOALLOC_SCRATCH_BYTES (32u << 20)
DS4G_API ds4g_status ds4g_moe_forward_noalloc(const ds4g_moe_desc *desc, const uint16_t *x,
                                              const float *logits, int32_t T, float *y,
                                              void *stream);

/* Static text for a status code ("ok", "invalid argument", ...). */
DS4G_API const char *ds4g_status_string(ds4g_status status);

/*
 * ds4g_expert_cache -- a device-resident cache of routed experts whose
 * weights live in host memory.  Passage: routed MoE experts streamed from an
 * in-memory cache on cache misses, with configurable expert-cache budgets
 * (opensourcealternatives.to, FAQ; DwarfStar 4 on aiany.app, "What Sets It
 * Apart"; SSD streaming of the routed experts in the ds4 README mirror).
 * Here the backing store is host memory and a miss is an asynchronous
 * host-to-device copy of the expert's three matrices.
 *
 * ds4g_expert_cache_create: `host_desc` describes the layer with w_gate,
 * w_up and w_down in host memory (page-locked, e.g. cudaHostAlloc, so that
 * the copies are asynchronous; 16-byte aligned) and n_slots = 0; codebook,
 * when used, is a device pointer as usual.  The cache allocates, on the
 * current device, n_slots expert slots (n_slots * (2 * gate_up_expert_stride
 * + down_expert_stride) bytes) and the expert-to-slot map; this entry point
 * and ds4g_expert_cache_destroy are the library's only device allocations.
 * Errors: DS4G_ERR_INVALID (descriptor, null out, n_slots < top_k or
 * n_slots > n_experts, host_desc->n_slots != 0); the descriptor errors of
 * ds4g_moe_forward; DS4G_ERR_CUDA (allocation).
 * ds4g_expert_cache_workspace_bytes: device workspace of a forward of T
 * tokens (0 when T is invalid).
 * ds4g_expert_cache_forward: one layer call, arguments as ds4g_moe_forward
 * (device x, logits, y and workspace).  It routes on the device, reads back
 * which experts the call uses (synchronizing `stream`), uploads the missing
 * ones into the least recently used slots that this call does not use
 * (three cudaMemcpyAsync per expert on `stream`), uploads the map, then runs
 * the layer on the slots: y is bit-identical to ds4g_moe_forward on a
 * device-resident copy of the weights.  The uploads precede the layer on
 * `stream` (the fused layer needs every routed expert resident before it
 * starts).  Calls on one cache must not overlap (one stream, or
 * synchronized).  Errors: those of ds4g_moe_forward, plus
 * DS4G_ERR_UNSUPPORTED when the call routes to more distinct experts than
 * the cache has slots (nothing runs after the routing).
 * ds4g_expert_cache_stats: expert hits, misses (uploads) and bytes uploaded
 * since creation (any out pointer may be NULL).
 * ds4g_expert_cache_destroy: frees the slots (synchronizes the device).
 */
typedef struct ds4g_expert_cache ds4g_expert_cache;
DS4G_API ds4g_status ds4g_expert_cache_create(const ds4g_moe_desc *host_desc, int32_t n_slots,
                                              ds4g_expert_cache **out);
DS4G_API size_t ds4g_expert_cache_workspace_bytes(const ds4g_expert_cache *cache, int32_t T);
DS4G_API ds4g_status ds4g_expert_cache_forward(ds4g_expert_cache *cache, const uint16_t *x,
                                               const float *logits, int32_t T, float *y,
                                               void *workspace, size_t ws_bytes, void *stream);
DS4G_API ds4g_status ds4g_expert_cache_stats(const ds4g_expert_cache *cache, int64_t *hits,
                                             int64_t *misses, int64_t *bytes_uploaded);
DS4G_API void ds4g_expert_cache_destroy(ds4g_expert_cache *cache);

/*
 * ds4g_moe_noalloc_status -- no counterpart on the pages (failure detection of
 * this library).  The device status word of the last
 * ds4g_moe_forward_noalloc of this layer and T on the current device:
 * DS4G_OK, DS4G_ERR_TIMEOUT (a bounded wait expired) or DS4G_ERR_INVALID (a
 * routed expert's slot was out of range).  Synchronizes `stream`.  Errors:
 * DS4G_ERR_INVALID, the descriptor errors of ds4g_moe_forward,
 * DS4G_ERR_WORKSPACE (the layer does not fit the static scratch),
 * DS4G_ERR_CUDA.
 */
DS4G_API ds4g_status ds4g_moe_noalloc_status(const ds4g_moe_desc *desc, int32_t T,
                                             int32_t *status_out, void *stream);

/* DS4G_ABI_VERSION of the loaded library. */
DS4G_API int32_t ds4g_abi_version(void);

/* The cudaError_t behind the calling thread's most recent DS4G_ERR_CUDA
 * (0 when none occurred yet).  Pure host call. */
DS4G_API int32_t ds4g_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DS4G_H */
