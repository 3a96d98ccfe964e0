// ds4g_api.cu -- the C ABI of libds4g: argument validation, the workspace
// plan and the launch sequence of one routed-MoE layer call.  Every entry
// point validates on the host before launching anything and returns a
// ds4g_status; no entry point allocates device memory except the expert
// cache's create (cache.cu).
#include <mutex>

#include "ds4g_common.cuh"

namespace ds4g {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local int g_last_cuda_error = 0;

ds4g_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return DS4G_OK;
    g_last_cuda_error = (int)e;
    return DS4G_ERR_CUDA;
}

std::mutex g_dev_mu;
DeviceInfo g_dev[64];
bool g_dev_ok[64];

}  // namespace

ds4g_status status_from_cuda(cudaError_t e) { return from_cuda(e); }

ds4g_status device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DS4G_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo info{};
        if (cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&info.max_smem_optin,
                                   cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return DS4G_ERR_CUDA;
        g_dev[dev] = info;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return DS4G_OK;
}

ds4g_status make_plan(const ds4g_moe_desc *d, int32_t T, Plan *p)
{
    if (!d || !p) return DS4G_ERR_INVALID;
    if (T < 0) return DS4G_ERR_INVALID;
    if (d->n_experts < 1 || d->n_experts > DS4G_MAX_EXPERTS) return DS4G_ERR_INVALID;
    if (d->top_k < 1 || d->top_k > DS4G_MAX_TOPK || d->top_k > d->n_experts)
        return DS4G_ERR_INVALID;
    if (d->score != DS4G_SCORE_SOFTMAX && d->score != DS4G_SCORE_SIGMOID) return DS4G_ERR_INVALID;
    // routed gate/up: Q2_K, codebook, Q4_K, Q5_K, MXFP4; routed down: also Q6_K
    if (d->format != DS4G_FMT_Q2K && d->format != DS4G_FMT_CB2 && d->format != DS4G_FMT_Q4K &&
        d->format != DS4G_FMT_Q5K && d->format != DS4G_FMT_MXFP4)
        return DS4G_ERR_INVALID;
    if (block_bytes_of(d->down_format) == 0) return DS4G_ERR_INVALID;
    if (d->n_slots < 0 || (d->n_slots == 0) != (d->expert_slot == nullptr))
        return DS4G_ERR_INVALID;
    if ((d->flags & ~(DS4G_FORCE_GEMV | DS4G_FORCE_TC | DS4G_DEBUG_STALL)) != 0)
        return DS4G_ERR_INVALID;
    if ((d->flags & DS4G_FORCE_GEMV) && (d->flags & DS4G_FORCE_TC)) return DS4G_ERR_INVALID;
    if (d->tc_min_tokens < 0) return DS4G_ERR_INVALID;
    if (!d->w_gate || !d->w_up || !d->w_down) return DS4G_ERR_INVALID;
    if ((d->format == DS4G_FMT_CB2 || d->down_format == DS4G_FMT_CB2) && !d->codebook)
        return DS4G_ERR_INVALID;
    if (T > DS4G_MAX_TOKENS) return DS4G_ERR_SHAPE;
    if (d->hidden < kQK || d->hidden > DS4G_MAX_HIDDEN || d->hidden % kQK != 0)
        return DS4G_ERR_SHAPE;
    if (d->inter < 1 || d->inter > DS4G_MAX_INTER) return DS4G_ERR_SHAPE;

    Plan q{};
    q.T = T;
    q.H = d->hidden;
    q.I = d->inter;
    q.E = d->n_experts;
    q.k = d->top_k;
    q.A = T * d->top_k;
    q.I_pad = (d->inter + kQK - 1) / kQK * kQK;
    q.H_blocks = d->hidden / kQK;
    q.I_blocks = q.I_pad / kQK;
    q.gu_block_bytes = block_bytes_of(d->format);
    q.dn_block_bytes = block_bytes_of(d->down_format);

    const int64_t gu_logical = (int64_t)q.H_blocks * q.gu_block_bytes;
    const int64_t dn_logical = (int64_t)q.I_blocks * q.dn_block_bytes;
    // Q2_K, Q4_K and Q5_K rows hold 4-byte aligned blocks, codebook and Q6_K
    // rows 2-byte aligned ones
    const int64_t gu_mult = q.gu_block_bytes % 4 == 0 ? 4 : 2;
    const int64_t dn_mult = q.dn_block_bytes % 4 == 0 ? 4 : 2;
    if (d->gate_up_row_bytes < gu_logical || d->down_row_bytes < dn_logical)
        return DS4G_ERR_LAYOUT;
    if (d->gate_up_row_bytes % gu_mult || d->down_row_bytes % dn_mult) return DS4G_ERR_LAYOUT;
    if (d->gate_up_expert_stride < (int64_t)q.I * d->gate_up_row_bytes ||
        d->down_expert_stride < (int64_t)q.H * d->down_row_bytes)
        return DS4G_ERR_LAYOUT;
    if (d->gate_up_expert_stride % 16 || d->down_expert_stride % 16) return DS4G_ERR_LAYOUT;
    if (!aligned(d->w_gate, 16) || !aligned(d->w_up, 16) || !aligned(d->w_down, 16))
        return DS4G_ERR_LAYOUT;
    if (d->expert_slot && !aligned(d->expert_slot, 4)) return DS4G_ERR_LAYOUT;
    if ((d->flags & DS4G_FORCE_TC) &&
        (d->gate_up_row_bytes % 16 != 0 || d->down_row_bytes % 16 != 0))
        return DS4G_ERR_LAYOUT;

    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    const size_t A = (size_t)q.A;
    q.ids = take(A * 4);
    q.wts = take(A * 4);
    q.counts = take((size_t)q.E * 4);
    q.offsets = take((size_t)(q.E + 1) * 4);
    q.perm = take(A * 4);
    q.slot_pos = take(A * 4);
    q.active = take((size_t)q.E * 4);
    q.meta = take(kMetaWords * 4);
    q.status = take(4);
    q.sync = take((size_t)decode_sync_words(q.E, q.H) * 4);
    q.gpart = take(decode_gpart_bytes(q.A, q.I_pad));
    q.xp = take((size_t)T * q.H * 2);
    q.xs = take((size_t)T * (q.H / 16) * 4);
    q.hp = take(A * q.I_pad * 2);
    q.hs = take(A * (q.I_pad / 16) * 4);
    q.hbuf = take(A * q.I_pad * 4);
    q.yslot = take(A * q.H * 4);
    q.xseg = take(A * q.H * 2);
    q.tiles = take((size_t)tc_max_tiles(q.E, q.A) * 16);
    q.wseg = take(A * 4);
    q.texp = take((size_t)T * 4);
    q.eseg = take(A * 4);
    q.light = take((size_t)q.E * 4);
    q.x_stage = take((size_t)T * q.H * 2);
    q.l_stage = take((size_t)T * q.E * 4);
    q.y_stage = take((size_t)T * q.H * 4);
    q.total = off;
    *p = q;
    return DS4G_OK;
}

namespace {

enum class Path { kDecode, kTensorCore, kGeneral };

// Up to kDecodeOverTcT tokens the Q2_K decode kernels beat the tensor-core
// kernels; from four tokens on the tensor-core kernels win where they apply
// (7168/2048/256/top-8, measured: 0.088 against 0.127 ms at one token, 0.17
// against 0.20 at two, 0.35 against 0.38 at four, 1.48 against 1.86 at 32).
constexpr int kDecodeOverTcT = 3;

// The Q2_K decode kernels up to kDecodeOverTcT tokens, and up to kDecodeMaxT
// where the tensor-core kernels do not apply (mma.sync up to kDecodePreferT,
// tcgen05 above); otherwise the tensor-core kernels for rows of a multiple of
// 16 bytes, in every format; the general kernels where neither applies.
Path choose_path(const ds4g_moe_desc *d, const Plan &p)
{
    if (d->flags & DS4G_FORCE_TC) return Path::kTensorCore;
    const bool decode = decode_path_supported(p, d);
    if (d->flags & DS4G_FORCE_GEMV) return decode ? Path::kDecode : Path::kGeneral;
    const bool tc = tc_path_supported(p, d);
    if (decode && (p.T <= kDecodeOverTcT || !tc)) return Path::kDecode;
    if (tc) return Path::kTensorCore;
    return Path::kGeneral;
}

// Records events[i] (when given) at the phase boundaries of one forward.
struct PhaseEvents {
    cudaEvent_t ev[5];
    bool on;
    cudaError_t mark(int i, cudaStream_t s) const
    {
        return on ? record_phase(ev[i], s) : cudaSuccess;
    }
};

ds4g_status forward_impl(const ds4g_moe_desc *d, const Plan &p, const uint16_t *x,
                         const float *logits, float *y, uint8_t *ws, cudaStream_t s,
                         const PhaseEvents &pe)
{
    DeviceInfo dev;
    ds4g_status st = device_info(&dev);
    if (st != DS4G_OK) return st;
    int32_t *ids = reinterpret_cast<int32_t *>(ws + p.ids);
    float *wts = reinterpret_cast<float *>(ws + p.wts);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + p.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + p.offsets);
    int32_t *perm = reinterpret_cast<int32_t *>(ws + p.perm);
    int32_t *slot_pos = reinterpret_cast<int32_t *>(ws + p.slot_pos);
    int32_t *active = reinterpret_cast<int32_t *>(ws + p.active);
    int32_t *meta = reinterpret_cast<int32_t *>(ws + p.meta);
    int32_t *status = reinterpret_cast<int32_t *>(ws + p.status);
    int32_t *sync = reinterpret_cast<int32_t *>(ws + p.sync);
    __half *xp = reinterpret_cast<__half *>(ws + p.xp);
    float *xs = reinterpret_cast<float *>(ws + p.xs);
    const Path path = choose_path(d, p);
    if (path == Path::kTensorCore && !tc_path_supported(p, d)) return DS4G_ERR_UNSUPPORTED;
    const bool decode = path == Path::kDecode;
    if (pe.mark(0, s) != cudaSuccess) return DS4G_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (!decode)
        e = launch_route(logits, p.T, p.E, p.k, d->score, ids, wts, counts, offsets, perm,
                         slot_pos, active, meta + kMetaActive, nullptr, p.H,
                         xp, xs, status, nullptr, 0, s);
    if (e != cudaSuccess) return from_cuda(e);
    LayerArgs a{};
    a.H = p.H;
    a.I = p.I;
    a.I_pad = p.I_pad;
    a.E = p.E;
    a.k = p.k;
    a.A = p.A;
    a.T = p.T;
    a.gu_format = d->format;
    a.dn_format = d->down_format;
    a.w_gate = static_cast<const uint8_t *>(d->w_gate);
    a.w_up = static_cast<const uint8_t *>(d->w_up);
    a.w_down = static_cast<const uint8_t *>(d->w_down);
    a.gu_row = d->gate_up_row_bytes;
    a.dn_row = d->down_row_bytes;
    a.gu_stride = d->gate_up_expert_stride;
    a.dn_stride = d->down_expert_stride;
    a.wslot = d->n_slots > 0 ? d->expert_slot : nullptr;
    a.n_wslots = d->n_slots > 0 ? d->n_slots : p.E;
    a.status = status;
    a.codebook = d->codebook;
    a.x = x;
    a.wts = wts;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.slot_pos = slot_pos;
    a.active = active;
    a.n_active = meta + kMetaActive;
    a.hbuf = reinterpret_cast<float *>(ws + p.hbuf);
    a.yslot = reinterpret_cast<float *>(ws + p.yslot);
    a.y = y;
    TcBufs tb{reinterpret_cast<__half *>(ws + p.xseg), reinterpret_cast<__half *>(ws + p.hp),
              reinterpret_cast<int32_t *>(ws + p.tiles), meta + kMetaTiles, status,
              reinterpret_cast<float *>(ws + p.wseg), reinterpret_cast<int32_t *>(ws + p.texp),
              reinterpret_cast<int32_t *>(ws + p.eseg), reinterpret_cast<int32_t *>(ws + p.light),
              meta + kMetaLight, d->tc_min_tokens};
    // the activation gather of the tensor-core path belongs to the routing phase
    if (path == Path::kTensorCore && (e = launch_tc_prep(a, tb, dev, s)) != cudaSuccess)
        return from_cuda(e);
    if (!decode && pe.mark(1, s) != cudaSuccess) return DS4G_ERR_CUDA;
    const bool stall = (d->flags & DS4G_DEBUG_STALL) != 0;
    const uint64_t wait_ns = stall ? kStallWaitNs : kWaitNs;
    if (decode) {
        DecodeBufs b{logits, ids, d->score, xp, xs, reinterpret_cast<__half *>(ws + p.hp),
                     reinterpret_cast<float *>(ws + p.hs), status, sync,
                     reinterpret_cast<float *>(ws + p.gpart),
                     reinterpret_cast<int32_t *>(ws + p.texp)};
        return from_cuda(launch_decode_path(a, b, dev, s, pe.on ? pe.ev : nullptr, wait_ns,
                                            stall));
    }
    if (path == Path::kTensorCore)
        return from_cuda(launch_tc_path(a, tb, dev, s, pe.on ? pe.ev : nullptr, wait_ns, stall));
    return from_cuda(launch_gemv_path(a, dev, s, pe.on ? pe.ev : nullptr));
}

int32_t route_launches(int32_t T) { return T <= kRouteSmallT ? 1 : 2; }

ds4g_status check_forward_args(const ds4g_moe_desc *d, const void *x, const void *logits,
                               const void *y, void *ws, size_t ws_bytes, int32_t T, Plan *p)
{
    ds4g_status st = make_plan(d, T, p);
    if (st != DS4G_OK) return st;
    if (T == 0) return DS4G_OK;
    if (!x || !logits || !y || !ws) return DS4G_ERR_INVALID;
    if (!aligned(ws, kAlign)) return DS4G_ERR_WORKSPACE;
    if (ws_bytes < p->total) return DS4G_ERR_WORKSPACE;
    return DS4G_OK;
}

}  // namespace
}  // namespace ds4g

using namespace ds4g;

extern "C" {

ds4g_status ds4g_route_topk(const float *logits, int32_t T, int32_t E, int32_t k, int32_t score,
                            int32_t *ids, float *weights, int32_t *counts, int32_t *offsets,
                            int32_t *perm, void *stream)
{
    if (!logits || !ids || !weights) return DS4G_ERR_INVALID;
    if (T < 0 || E < 1 || E > DS4G_MAX_EXPERTS || k < 1 || k > DS4G_MAX_TOPK || k > E)
        return DS4G_ERR_INVALID;
    if (score != DS4G_SCORE_SOFTMAX && score != DS4G_SCORE_SIGMOID) return DS4G_ERR_INVALID;
    if (T > DS4G_MAX_TOKENS) return DS4G_ERR_SHAPE;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(weights, 4) ||
        !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4))
        return DS4G_ERR_LAYOUT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(launch_route(logits, T, E, k, score, ids, weights, counts, offsets, perm,
                                  nullptr, nullptr, nullptr, nullptr, 0, nullptr, nullptr, nullptr,
                                  nullptr, 0, s));
}

ds4g_status ds4g_q2k_dequant(const void *blocks, int64_t n_blocks, void *out, int32_t out_dtype,
                             void *stream)
{
    if (n_blocks < 0) return DS4G_ERR_INVALID;
    if (out_dtype != DS4G_F32 && out_dtype != DS4G_F16 && out_dtype != DS4G_BF16)
        return DS4G_ERR_INVALID;
    if (n_blocks == 0) return DS4G_OK;
    if (!blocks || !out) return DS4G_ERR_INVALID;
    if (!aligned(blocks, 4) || !aligned(out, 16)) return DS4G_ERR_LAYOUT;
    return from_cuda(launch_q2k_dequant(static_cast<const uint8_t *>(blocks), n_blocks, out,
                                        out_dtype, static_cast<cudaStream_t>(stream)));
}

namespace {
ds4g_status kquant_dequant(int fmt, const void *blocks, int64_t n_blocks, void *out,
                           int32_t out_dtype, void *stream)
{
    if (n_blocks < 0) return DS4G_ERR_INVALID;
    if (out_dtype != DS4G_F32 && out_dtype != DS4G_F16 && out_dtype != DS4G_BF16)
        return DS4G_ERR_INVALID;
    if (n_blocks == 0) return DS4G_OK;
    if (!blocks || !out) return DS4G_ERR_INVALID;
    // every block of a 4-byte aligned Q4_K / Q5_K array is 4-byte aligned, and
    // so is every 136-byte MXFP4 unit; Q6_K blocks (210 bytes) only 2-byte
    const size_t balign = fmt == DS4G_FMT_Q6K ? 2 : 4;
    if (!aligned(blocks, balign) || !aligned(out, 16)) return DS4G_ERR_LAYOUT;
    return from_cuda(launch_kquant_dequant(fmt, static_cast<const uint8_t *>(blocks), n_blocks, out,
                                           out_dtype, static_cast<cudaStream_t>(stream)));
}
}  // namespace

ds4g_status ds4g_q4k_dequant(const void *blocks, int64_t n_blocks, void *out, int32_t out_dtype,
                             void *stream)
{
    return kquant_dequant(DS4G_FMT_Q4K, blocks, n_blocks, out, out_dtype, stream);
}

ds4g_status ds4g_q5k_dequant(const void *blocks, int64_t n_blocks, void *out, int32_t out_dtype,
                             void *stream)
{
    return kquant_dequant(DS4G_FMT_Q5K, blocks, n_blocks, out, out_dtype, stream);
}

ds4g_status ds4g_q6k_dequant(const void *blocks, int64_t n_blocks, void *out, int32_t out_dtype,
                             void *stream)
{
    return kquant_dequant(DS4G_FMT_Q6K, blocks, n_blocks, out, out_dtype, stream);
}

ds4g_status ds4g_mxfp4_dequant(const void *blocks, int64_t n_blocks, void *out, int32_t out_dtype,
                               void *stream)
{
    return kquant_dequant(DS4G_FMT_MXFP4, blocks, n_blocks, out, out_dtype, stream);
}

ds4g_status ds4g_cb2_dequant(const void *blocks, int64_t n_blocks, const int8_t *codebook,
                             void *out, int32_t out_dtype, void *stream)
{
    if (n_blocks < 0) return DS4G_ERR_INVALID;
    if (out_dtype != DS4G_F32 && out_dtype != DS4G_F16 && out_dtype != DS4G_BF16)
        return DS4G_ERR_INVALID;
    if (n_blocks == 0) return DS4G_OK;
    if (!blocks || !out || !codebook) return DS4G_ERR_INVALID;
    if (!aligned(blocks, 2) || !aligned(out, 16)) return DS4G_ERR_LAYOUT;
    return from_cuda(launch_cb2_dequant(static_cast<const uint8_t *>(blocks), n_blocks, codebook,
                                        out, out_dtype, static_cast<cudaStream_t>(stream)));
}

size_t ds4g_moe_workspace_bytes(const ds4g_moe_desc *desc, int32_t T)
{
    Plan p;
    if (make_plan(desc, T, &p) != DS4G_OK) return 0;
    return p.total;
}

ds4g_status ds4g_moe_forward(const ds4g_moe_desc *desc, const uint16_t *x, const float *logits,
                             int32_t T, float *y, void *workspace, size_t ws_bytes, void *stream)
{
    Plan p;
    ds4g_status st = check_forward_args(desc, x, logits, y, workspace, ws_bytes, T, &p);
    if (st != DS4G_OK || T == 0) return st;
    if (!aligned(x, 16) || !aligned(logits, 4) || !aligned(y, 16)) return DS4G_ERR_LAYOUT;
    return forward_impl(desc, p, x, logits, y, static_cast<uint8_t *>(workspace),
                        static_cast<cudaStream_t>(stream), PhaseEvents{{}, false});
}

ds4g_status ds4g_moe_forward_phased(const ds4g_moe_desc *desc, const uint16_t *x,
                                    const float *logits, int32_t T, float *y, void *workspace,
                                    size_t ws_bytes, void *stream, void *const *events,
                                    int32_t n_events)
{
    Plan p;
    ds4g_status st = check_forward_args(desc, x, logits, y, workspace, ws_bytes, T, &p);
    if (st != DS4G_OK || T == 0) return st;
    if (!events || n_events != 5) return DS4G_ERR_INVALID;
    PhaseEvents pe{};
    pe.on = true;
    for (int i = 0; i < 5; ++i) {
        if (!events[i]) return DS4G_ERR_INVALID;
        pe.ev[i] = static_cast<cudaEvent_t>(events[i]);
    }
    if (!aligned(x, 16) || !aligned(logits, 4) || !aligned(y, 16)) return DS4G_ERR_LAYOUT;
    return forward_impl(desc, p, x, logits, y, static_cast<uint8_t *>(workspace),
                        static_cast<cudaStream_t>(stream), pe);
}

int32_t ds4g_moe_forward_launches(const ds4g_moe_desc *desc, int32_t T)
{
    Plan p;
    if (T <= 0 || make_plan(desc, T, &p) != DS4G_OK) return 0;
    const Path path = choose_path(desc, p);
    if (path == Path::kDecode) return 2;     // reset/convert, fused layer kernel
    if (path == Path::kTensorCore && !tc_path_supported(p, desc)) return 0;   // refused
    return route_launches(T) +
           (path == Path::kDecode       ? 0
            : path == Path::kTensorCore ? kTcPathLaunches + (desc->tc_min_tokens > 0 ? kSplitLaunches : 0)
                                        : gemv_path_launches(p));
}

ds4g_status ds4g_moe_forward_host(const ds4g_moe_desc *desc, const uint16_t *x_host,
                                  const float *logits_host, int32_t T, float *y_host,
                                  void *workspace, size_t ws_bytes, void *stream)
{
    Plan p;
    ds4g_status st = check_forward_args(desc, x_host, logits_host, y_host, workspace, ws_bytes, T,
                                        &p);
    if (st != DS4G_OK || T == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint16_t *x = reinterpret_cast<uint16_t *>(ws + p.x_stage);
    float *lg = reinterpret_cast<float *>(ws + p.l_stage);
    float *y = reinterpret_cast<float *>(ws + p.y_stage);
    const size_t xb = (size_t)T * p.H * 2, lb = (size_t)T * p.E * 4, yb = (size_t)T * p.H * 4;
    if (cudaMemcpyAsync(x, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DS4G_ERR_CUDA;
    if (cudaMemcpyAsync(lg, logits_host, lb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DS4G_ERR_CUDA;
    st = forward_impl(desc, p, x, lg, y, ws, s, PhaseEvents{{}, false});
    if (st != DS4G_OK) return st;
    if (cudaMemcpyAsync(y_host, y, yb, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return DS4G_ERR_CUDA;
    return from_cuda(cudaStreamSynchronize(s));
}

ds4g_status ds4g_moe_routing_view(const ds4g_moe_desc *desc, int32_t T, void *workspace,
                                  size_t ws_bytes, int32_t **ids, float **weights,
                                  int32_t **counts, int32_t **offsets, int32_t **perm)
{
    Plan p;
    ds4g_status st = make_plan(desc, T, &p);
    if (st != DS4G_OK) return st;
    if (!workspace) return DS4G_ERR_INVALID;
    if (!aligned(workspace, kAlign) || ws_bytes < p.total) return DS4G_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (ids) *ids = reinterpret_cast<int32_t *>(ws + p.ids);
    if (weights) *weights = reinterpret_cast<float *>(ws + p.wts);
    if (counts) *counts = reinterpret_cast<int32_t *>(ws + p.counts);
    if (offsets) *offsets = reinterpret_cast<int32_t *>(ws + p.offsets);
    if (perm) *perm = reinterpret_cast<int32_t *>(ws + p.perm);
    return DS4G_OK;
}

ds4g_status ds4g_moe_device_status(const ds4g_moe_desc *desc, int32_t T, const void *workspace,
                                   size_t ws_bytes, int32_t *status_out, void *stream)
{
    Plan p;
    ds4g_status st = make_plan(desc, T, &p);
    if (st != DS4G_OK) return st;
    if (!workspace || !status_out) return DS4G_ERR_INVALID;
    if (!aligned(workspace, kAlign) || ws_bytes < p.total) return DS4G_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, static_cast<const uint8_t *>(workspace) + p.status, 4,
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DS4G_ERR_CUDA;
    *status_out = v;
    return DS4G_OK;
}

const char *ds4g_status_string(ds4g_status status)
{
    switch (status) {
    case DS4G_OK: return "ok";
    case DS4G_ERR_INVALID: return "invalid argument";
    case DS4G_ERR_SHAPE: return "unsupported shape";
    case DS4G_ERR_LAYOUT: return "misaligned pointer or unusable stride";
    case DS4G_ERR_WORKSPACE: return "workspace misaligned or too small";
    case DS4G_ERR_UNSUPPORTED: return "forced path not possible for these inputs";
    case DS4G_ERR_CUDA: return "CUDA error";
    case DS4G_ERR_TIMEOUT: return "device-side wait timed out";
    case DS4G_ERR_RANGE: return "MXFP4 block scale outside the tensor-core kernels' exact fp16 range";
    }
    return "unknown status";
}

int32_t ds4g_abi_version(void) { return DS4G_ABI_VERSION; }

int32_t ds4g_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward without a caller-provided workspace (ds4g_moe_forward_noalloc).
// The scratch is one file-scope device array per GPU.  Host code must not use
// the array's name as a device address; it asks the runtime for the address
// once per device and hands that pointer to the kernels.
// ---------------------------------------------------------------------------
namespace ds4g {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[DS4G_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];

// Device address of the scratch array on the current device, looked up on
// the first call for that device.
ds4g_status noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DS4G_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return from_cuda(e);
        if (!p) return DS4G_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return DS4G_OK;
}

}  // namespace
}  // namespace ds4g

extern "C" ds4g_status ds4g_moe_forward_noalloc(const ds4g_moe_desc *desc, const uint16_t *x,
                                                const float *logits, int32_t T, float *y,
                                                void *stream)
{
    Plan p;
    ds4g_status st = make_plan(desc, T, &p);
    if (st != DS4G_OK || T == 0) return st;
    if (!x || !logits || !y) return DS4G_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(logits, 4) || !aligned(y, 16)) return DS4G_ERR_LAYOUT;
    if (p.total > (size_t)DS4G_NOALLOC_SCRATCH_BYTES) return DS4G_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != DS4G_OK) return st;
    return forward_impl(desc, p, x, logits, y, static_cast<uint8_t *>(scratch),
                        static_cast<cudaStream_t>(stream), PhaseEvents{{}, false});
}

extern "C" ds4g_status ds4g_moe_noalloc_status(const ds4g_moe_desc *desc, int32_t T,
                                               int32_t *status_out, void *stream)
{
    using namespace ds4g;
    if (!status_out) return DS4G_ERR_INVALID;
    Plan p;
    ds4g_status st = make_plan(desc, T, &p);
    if (st != DS4G_OK) return st;
    if (p.total > DS4G_NOALLOC_SCRATCH_BYTES) return DS4G_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != DS4G_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(status_out, static_cast<uint8_t *>(scratch) + p.status,
                                    sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return from_cuda(e);
}
