// cache.cu -- the expert cache: routed experts whose weights live in host
// memory, kept in a fixed number of device slots and uploaded on misses
// (the in-memory expert cache with configurable budgets of the pages:
// opensourcealternatives.to, FAQ; DwarfStar 4 on aiany.app, "What Sets It
// Apart").  Host code only: the layer itself runs on the ordinary kernels,
// which read expert e's weights from slot expert_slot[e].
//
// One call: route on the device, read the per-expert counts back (the only
// host synchronization), give every routed expert a slot (hits keep theirs;
// misses take a free slot or the least recently used slot of an expert this
// call does not route to), upload the misses' three matrices with
// cudaMemcpyAsync, upload the map, run the layer.
#include <cstring>
#include <vector>

#include "ds4g_common.cuh"

struct ds4g_expert_cache {
    ds4g_moe_desc host;              // the caller's layer, weights in host memory
    ds4g_moe_desc dev;               // the same layer on the device slots
    int32_t n_slots = 0;
    uint8_t *d_gate = nullptr, *d_up = nullptr, *d_down = nullptr;
    int32_t *d_map = nullptr;        // [E] slot of each expert (-1: none)
    int32_t *h_map = nullptr;        // [E] page-locked staging copy of the map
    int32_t *h_counts = nullptr;     // [E] page-locked routing counts of the call
    std::vector<int32_t> slot_of;    // [E] host copy of the map
    std::vector<int32_t> owner;      // [n_slots] expert in each slot (-1: free)
    std::vector<uint64_t> stamp;     // [n_slots] last call that used the slot
    uint64_t calls = 0;
    int64_t hits = 0, misses = 0, bytes = 0;
};

namespace {

void release(ds4g_expert_cache *c)
{
    cudaFree(c->d_gate);
    cudaFree(c->d_up);
    cudaFree(c->d_down);
    cudaFree(c->d_map);
    cudaFreeHost(c->h_map);
    cudaFreeHost(c->h_counts);
    delete c;
}

}  // namespace

ds4g_status ds4g_expert_cache_create(const ds4g_moe_desc *host_desc, int32_t n_slots,
                                     ds4g_expert_cache **out)
{
    using namespace ds4g;
    if (!host_desc || !out) return DS4G_ERR_INVALID;
    *out = nullptr;
    if (host_desc->n_slots != 0 || host_desc->expert_slot) return DS4G_ERR_INVALID;
    Plan p;
    ds4g_status st = make_plan(host_desc, 1, &p);
    if (st != DS4G_OK) return st;
    if (n_slots < host_desc->top_k || n_slots > host_desc->n_experts) return DS4G_ERR_INVALID;
    auto *c = new ds4g_expert_cache();
    c->host = *host_desc;
    c->n_slots = n_slots;
    const int E = host_desc->n_experts;
    const size_t gu = (size_t)host_desc->gate_up_expert_stride * n_slots;
    const size_t dn = (size_t)host_desc->down_expert_stride * n_slots;
    cudaError_t e;
    if ((e = cudaMalloc(&c->d_gate, gu)) != cudaSuccess || (e = cudaMalloc(&c->d_up, gu)) != cudaSuccess ||
        (e = cudaMalloc(&c->d_down, dn)) != cudaSuccess ||
        (e = cudaMalloc(&c->d_map, sizeof(int32_t) * E)) != cudaSuccess ||
        (e = cudaHostAlloc(&c->h_map, sizeof(int32_t) * E, cudaHostAllocDefault)) != cudaSuccess ||
        (e = cudaHostAlloc(&c->h_counts, sizeof(int32_t) * E, cudaHostAllocDefault)) != cudaSuccess ||
        (e = cudaMemset(c->d_map, 0xFF, sizeof(int32_t) * E)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        release(c);
        return status_from_cuda(e);
    }
    c->slot_of.assign(E, -1);
    c->owner.assign(n_slots, -1);
    c->stamp.assign(n_slots, 0);
    std::memset(c->h_map, 0xFF, sizeof(int32_t) * E);
    c->dev = *host_desc;
    c->dev.w_gate = c->d_gate;
    c->dev.w_up = c->d_up;
    c->dev.w_down = c->d_down;
    c->dev.n_slots = n_slots;
    c->dev.expert_slot = c->d_map;
    *out = c;
    return DS4G_OK;
}

size_t ds4g_expert_cache_workspace_bytes(const ds4g_expert_cache *c, int32_t T)
{
    return c ? ds4g_moe_workspace_bytes(&c->dev, T) : 0;
}

ds4g_status ds4g_expert_cache_forward(ds4g_expert_cache *c, const uint16_t *x, const float *logits,
                                      int32_t T, float *y, void *workspace, size_t ws_bytes,
                                      void *stream)
{
    using namespace ds4g;
    if (!c) return DS4G_ERR_INVALID;
    Plan p;
    ds4g_status st = make_plan(&c->dev, T, &p);
    if (st != DS4G_OK) return st;
    if (T == 0) return DS4G_OK;
    if (!x || !logits || !y || !workspace) return DS4G_ERR_INVALID;
    if (ws_bytes < p.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return DS4G_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int E = p.E;
    // which experts this call routes to (the layer routes again, identically)
    int32_t *counts = reinterpret_cast<int32_t *>(ws + p.counts);
    st = ds4g_route_topk(logits, T, E, p.k, c->host.score, reinterpret_cast<int32_t *>(ws + p.ids),
                         reinterpret_cast<float *>(ws + p.wts), counts,
                         reinterpret_cast<int32_t *>(ws + p.offsets),
                         reinterpret_cast<int32_t *>(ws + p.perm), stream);
    if (st != DS4G_OK) return st;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(c->h_counts, counts, sizeof(int32_t) * E, cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return status_from_cuda(e);
    // hits first: every slot this call uses is stamped with the call, so the
    // victims of the misses are never among them
    const uint64_t now = ++c->calls;
    int n_routed = 0;
    for (int ex = 0; ex < E; ++ex) {
        if (c->h_counts[ex] <= 0) continue;
        ++n_routed;
        if (c->slot_of[ex] >= 0) c->stamp[c->slot_of[ex]] = now;
    }
    if (n_routed > c->n_slots) return DS4G_ERR_UNSUPPORTED;
    const size_t gus = (size_t)c->host.gate_up_expert_stride, dns = (size_t)c->host.down_expert_stride;
    const uint8_t *hg = static_cast<const uint8_t *>(c->host.w_gate);
    const uint8_t *hu = static_cast<const uint8_t *>(c->host.w_up);
    const uint8_t *hd = static_cast<const uint8_t *>(c->host.w_down);
    bool changed = false;
    for (int ex = 0; ex < E; ++ex) {
        if (c->h_counts[ex] <= 0) continue;
        if (c->slot_of[ex] >= 0) {
            ++c->hits;
            continue;
        }
        // a free slot, else the least recently used one not used by this call
        int v = -1;
        for (int sl = 0; sl < c->n_slots; ++sl) {
            if (c->stamp[sl] == now) continue;           // used by this call
            if (c->owner[sl] < 0) {                      // free
                v = sl;
                break;
            }
            if (v < 0 || c->stamp[sl] < c->stamp[v]) v = sl;
        }
        if (v < 0) return DS4G_ERR_UNSUPPORTED;          // unreachable: n_routed <= n_slots
        if (c->owner[v] >= 0) {
            c->slot_of[c->owner[v]] = -1;
            c->h_map[c->owner[v]] = -1;
        }
        c->owner[v] = ex;
        c->slot_of[ex] = v;
        c->h_map[ex] = v;
        c->stamp[v] = now;
        if ((e = cudaMemcpyAsync(c->d_gate + v * gus, hg + ex * gus, gus, cudaMemcpyHostToDevice, s)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(c->d_up + v * gus, hu + ex * gus, gus, cudaMemcpyHostToDevice, s)) !=
                cudaSuccess ||
            (e = cudaMemcpyAsync(c->d_down + v * dns, hd + ex * dns, dns, cudaMemcpyHostToDevice, s)) !=
                cudaSuccess)
            return status_from_cuda(e);
        ++c->misses;
        c->bytes += (int64_t)(2 * gus + dns);
        changed = true;
    }
    if (changed && (e = cudaMemcpyAsync(c->d_map, c->h_map, sizeof(int32_t) * E,
                                        cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return status_from_cuda(e);
    return ds4g_moe_forward(&c->dev, x, logits, T, y, workspace, ws_bytes, stream);
}

ds4g_status ds4g_expert_cache_stats(const ds4g_expert_cache *c, int64_t *hits, int64_t *misses,
                                    int64_t *bytes_uploaded)
{
    if (!c) return DS4G_ERR_INVALID;
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (bytes_uploaded) *bytes_uploaded = c->bytes;
    return DS4G_OK;
}

void ds4g_expert_cache_destroy(ds4g_expert_cache *c)
{
    if (!c) return;
    cudaDeviceSynchronize();
    release(c);
}
