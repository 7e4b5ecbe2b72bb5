// C ABI entry points: argument checks, split-count policy and launches.
// Every entry point validates its host-side arguments, launches on the caller's stream and
// returns a va_status; nothing is allocated, freed or synchronized here.
#include <cmath>
#include <mutex>

#include "va_internal.cuh"

#ifndef VA_MIN_SPLIT_TILES
#define VA_MIN_SPLIT_TILES 2
#endif

namespace va {

int device_sm_count();   // also called by codec.cu

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];  // 0 = not queried yet
std::mutex g_mu;
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace va

namespace {

using va::device_sm_count;

va_status from_cuda(cudaError_t e) { return e == cudaSuccess ? VA_OK : VA_CUDA_ERROR; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

va_status check_attn_common(const va_bf16* q, int n_rows, int n_live, const va_bf16* k, const va_bf16* v,
                            int slots, const int32_t* pos, float scale, int n_splits, const float* part_o,
                            const float* part_lse) {
    if (!q || !k || !v || !pos || !part_o || !part_lse) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(part_o) || !aligned16(part_lse))
        return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_ROWS || n_live < 0 || n_live > n_rows) return VA_INVALID_ARG;
    if (slots < 1) return VA_INVALID_ARG;
    if (!std::isfinite(scale)) return VA_INVALID_ARG;
    if (n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    return VA_OK;
}

}  // namespace

namespace va {

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
    struct Entry { const void* kernel; int device; int bytes; };
    static Entry done[256];
    static int n_done = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].kernel == kernel && done[i].device == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && n_done < 256) done[n_done++] = Entry{kernel, dev, bytes};
    return e;
}

}  // namespace va

extern "C" {

va_status kv_ring_append(const va_bf16* k_new, const va_bf16* v_new, int n_live, va_bf16* k_cache,
                         va_bf16* v_cache, int slots, const int32_t* pos, int32_t* dev_status,
                         va_stream stream) {
    if (n_live < 0 || n_live > VA_MAX_TREE_NODES || slots < 1) return VA_INVALID_ARG;
    if (n_live == 0) return VA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !pos) return VA_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache)) return VA_INVALID_ARG;
    return from_cuda(va::launch_append(k_new, v_new, n_live, k_cache, v_cache, slots, pos, dev_status,
                                       (cudaStream_t)stream));
}

va_status verify_attn_full(const va_bf16* q, int n_rows, int n_live, const va_bf16* k_cache,
                           const va_bf16* v_cache, int capacity, const int32_t* pos, float scale,
                           int n_splits, float* part_o, float* part_lse, int* splits_used,
                           int32_t* dev_status, va_stream stream) {
    va_status st = check_attn_common(q, n_rows, n_live, k_cache, v_cache, capacity, pos, scale, n_splits,
                                     part_o, part_lse);
    if (st != VA_OK) return st;
    if (n_splits == 0) n_splits = va_auto_splits(capacity, 0);
    va::AttnArgs a;
    a.q = q; a.k = k_cache; a.v = v_cache; a.pos = pos;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = capacity; a.window = 0;
    a.n_splits = n_splits;
    a.tree = nullptr; a.n_groups = 1;
    st = from_cuda(va::launch_attn(a, (cudaStream_t)stream));
    if (st == VA_OK && splits_used) *splits_used = n_splits;
    return st;
}

va_status verify_attn_swa(const va_bf16* q, int n_rows, int n_live, const va_bf16* k_ring,
                          const va_bf16* v_ring, int ring_slots, int window, const int32_t* pos, float scale,
                          int n_splits, float* part_o, float* part_lse, int* splits_used, int32_t* dev_status,
                          va_stream stream) {
    va_status st = check_attn_common(q, n_rows, n_live, k_ring, v_ring, ring_slots, pos, scale, n_splits,
                                     part_o, part_lse);
    if (st != VA_OK) return st;
    if (window < 1) return VA_INVALID_ARG;
    if (ring_slots % VA_TILE != 0) return VA_UNSUPPORTED;
    if ((long long)ring_slots < (long long)window + (n_live > 0 ? n_live - 1 : 0)) return VA_RING_TOO_SMALL;
    if (n_splits == 0) n_splits = va_auto_splits(window + (n_live > 0 ? n_live - 1 : 0), window);
    va::AttnArgs a;
    a.q = q; a.k = k_ring; a.v = v_ring; a.pos = pos;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = ring_slots; a.window = window;
    a.n_splits = n_splits;
    a.tree = nullptr; a.n_groups = 1;
    st = from_cuda(va::launch_attn(a, (cudaStream_t)stream));
    if (st == VA_OK && splits_used) *splits_used = n_splits;
    return st;
}

va_status verify_attn_tree(const va_bf16* q, int n_rows, int n_nodes, const va_bf16* k_cache,
                           const va_bf16* v_cache, int slots, int window, const int32_t* tree, float scale,
                           int n_splits, float* part_o, float* part_lse, int* splits_used, int32_t* dev_status,
                           va_stream stream) {
    if (!q || !k_cache || !v_cache || !tree || !part_o || !part_lse) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(part_o) || !aligned16(part_lse))
        return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_TREE_NODES || n_nodes < 0 || n_nodes > n_rows || slots < 1) return VA_INVALID_ARG;
    if (!std::isfinite(scale) || window < 0 || n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    const int groups = (n_rows + VA_MAX_ROWS - 1) / VA_MAX_ROWS;
    if (window > 0) {
        if (window < n_nodes) return VA_UNSUPPORTED;   // every ancestor must lie inside every window
        if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
        if ((long long)slots < (long long)window + (n_nodes > 0 ? n_nodes - 1 : 0)) return VA_RING_TOO_SMALL;
    }
    if (n_splits == 0) {
        // the node groups share the SMs: at most one CTA per SM over all groups
        const int sms = device_sm_count();
        const int extent = window > 0 ? window + (n_nodes > 0 ? n_nodes - 1 : 0) : slots;
        n_splits = va_auto_splits_for(extent, window, (sms > 0 ? sms : 148) / groups);
    }
    va::AttnArgs a;
    a.q = q; a.k = k_cache; a.v = v_cache; a.pos = nullptr; a.tree = tree;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_nodes; a.slots = slots; a.window = window;
    a.n_splits = n_splits; a.n_groups = groups;
    va_status st = from_cuda(va::launch_attn(a, (cudaStream_t)stream));
    if (st == VA_OK && splits_used) *splits_used = n_splits;
    return st;
}

va_status attn_split_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                             int n_rows, int n_live, va_bf16* out, float* out_lse, va_stream stream) {
    if (!out || n_rows < 1 || n_rows > VA_MAX_TREE_NODES || n_live < 0 || n_live > n_rows) return VA_INVALID_ARG;
    if (n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    if (n_splits > 0 && (!part_o || !part_lse)) return VA_INVALID_ARG;
    if (!aligned16(out) || (n_splits > 0 && (!aligned16(part_o) || !aligned16(part_lse)))) return VA_INVALID_ARG;
    return from_cuda(va::launch_combine(part_o, part_lse, n_splits, sink, n_rows, n_live, out, out_lse,
                                        (cudaStream_t)stream));
}

va_status verify_attn_step(const va_bf16* q, const va_bf16* k_new, const va_bf16* v_new, int n_rows, int n_live,
                           va_bf16* k_cache, va_bf16* v_cache, int slots, int window, const int32_t* pos,
                           const float* sink, float scale, int n_splits, float* workspace, va_bf16* out,
                           float* out_lse, int* splits_used, int32_t* dev_status, va_stream stream) {
    if (!out || !aligned16(out)) return VA_INVALID_ARG;
    if (n_live > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return VA_INVALID_ARG;
    if (window < 0 || n_splits < 0 || n_splits > VA_MAX_SPLITS || !workspace) return VA_INVALID_ARG;
    if (n_splits == 0)
        n_splits = window > 0 ? va_auto_splits(window + (n_live > 0 ? n_live - 1 : 0), window)
                              : va_auto_splits(slots, 0);
    float* part_o = workspace;
    float* part_lse = workspace + (size_t)n_splits * VA_MAX_ROWS * VA_Q_HEADS * VA_HEAD_DIM;
    va_status st = check_attn_common(q, n_rows, n_live, k_cache, v_cache, slots, pos, scale, n_splits, part_o,
                                     part_lse);
    if (st != VA_OK) return st;
    if (window > 0) {
        if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
        if ((long long)slots < (long long)window + (n_live > 0 ? n_live - 1 : 0)) return VA_RING_TOO_SMALL;
    }
    va::AttnArgs a;
    a.q = q; a.k = k_cache; a.v = v_cache; a.pos = pos;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = slots; a.window = window;
    a.n_splits = n_splits;
    a.tree = nullptr; a.n_groups = 1;
    if (n_live > 0) {
        a.k_new = k_new;
        a.v_new = v_new;
    }
    st = from_cuda(va::launch_attn(a, (cudaStream_t)stream));
    if (st != VA_OK) return st;
    st = from_cuda(va::launch_combine(part_o, part_lse, n_splits, sink, n_rows, n_live, out, out_lse,
                                      (cudaStream_t)stream));
    if (st == VA_OK && splits_used) *splits_used = n_splits;
    return st;
}

size_t va_workspace_bytes(int n_splits) {
    if (n_splits < 1 || n_splits > VA_MAX_SPLITS) return 0;
    return sizeof(float) * (size_t)n_splits * VA_MAX_ROWS * VA_Q_HEADS * (VA_HEAD_DIM + 1);
}

int va_auto_splits_for(int extent_hint, int window, int sm_count) {
    // One split per SM at most (the split kernel holds a whole SM's shared memory); at least
    // VA_MIN_SPLIT_TILES 64-position tiles per split so that each split amortises its partial write.
    if (sm_count < 1) sm_count = 148;
    long long extent = extent_hint > 0 ? extent_hint : 1;
    if (window > 0 && extent > (long long)window + VA_MAX_ROWS - 1) extent = (long long)window + VA_MAX_ROWS - 1;
    const long long tiles = (extent + VA_TILE - 1) / VA_TILE + (window > 0 ? 1 : 0);
    long long s = (tiles + VA_MIN_SPLIT_TILES - 1) / VA_MIN_SPLIT_TILES;
    if (s > sm_count) s = sm_count;
    if (s < 1) s = 1;
    return (int)s;
}

int va_auto_splits(int extent_hint, int window) {
    return va_auto_splits_for(extent_hint, window, device_sm_count());
}

const char* va_status_string(va_status status) {
    switch (status) {
        case VA_OK: return "VA_OK";
        case VA_INVALID_ARG: return "VA_INVALID_ARG";
        case VA_UNSUPPORTED: return "VA_UNSUPPORTED";
        case VA_RING_TOO_SMALL: return "VA_RING_TOO_SMALL";
        case VA_CUDA_ERROR: return "VA_CUDA_ERROR";
        default: return "VA_UNKNOWN_STATUS";
    }
}

}  // extern "C"
