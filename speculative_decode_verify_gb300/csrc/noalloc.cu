// verify_attn_full_noalloc: the full-attention verify call plus the combine, with the split partials in a
// fixed buffer that this library owns, for callers that cannot allocate device memory.
//
// Some callers of this library cannot allocate device memory at the time they call it: a decode loop
// embedded in another runtime that hands it only tensors and a stream (and no allocator), or a latency-
// critical loop that must not call cudaMalloc because cudaMalloc can synchronise the device.  They cannot
// provide the part_o / part_lse workspace that verify_attn_full needs, so this entry point keeps the
// partials in a file-scope device array instead.
#include <mutex>

#include "va_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kScratchFloats =
    (size_t)VA_NOALLOC_MAX_SPLITS * VA_MAX_ROWS * VA_Q_HEADS * (VA_HEAD_DIM + 1);   // part_o then part_lse

// Held in the memory of every GPU that loads this library's device code, until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device (nullptr: not yet)

// Device address of the scratch array on the current device.  The first call on a device looks it up
// with cudaGetSymbolAddress (with that device current); later calls reuse it.
cudaError_t scratch_on_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" VA_API va_status verify_attn_full_noalloc(const va_bf16* q, int n_rows, int n_live, const va_bf16* k_cache,
                                                     const va_bf16* v_cache, int capacity, const int32_t* pos,
                                                     float scale, int n_splits, const float* sink, va_bf16* out,
                                                     float* out_lse, int* splits_used, int32_t* dev_status,
                                                     va_stream stream) {
    if (!q || !k_cache || !v_cache || !pos || !out) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_ROWS || n_live < 0 || n_live > n_rows || capacity < 1) return VA_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return VA_INVALID_ARG;
    if (n_splits < 0) return VA_INVALID_ARG;
    // auto: the library's split choice, capped at what the fixed scratch holds (a GPU with more SMs than
    // VA_NOALLOC_MAX_SPLITS then runs fewer, longer splits instead of failing)
    if (n_splits == 0) n_splits = va_auto_splits(capacity, 0) < VA_NOALLOC_MAX_SPLITS ? va_auto_splits(capacity, 0)
                                                                                     : VA_NOALLOC_MAX_SPLITS;
    if (n_splits < 1 || n_splits > VA_NOALLOC_MAX_SPLITS) return VA_INVALID_ARG;   // beyond the fixed scratch

    float* scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return VA_CUDA_ERROR;
    // The partials are fully rewritten by every call: nothing in the scratch needs clearing.
    float* part_o = scratch;
    float* part_lse = scratch + (size_t)n_splits * n_rows * VA_Q_HEADS * VA_HEAD_DIM;

    va::AttnArgs a;
    a.q = q; a.k = k_cache; a.v = v_cache; a.pos = pos;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = capacity; a.window = 0;
    a.n_splits = n_splits;
    a.tree = nullptr; a.n_groups = 1;
    if (va::launch_attn(a, (cudaStream_t)stream) != cudaSuccess) return VA_CUDA_ERROR;
    if (va::launch_combine(part_o, part_lse, n_splits, sink, n_rows, n_live, out, out_lse, (cudaStream_t)stream) !=
        cudaSuccess)
        return VA_CUDA_ERROR;
    if (splits_used) *splits_used = n_splits;
    return VA_OK;
}
