// The quantised K/V cache ("Qwen3.8-27B on one RTX 4090", section "A cheaper cache and state"): the
// encoding append (keys rotated by the +-1 Hadamard butterfly and coded E4M3, values coded INT8, one
// scale per row) and the C ABI of the cache's append and verify attention.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "codec_dev.cuh"
#include "kv_codec.h"
#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

cudaError_t launch_attn_q8(const AttnArgs& a, const float* k_scale, const float* v_scale, cudaStream_t stream);
int device_sm_count();   // abi.cu: multiprocessors of the current device (0 if the query fails)

namespace codec {

// One CTA per live row: warp 0 codes its key, warp 1 its value.  Lane l holds elements 4 l .. 4 l + 3.
__global__ void __launch_bounds__(64) append_q8_kernel(const uint2* __restrict__ k_new, const uint2* __restrict__ v_new,
                                                       uint8_t* __restrict__ k_codes, int8_t* __restrict__ v_codes,
                                                       float* __restrict__ k_scale, float* __restrict__ v_scale, int slots,
                                                       const int32_t* __restrict__ pos, int32_t* dev_status) {
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const uint2 raw = __ldcg((warp == 0 ? k_new : v_new) + (size_t)r * 32 + lane);
    const int p = __ldcg(pos + r);
    if (p < 0) {
        if (threadIdx.x == 0 && dev_status) atomicOr(dev_status, VA_DEV_NEGATIVE_POS);
        return;
    }
    const size_t slot = (size_t)(p % slots);
    // rows land as if written in row order where the next row writes the same slot (verify rows share
    // a slot only when they share a position, and then they are adjacent): the earlier row is skipped
    if (r + 1 < (int)gridDim.x) {
        const int pn = __ldcg(pos + r + 1);
        if (pn >= 0 && (size_t)(pn % slots) == slot) return;
    }
    if (warp == 0) code_key_row(raw, lane, k_codes + slot * kD, k_scale + slot);
    else code_value_row(raw, lane, v_codes + slot * kD, v_scale + slot);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace codec
}  // namespace va

extern "C" {

va_status kv_ring_append_q8(const va_bf16* k_new, const va_bf16* v_new, int n_live, uint8_t* k_codes, int8_t* v_codes,
                            float* k_scale, float* v_scale, int slots, const int32_t* pos, int32_t* dev_status,
                            va_stream stream) {
    using va::codec::aligned16;
    if (n_live < 0 || n_live > VA_Q8_MAX_APPEND || slots < 1) return VA_INVALID_ARG;
    if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
    if (n_live == 0) return VA_OK;
    if (!k_new || !v_new || !k_codes || !v_codes || !k_scale || !v_scale || !pos) return VA_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) ||
        !aligned16(v_scale))
        return VA_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    va::pdl_config(&cfg, attr, dim3(n_live), dim3(64), 0, (cudaStream_t)stream);
    cudaError_t e = cudaLaunchKernelEx(&cfg, va::codec::append_q8_kernel, reinterpret_cast<const uint2*>(k_new),
                                       reinterpret_cast<const uint2*>(v_new), k_codes, v_codes, k_scale, v_scale, slots,
                                       pos, dev_status);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? VA_OK : VA_CUDA_ERROR;
}

va_status verify_attn_q8(const va_bf16* q, int n_rows, int n_live, const uint8_t* k_codes, const int8_t* v_codes,
                         const float* k_scale, const float* v_scale, int slots, int window, const int32_t* pos,
                         float scale, int n_splits, float* part_o, float* part_lse, int* splits_used,
                         int32_t* dev_status, va_stream stream) {
    using va::codec::aligned16;
    if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !pos || !part_o || !part_lse) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale) ||
        !aligned16(part_o) || !aligned16(part_lse))
        return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_ROWS || n_live < 0 || n_live > n_rows || slots < 1) return VA_INVALID_ARG;
    if (!std::isfinite(scale) || window < 0 || n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
    if (window > 0 && (long long)slots < (long long)window + (n_live > 0 ? n_live - 1 : 0)) return VA_RING_TOO_SMALL;
    if (n_splits == 0) n_splits = va_auto_splits(window > 0 ? window + (n_live > 0 ? n_live - 1 : 0) : slots, window);
    va::AttnArgs a;
    a.q = q; a.k = reinterpret_cast<const uint16_t*>(k_codes); a.v = reinterpret_cast<const uint16_t*>(v_codes);
    a.pos = pos; a.tree = nullptr;   // the byte codes travel in the bf16 pointers of AttnArgs
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = slots; a.window = window;
    a.n_splits = n_splits; a.n_groups = 1;
    const cudaError_t e = va::launch_attn_q8(a, k_scale, v_scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return VA_CUDA_ERROR;
    if (splits_used) *splits_used = n_splits;
    return VA_OK;
}

va_status verify_attn_q8_step(const va_bf16* q, const va_bf16* k_new, const va_bf16* v_new, int n_rows, int n_live,
                              uint8_t* k_codes, int8_t* v_codes, float* k_scale, float* v_scale, int slots, int window,
                              const int32_t* pos, const float* sink, float scale, int n_splits, float* workspace,
                              va_bf16* out, float* out_lse, int* splits_used, int32_t* dev_status, va_stream stream) {
    using va::codec::aligned16;
    if (!out || !aligned16(out) || !workspace || !aligned16(workspace)) return VA_INVALID_ARG;
    if (n_live > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))) return VA_INVALID_ARG;
    if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !pos) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale))
        return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_ROWS || n_live < 0 || n_live > n_rows || slots < 1) return VA_INVALID_ARG;
    if (!std::isfinite(scale) || window < 0 || n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
    if (window > 0 && (long long)slots < (long long)window + (n_live > 0 ? n_live - 1 : 0)) return VA_RING_TOO_SMALL;
    if (n_splits == 0) n_splits = va_auto_splits(window > 0 ? window + (n_live > 0 ? n_live - 1 : 0) : slots, window);
    float* part_o = workspace;
    float* part_lse = workspace + (size_t)n_splits * VA_MAX_ROWS * VA_Q_HEADS * VA_HEAD_DIM;
    if (!VA_Q8_FUSED_APPEND) {
        const va_status st = kv_ring_append_q8(k_new, v_new, n_live, k_codes, v_codes, k_scale, v_scale, slots, pos,
                                               dev_status, stream);
        if (st != VA_OK) return st;
    }
    va::AttnArgs a;
    a.q = q; a.k = reinterpret_cast<const uint16_t*>(k_codes); a.v = reinterpret_cast<const uint16_t*>(v_codes);
    a.pos = pos; a.tree = nullptr;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_live; a.slots = slots; a.window = window;
    a.n_splits = n_splits; a.n_groups = 1;
    if (VA_Q8_FUSED_APPEND && n_live > 0) {   // the live rows are coded by the attention launch itself
        a.k_new = reinterpret_cast<const uint16_t*>(k_new);
        a.v_new = reinterpret_cast<const uint16_t*>(v_new);
    }
    cudaError_t e = va::launch_attn_q8(a, k_scale, v_scale, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = va::launch_combine(part_o, part_lse, n_splits, sink, n_rows, n_live, out, out_lse, (cudaStream_t)stream);
    if (e != cudaSuccess) return VA_CUDA_ERROR;
    if (splits_used) *splits_used = n_splits;
    return VA_OK;
}

va_status verify_attn_q8_tree(const va_bf16* q, int n_rows, int n_nodes, const uint8_t* k_codes, const int8_t* v_codes,
                              const float* k_scale, const float* v_scale, int slots, int window, const int32_t* tree,
                              float scale, int n_splits, float* part_o, float* part_lse, int* splits_used,
                              int32_t* dev_status, va_stream stream) {
    using va::codec::aligned16;
    if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !tree || !part_o || !part_lse) return VA_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale) ||
        !aligned16(part_o) || !aligned16(part_lse))
        return VA_INVALID_ARG;
    if (n_rows < 1 || n_rows > VA_MAX_TREE_NODES || n_nodes < 0 || n_nodes > n_rows || slots < 1) return VA_INVALID_ARG;
    if (!std::isfinite(scale) || window < 0 || n_splits < 0 || n_splits > VA_MAX_SPLITS) return VA_INVALID_ARG;
    if (slots % VA_TILE != 0) return VA_UNSUPPORTED;
    if (window > 0) {
        if (window < n_nodes) return VA_UNSUPPORTED;   // every ancestor must lie inside every window
        if ((long long)slots < (long long)window + (n_nodes > 0 ? n_nodes - 1 : 0)) return VA_RING_TOO_SMALL;
    }
    const int groups = (n_rows + VA_MAX_ROWS - 1) / VA_MAX_ROWS;
    if (n_splits == 0) {
        // the node groups share the SMs: at most one CTA per SM over all groups
        const int sms = va::device_sm_count();
        const int extent = window > 0 ? window + (n_nodes > 0 ? n_nodes - 1 : 0) : slots;
        n_splits = va_auto_splits_for(extent, window, (sms > 0 ? sms : 148) / groups);
    }
    va::AttnArgs a;
    a.q = q; a.k = reinterpret_cast<const uint16_t*>(k_codes); a.v = reinterpret_cast<const uint16_t*>(v_codes);
    a.pos = nullptr; a.tree = tree;
    a.part_o = part_o; a.part_lse = part_lse; a.dev_status = dev_status;
    a.scale = scale; a.n_rows = n_rows; a.n_live = n_nodes; a.slots = slots; a.window = window;
    a.n_splits = n_splits; a.n_groups = groups;
    const cudaError_t e = va::launch_attn_q8(a, k_scale, v_scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return VA_CUDA_ERROR;
    if (splits_used) *splits_used = n_splits;
    return VA_OK;
}

}  // extern "C"
