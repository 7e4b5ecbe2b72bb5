// Ring / cache append of the verify rows' new K and V.
// IQuestRT report, "Read only the KV tiles needed by the current positions": verification writes
// its KV rows before reading them; position p lives in slot p mod ring_slots.
#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

// One warp per live row: lanes 0..15 copy K (16 B each), lanes 16..31 copy V.  The rows land as if written
// in row order: a row whose slot a later row also writes is skipped (rows <= 16, so lane l holds row l's
// position).
__global__ void __launch_bounds__(32) kv_append_kernel(const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       int slots, const int32_t* __restrict__ pos,
                                                       int32_t* dev_status) {
    const int r = blockIdx.x;
    const int lane = threadIdx.x;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // every global access comes after this
    constexpr int kChunks = kD * 2 / 16;   // 16 chunks of 16 B per row
    const int c = lane & (kChunks - 1);
    // the row and the positions are loaded together (one memory round trip)
    const int n = gridDim.x;
    const uint4 val = lane < kChunks ? __ldcg(k_new + (long long)r * kChunks + c) : __ldcg(v_new + (long long)r * kChunks + c);
    const int pl = lane < n ? __ldcg(pos + lane) : -1;
    const int p = __shfl_sync(0xffffffffu, pl, r);
    if (p < 0) {
        if (lane == 0 && dev_status) atomicOr(dev_status, VA_DEV_NEGATIVE_POS);
        return;
    }
    const long long slot = (long long)p % slots;
    if (__any_sync(0xffffffffu, lane > r && pl >= 0 && (long long)pl % slots == slot)) return;
    if (lane < kChunks)
        k_cache[slot * kChunks + c] = val;
    else
        v_cache[slot * kChunks + c] = val;
}

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, int n_live, uint16_t* k_cache,
                          uint16_t* v_cache, int slots, const int32_t* pos, int32_t* dev_status,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3(n_live), dim3(32), 0, stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kv_append_kernel, reinterpret_cast<const uint4*>(k_new),
                                             reinterpret_cast<const uint4*>(v_new), reinterpret_cast<uint4*>(k_cache),
                                             reinterpret_cast<uint4*>(v_cache), slots, pos, dev_status);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
