// Log-sum-exp merge of the split partials with the learned sink folded in.
// IQuestRT report, "Read only the KV tiles needed by the current positions": a separate combine
// kernel issues the partial loads together and uses four independent FP32 accumulation chains;
// "Expose more parallelism in attention": the combine applies the sink correction and keeps the
// BF16 rounding boundary (the output is rounded to bf16 once, here).
#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = 32 * kCombineWarps;

// One CTA per matrix row m = r * 6 + h.  Warp w accumulates the splits s = w, w + 8, ...: each lane owns
// four output columns and keeps four independent accumulators (one per unrolled split), with the four
// splits' loads issued before any of them is used.  The eight warp totals are then added in a fixed
// order.  Shared memory holds the split weights exp(lse_s - L).
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  int n_splits, const float* __restrict__ sink,
                                                                  int n_rows, int n_live,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ out_lse) {
    extern __shared__ float w[];          // [n_splits]
    __shared__ float red[kCombineWarps];
    __shared__ float4 part[kCombineWarps][kD / 4];
    __shared__ float s_mx, s_L;
    const int m = blockIdx.x;
    const int r = m / kH, h = m - r * kH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = n_rows * kH;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // every global access comes after this
    if (r >= n_live) {
        if (tid < kD) out[(long long)m * kD + tid] = __float2bfloat16_rn(0.0f);
        if (out_lse && tid == 0) out_lse[m] = -INFINITY;
        return;
    }
    const float sk = sink ? __ldcg(sink + h) : -INFINITY;

    // L = logsumexp({lse_s} U {sink})
    float mx = sk;
    for (int s = tid; s < n_splits; s += kCombineThreads) {
        const float l = __ldcg(part_lse + (long long)s * M + m);
        w[s] = l;
        mx = fmaxf(mx, l);
    }
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) {
        float t = red[0];
        for (int i = 1; i < kCombineWarps; ++i) t = fmaxf(t, red[i]);
        s_mx = t;
    }
    __syncthreads();
    mx = s_mx;
    if (mx == -INFINITY) {  // nothing visible and no sink
        if (tid < kD) out[(long long)m * kD + tid] = __float2bfloat16_rn(0.0f);
        if (out_lse && tid == 0) out_lse[m] = -INFINITY;
        return;
    }
    float z = (tid == 0) ? expf(sk - mx) : 0.0f;
    for (int s = tid; s < n_splits; s += kCombineThreads) z += expf(w[s] - mx);
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane == 0) red[warp] = z;
    __syncthreads();
    if (tid == 0) {
        float zt = 0.0f;
        for (int i = 0; i < kCombineWarps; ++i) zt += red[i];
        s_L = mx + logf(zt);
    }
    __syncthreads();
    const float L = s_L;
    for (int s = tid; s < n_splits; s += kCombineThreads) w[s] = expf(w[s] - L);
    __syncthreads();

    // out[d] = sum_s w_s o_s[d]
    const float4* po = reinterpret_cast<const float4*>(part_o + (long long)m * kD) + lane;
    const long long stride4 = (long long)M * kD / 4;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
    int s = warp;
    for (; s + 3 * kCombineWarps < n_splits; s += 4 * kCombineWarps) {
        const float4 o0 = __ldcg(po + (long long)(s + 0 * kCombineWarps) * stride4);
        const float4 o1 = __ldcg(po + (long long)(s + 1 * kCombineWarps) * stride4);
        const float4 o2 = __ldcg(po + (long long)(s + 2 * kCombineWarps) * stride4);
        const float4 o3 = __ldcg(po + (long long)(s + 3 * kCombineWarps) * stride4);
        const float w0 = w[s], w1 = w[s + kCombineWarps], w2 = w[s + 2 * kCombineWarps], w3 = w[s + 3 * kCombineWarps];
        a0.x = fmaf(w0, o0.x, a0.x); a0.y = fmaf(w0, o0.y, a0.y); a0.z = fmaf(w0, o0.z, a0.z); a0.w = fmaf(w0, o0.w, a0.w);
        a1.x = fmaf(w1, o1.x, a1.x); a1.y = fmaf(w1, o1.y, a1.y); a1.z = fmaf(w1, o1.z, a1.z); a1.w = fmaf(w1, o1.w, a1.w);
        a2.x = fmaf(w2, o2.x, a2.x); a2.y = fmaf(w2, o2.y, a2.y); a2.z = fmaf(w2, o2.z, a2.z); a2.w = fmaf(w2, o2.w, a2.w);
        a3.x = fmaf(w3, o3.x, a3.x); a3.y = fmaf(w3, o3.y, a3.y); a3.z = fmaf(w3, o3.z, a3.z); a3.w = fmaf(w3, o3.w, a3.w);
    }
    for (; s < n_splits; s += kCombineWarps) {
        const float4 o0 = __ldcg(po + (long long)s * stride4);
        const float w0 = w[s];
        a0.x = fmaf(w0, o0.x, a0.x); a0.y = fmaf(w0, o0.y, a0.y); a0.z = fmaf(w0, o0.z, a0.z); a0.w = fmaf(w0, o0.w, a0.w);
    }
    part[warp][lane] = make_float4((a0.x + a1.x) + (a2.x + a3.x), (a0.y + a1.y) + (a2.y + a3.y),
                                   (a0.z + a1.z) + (a2.z + a3.z), (a0.w + a1.w) + (a2.w + a3.w));
    __syncthreads();
    if (tid < kD) {
        const float* pf = reinterpret_cast<const float*>(part);
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < kCombineWarps; ++i) acc += pf[i * kD + tid];
        out[(long long)m * kD + tid] = __float2bfloat16_rn(acc);
        if (out_lse && tid == 0) out_lse[m] = L;
    }
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                           int n_rows, int n_live, uint16_t* out, float* out_lse, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)(n_splits > 0 ? n_splits : 1);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3(n_rows * kH), dim3(kCombineThreads), smem, stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, part_o, part_lse, n_splits, sink, n_rows, n_live,
                                             reinterpret_cast<__nv_bfloat16*>(out), out_lse);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
