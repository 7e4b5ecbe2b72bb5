// Log-sum-exp merge of the split partials with the learned sink folded in.
// IQuestRT report, "Read only the KV tiles needed by the current positions": a separate combine
// kernel issues the partial loads together and uses four independent FP32 accumulation chains;
// "Expose more parallelism in attention": the combine applies the sink correction and keeps the
// BF16 rounding boundary (the output is rounded to bf16 once, here).
#include <cuda_bf16.h>

#include "va_internal.cuh"

namespace va {

constexpr int kCombineThreads = kD;   // one thread per output column d

// One CTA per matrix row m = r * 6 + h.  Shared memory holds the split weights exp(lse_s - L).
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  int n_splits, const float* __restrict__ sink,
                                                                  int n_rows, int n_live,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ out_lse) {
    extern __shared__ float w[];          // [n_splits]
    __shared__ float red[kCombineThreads / 32];
    __shared__ float s_L;
    const int m = blockIdx.x;
    const int r = m / kH, h = m - r * kH;
    const int d = threadIdx.x;
    const int M = n_rows * kH;
    if (r >= n_live) {
        out[(long long)m * kD + d] = __float2bfloat16_rn(0.0f);
        if (out_lse && d == 0) out_lse[m] = -INFINITY;
        return;
    }
    const float sk = sink ? __ldg(sink + h) : -INFINITY;

    // L = logsumexp({lse_s} U {sink})
    float mx = sk;
    for (int s = d; s < n_splits; s += kCombineThreads) {
        const float l = __ldg(part_lse + (long long)s * M + m);
        w[s] = l;
        mx = fmaxf(mx, l);
    }
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((d & 31) == 0) red[d >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int i = 1; i < kCombineThreads / 32; ++i) mx = fmaxf(mx, red[i]);
    __syncthreads();
    if (mx == -INFINITY) {  // nothing visible and no sink
        out[(long long)m * kD + d] = __float2bfloat16_rn(0.0f);
        if (out_lse && d == 0) out_lse[m] = -INFINITY;
        return;
    }
    float z = (d == 0) ? expf(sk - mx) : 0.0f;
    for (int s = d; s < n_splits; s += kCombineThreads) z += expf(w[s] - mx);
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if ((d & 31) == 0) red[d >> 5] = z;
    __syncthreads();
    if (d == 0) {
        float zt = 0.0f;
        for (int i = 0; i < kCombineThreads / 32; ++i) zt += red[i];
        s_L = mx + logf(zt);
    }
    __syncthreads();
    const float L = s_L;
    for (int s = d; s < n_splits; s += kCombineThreads) w[s] = expf(w[s] - L);
    __syncthreads();

    // out[d] = sum_s w_s * o_s[d]: four independent chains, loads issued together
    const float* po = part_o + (long long)m * kD + d;
    const long long stride = (long long)M * kD;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 4 <= n_splits; s += 4) {
        const float o0 = __ldg(po + (s + 0) * stride);
        const float o1 = __ldg(po + (s + 1) * stride);
        const float o2 = __ldg(po + (s + 2) * stride);
        const float o3 = __ldg(po + (s + 3) * stride);
        acc0 = fmaf(w[s + 0], o0, acc0);
        acc1 = fmaf(w[s + 1], o1, acc1);
        acc2 = fmaf(w[s + 2], o2, acc2);
        acc3 = fmaf(w[s + 3], o3, acc3);
    }
    if (s + 0 < n_splits) acc0 = fmaf(w[s + 0], __ldg(po + (s + 0) * stride), acc0);
    if (s + 1 < n_splits) acc1 = fmaf(w[s + 1], __ldg(po + (s + 1) * stride), acc1);
    if (s + 2 < n_splits) acc2 = fmaf(w[s + 2], __ldg(po + (s + 2) * stride), acc2);
    out[(long long)m * kD + d] = __float2bfloat16_rn((acc0 + acc1) + (acc2 + acc3));
    if (out_lse && d == 0) out_lse[m] = L;
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                           int n_rows, int n_live, uint16_t* out, float* out_lse, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)(n_splits > 0 ? n_splits : 1);
    combine_kernel<<<n_rows * kH, kCombineThreads, smem, stream>>>(
        part_o, part_lse, n_splits, sink, n_rows, n_live, reinterpret_cast<__nv_bfloat16*>(out), out_lse);
    return cudaGetLastError();
}

}  // namespace va
