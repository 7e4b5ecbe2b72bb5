// Log-sum-exp merge of the split partials with the learned sink folded in.
// IQuestRT report, "Read only the KV tiles needed by the current positions": a separate combine
// kernel issues the partial loads together and uses independent FP32 accumulation chains;
// "Expose more parallelism in attention": the combine applies the sink correction and keeps the
// BF16 rounding boundary (the output is rounded to bf16 once, here).
#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

constexpr int kCombineThreads = 256;
constexpr int kQuarters = 4;                       // column quarters of a matrix row: 32 columns each
constexpr int kChunks = kD / kQuarters / 4;        // float4 chunks per quarter: 8
constexpr int kGroups = kCombineThreads / kChunks; // split groups: 32
constexpr int kBatch = 8;                          // splits per thread loaded together

// One CTA per (matrix row m = 6 r + h, column quarter).  Thread t owns float4 chunk t % 8 of the quarter
// and the splits s = t / 8 + 32 i: it issues all of its partial and LSE loads before using any of them
// (the partials do not depend on the maximum, so normalisation waits until the end:
// out = sum_s e^(lse_s - M) o_s / (sum_s e^(lse_s - M) + e^(sink - M)), M the maximum over {lse_s} U {sink}).
// Every thread keeps its own FP32 chains; the 32 per-chunk totals are added in a fixed order.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  int n_splits, const float* __restrict__ sink,
                                                                  int n_rows, int n_live,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ out_lse) {
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 part[kGroups][kChunks];
    __shared__ float zpart[kGroups];
    __shared__ float s_mx;
    const int m = blockIdx.x, quarter = blockIdx.y;
    const int r = m / kH, h = m - r * kH;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = tid % kChunks, group = tid / kChunks;
    const int M = n_rows * kH;
    const int col0 = quarter * (kD / kQuarters) + 4 * chunk;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // every global access comes after this
    if (r >= n_live) {
        if (tid < kD / kQuarters) out[(long long)m * kD + quarter * (kD / kQuarters) + tid] = __float2bfloat16_rn(0.0f);
        if (out_lse && quarter == 0 && tid == 0) out_lse[m] = -INFINITY;
        return;
    }
    const float sk = sink ? __ldcg(sink + h) : -INFINITY;

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float z = 0.0f, mx = sk;   // running maximum over the splits seen so far and the sink
    // Splits in batches of kGroups * kBatch (256 for 152 or fewer splits: one batch).
    for (int base = 0; base < n_splits; base += kGroups * kBatch) {
        float4 o[kBatch];
        float l[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int s = base + group + kGroups * i;
            if (s < n_splits) {
                l[i] = __ldcg(part_lse + (long long)s * M + m);
                o[i] = __ldcg(reinterpret_cast<const float4*>(part_o + ((long long)s * M + m) * kD + col0));
            } else {
                l[i] = -INFINITY;
                o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        // maximum over this batch and the sink (whole block), then rescale what was accumulated so far
        float bm = sk;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) bm = fmaxf(bm, l[i]);
        for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        if (lane == 0) red[warp] = bm;
        __syncthreads();
        if (tid == 0) {
            float t = red[0];
            for (int i = 1; i < kCombineThreads / 32; ++i) t = fmaxf(t, red[i]);
            s_mx = t;
        }
        __syncthreads();
        const float nm = fmaxf(mx, s_mx);
        if (nm != -INFINITY) {
            const float a = (mx == -INFINITY) ? 0.0f : expf(mx - nm);
            acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
            z *= a;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const float w = (l[i] == -INFINITY) ? 0.0f : expf(l[i] - nm);
                acc.x = fmaf(w, o[i].x, acc.x);
                acc.y = fmaf(w, o[i].y, acc.y);
                acc.z = fmaf(w, o[i].z, acc.z);
                acc.w = fmaf(w, o[i].w, acc.w);
                z += w;
            }
        }
        mx = nm;
        __syncthreads();   // red / s_mx are reused by the next batch
    }
    part[group][chunk] = acc;
    if (chunk == 0) zpart[group] = z;
    __syncthreads();
    if (mx == -INFINITY) {   // nothing visible and no sink
        if (tid < kD / kQuarters) out[(long long)m * kD + quarter * (kD / kQuarters) + tid] = __float2bfloat16_rn(0.0f);
        if (out_lse && quarter == 0 && tid == 0) out_lse[m] = -INFINITY;
        return;
    }
    // Totals: output column o = 4 c + e (32 per quarter) is summed over the 32 groups by the 8 threads
    // 8 o .. 8 o + 7 (four groups each, then a fixed xor-shuffle tree); the 32 partial sums of z likewise.
    {
        const int o = tid >> 3, k = tid & 7, c = o >> 2, e = o & 3;
        float sum = 0.0f, zt = 0.0f;
#pragma unroll
        for (int i = 0; i < kGroups / 8; ++i) {
            const int g = k + 8 * i;
            const float4 v = part[g][c];
            sum += (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
            zt += zpart[g];
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, off);
            zt += __shfl_xor_sync(0xffffffffu, zt, off);
        }
        if (k == 0) {
            zt += (sk == -INFINITY) ? 0.0f : expf(sk - mx);
            out[(long long)m * kD + quarter * (kD / kQuarters) + o] = __float2bfloat16_rn(sum / zt);
            if (out_lse && quarter == 0 && o == 0) out_lse[m] = mx + logf(zt);
        }
    }
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                           int n_rows, int n_live, uint16_t* out, float* out_lse, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3(n_rows * kH, kQuarters), dim3(kCombineThreads), 0, stream);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, part_o, part_lse, n_splits, sink, n_rows, n_live,
                                             reinterpret_cast<__nv_bfloat16*>(out), out_lse);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
