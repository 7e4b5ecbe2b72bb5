// Log-sum-exp merge of the split partials with the learned sink folded in.
// IQuestRT report, "Read only the KV tiles needed by the current positions": a separate combine
// kernel issues the partial loads together and uses independent FP32 accumulation chains;
// "Expose more parallelism in attention": the combine applies the sink correction and keeps the
// BF16 rounding boundary (the output is rounded to bf16 once, here).
#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {

// Block shapes (measured inside the verify call on GB300): up to 8 verify rows (48 matrix rows x 4 column
// quarters = 192 CTAs), 128 threads with 10 splits per thread (one round of loads for up to 160 splits),
// at most two CTAs on an SM: 22.70 us per 192K call against 23.46 us for 512 threads with 5 splits each
// (which its registers also hold to two an SM; 23.47 for 256 x 5).  Alone, back to back on the same
// partials, the 128-thread combine takes 2.6 us against 3.8 us; inside the call, where its CTAs start on
// the SMs that the split kernel frees first, it was slower (+0.8 us) until it was held to two CTAs an SM
// (three: -0.4 us, two: -0.77 us; 64 threads x 20 splits, two an SM: -0.36 us).  The cap is a request
// for shared memory that the kernel does not use.  A 16-node tree has 96 matrix rows (384 CTAs): there
// 128 threads with 5 splits each, at most three CTAs an SM (the small, uncapped combine there: +0.61 us per
// 16-node tree call at 192K).
constexpr int kQuarters = 4;                       // column quarters of a matrix row: 32 columns each
constexpr int kChunks = kD / kQuarters / 4;        // float4 chunks per quarter: 8
constexpr float kLog2e = 1.4426950408889634f;

// One CTA per (matrix row m = 6 r + h, column quarter).  Thread t owns float4 chunk t % 8 of the quarter
// and the splits s = t / 8 + kGroups i: it issues all of its partial and LSE loads before using any of them.
// Each warp merges its own splits against its own maximum (a two-level log-sum-exp merge), so the CTA
// needs one barrier: the warp totals are then rescaled to the CTA maximum (which includes the sink) and
// added in a fixed order: out = sum_s e^(lse_s - M) o_s / (sum_s e^(lse_s - M) + e^(sink - M)).  The
// exponentials are the hardware exp2 of log2e-scaled differences (the library exp costs a dependent chain
// of ~30 instructions per weight, which showed as ~1 us of the combine's time).
// Up to VA_COMBINE_SMALL splits (0: never), combine blocks of 128 threads at no more than 48 registers: small
// enough to sit on an SM beside a split-attention CTA (which holds 168 x 352 of the SM's 65,536 registers), so
// that the next call's split CTAs can start while this combine runs, and with 16 x 5 = 80 splits per load
// batch still one round of loads.  Measured on GB300 per verify call: 1K 10.09 -> 9.34 us, the 4,103-position
// window 10.72 -> 9.71 us; at 152 splits (two batches) +1.8 us, hence the bound.
#ifndef VA_COMBINE_SMALL
#define VA_COMBINE_SMALL 80
#endif
// VA_COMBINE_WARP: up to 48 splits, one warp per (matrix row, column quarter) with about splits / 4 splits a
// lane (combine_warp_kernel; 0: the 128-thread combine): measured on GB300 per verify call, 1K (9 splits)
// 8.43 -> 7.91 us, the 4,103-position window (33 splits) 9.14 -> 8.78 us, 4K (33) 8.66 -> 8.28 us,
// quantised 1K 9.40 -> 8.88 us; at 8K (65 splits, 20 a lane) it was 0.41 us slower than the 128-thread one.
#ifndef VA_COMBINE_WARP
#define VA_COMBINE_WARP 1
#endif
// VA_COMBINE_WARP_TREE: the one-warp combine also for more than 8 rows (trees; 16-node tree call at a 2K
// context, 17 splits: 10.10 -> 8.92 us).
#ifndef VA_COMBINE_WARP_TREE
#define VA_COMBINE_WARP_TREE 1
#endif
// Shape of the combine above 8 rows (trees) beyond the one-warp combine: threads and splits per thread (16-node
// tree call at 192K, 76 splits: 35.36 us with 256 x 8, 35.07 with 256 x 3, 34.64 with 128 x 5).
#ifndef VA_COMBINE_TREE_THREADS
#define VA_COMBINE_TREE_THREADS 128
#endif
#ifndef VA_COMBINE_TREE_BATCH
#define VA_COMBINE_TREE_BATCH 5
#endif
// Shape of the combine for more splits (up to 8 verify rows): threads per CTA and splits per thread.
#ifndef VA_COMBINE_BIG_THREADS
#define VA_COMBINE_BIG_THREADS 128
#endif
#ifndef VA_COMBINE_BIG_BATCH
#define VA_COMBINE_BIG_BATCH 10
#endif
// Dynamic shared memory requested by each of those CTAs (unused): it caps how many share an SM (80 KB: two
// of the 228 KB).  The same for the combine of more than 8 rows (trees, 60 KB: three an SM, -0.12 us per
// 16-node tree call at 192K; 0: no cap).
#ifndef VA_COMBINE_BIG_SMEM
#define VA_COMBINE_BIG_SMEM 81920
#endif
#ifndef VA_COMBINE_TREE_SMEM
#define VA_COMBINE_TREE_SMEM 61440
#endif


template <int kCombineThreads, int kBatch, int kMinBlocks = 1>   // kBatch: splits per thread loaded together
__global__ void __launch_bounds__(kCombineThreads, kMinBlocks) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  int n_splits, const float* __restrict__ sink,
                                                                  int n_rows, int n_live,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ out_lse) {
    constexpr int kGroups = kCombineThreads / kChunks;   // split groups
    constexpr int kWarps = kCombineThreads / 32;
    static_assert(kCombineThreads % 32 == 0 && kD / kQuarters <= kCombineThreads, "combine shape");
    __shared__ float4 part[kWarps][kChunks];   // per warp, per chunk: weighted sums (against the warp max)
    __shared__ float zpart[kWarps];            // per warp: sum of weights
    __shared__ float wmax[kWarps];             // per warp: its maximum lse
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
    float z = 0.0f, mx = -INFINITY;   // this warp's running maximum over the splits it has merged
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
        float bm = mx;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) bm = fmaxf(bm, l[i]);
        for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
        if (bm != -INFINITY) {
            const float a = (mx == -INFINITY) ? 0.0f : ptx::ex2((mx - bm) * kLog2e);
            acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
            z *= a;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const float w = (l[i] == -INFINITY) ? 0.0f : ptx::ex2((l[i] - bm) * kLog2e);
                acc.x = fmaf(w, o[i].x, acc.x);
                acc.y = fmaf(w, o[i].y, acc.y);
                acc.z = fmaf(w, o[i].z, acc.z);
                acc.w = fmaf(w, o[i].w, acc.w);
                z += w;
            }
            mx = bm;
        }
    }
    // within the warp: lanes with the same chunk (lane % kChunks) hold different splits -> add them
#pragma unroll
    for (int off = kChunks; off < 32; off <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
        z += __shfl_xor_sync(0xffffffffu, z, off);
    }
    if (lane < kChunks) part[warp][lane] = acc;
    if (lane == 0) {
        zpart[warp] = z;
        wmax[warp] = mx;
    }
    __syncthreads();
    // totals: thread o < 32 owns output column quarter*32 + o = chunk o/4, element o%4
    if (tid < kD / kQuarters) {
        const int c = tid >> 2, e = tid & 3;
        float M_ = sk;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M_ = fmaxf(M_, wmax[w]);
        float* dst_lse = (out_lse && quarter == 0 && tid == 0) ? out_lse + m : nullptr;
        __nv_bfloat16* dst = out + (long long)m * kD + quarter * (kD / kQuarters) + tid;
        if (M_ == -INFINITY) {   // nothing visible and no sink
            *dst = __float2bfloat16_rn(0.0f);
            if (dst_lse) *dst_lse = -INFINITY;
            return;
        }
        float sum = 0.0f, zt = (sk == -INFINITY) ? 0.0f : ptx::ex2((sk - M_) * kLog2e);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            if (wmax[w] == -INFINITY) continue;
            const float a = ptx::ex2((wmax[w] - M_) * kLog2e);
            const float4 v = part[w][c];
            sum = fmaf(a, (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w, sum);
            zt = fmaf(a, zpart[w], zt);
        }
        *dst = __float2bfloat16_rn(sum / zt);
        if (dst_lse) *dst_lse = M_ + logf(zt);
    }
}

// One warp per (matrix row, column quarter) for few splits (up to 4 x kBatch): lane = (split group g, float4
// chunk c); the lane loads the lse and chunk c of splits g, g + 4, ... at once, the warp takes the maximum
// over every split and the sink, weighs, and adds the four groups by shuffles; no shared memory and no
// block barrier.  Lanes 0..7 store the quarter's 32 columns.
template <int kBatch>
__global__ void __launch_bounds__(32) combine_warp_kernel(const float* __restrict__ part_o,
                                                         const float* __restrict__ part_lse, int n_splits,
                                                         const float* __restrict__ sink, int n_rows, int n_live,
                                                         __nv_bfloat16* __restrict__ out, float* __restrict__ out_lse) {
    const int m = blockIdx.x, quarter = blockIdx.y;
    const int r = m / kH, h = m - r * kH;
    const int lane = threadIdx.x, chunk = lane & (kChunks - 1), group = lane >> 3;
    const int M = n_rows * kH;
    const int col0 = quarter * (kD / kQuarters) + 4 * chunk;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();   // every global access comes after this
    __nv_bfloat16* dst = out + (long long)m * kD + col0;
    if (r >= n_live) {
        if (group == 0) {
            const __nv_bfloat162 z2 = __floats2bfloat162_rn(0.0f, 0.0f);
            reinterpret_cast<__nv_bfloat162*>(dst)[0] = z2;
            reinterpret_cast<__nv_bfloat162*>(dst)[1] = z2;
        }
        if (out_lse && quarter == 0 && lane == 0) out_lse[m] = -INFINITY;
        return;
    }
    const float sk = sink ? __ldcg(sink + h) : -INFINITY;
    float4 o[kBatch];
    float l[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
        const int s = group + 4 * i;
        if (s < n_splits) {
            l[i] = __ldcg(part_lse + (long long)s * M + m);
            o[i] = __ldcg(reinterpret_cast<const float4*>(part_o + ((long long)s * M + m) * kD + col0));
        } else {
            l[i] = -INFINITY;
            o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    float mx = sk;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) mx = fmaxf(mx, l[i]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    if (mx == -INFINITY) {   // nothing visible and no sink
        if (group == 0) {
            const __nv_bfloat162 z2 = __floats2bfloat162_rn(0.0f, 0.0f);
            reinterpret_cast<__nv_bfloat162*>(dst)[0] = z2;
            reinterpret_cast<__nv_bfloat162*>(dst)[1] = z2;
        }
        if (out_lse && quarter == 0 && lane == 0) out_lse[m] = -INFINITY;
        return;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
        const float w = (l[i] == -INFINITY) ? 0.0f : ptx::ex2((l[i] - mx) * kLog2e);
        acc.x = fmaf(w, o[i].x, acc.x);
        acc.y = fmaf(w, o[i].y, acc.y);
        acc.z = fmaf(w, o[i].z, acc.z);
        acc.w = fmaf(w, o[i].w, acc.w);
        z += w;
    }
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
        z += __shfl_xor_sync(0xffffffffu, z, off);
    }
    if (sk != -INFINITY) z += ptx::ex2((sk - mx) * kLog2e);
    if (group == 0) {
        reinterpret_cast<__nv_bfloat162*>(dst)[0] = __floats2bfloat162_rn(acc.x / z, acc.y / z);
        reinterpret_cast<__nv_bfloat162*>(dst)[1] = __floats2bfloat162_rn(acc.z / z, acc.w / z);
    }
    if (out_lse && quarter == 0 && lane == 0) out_lse[m] = mx + logf(z);
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                           int n_rows, int n_live, uint16_t* out, float* out_lse, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    const bool wide = n_rows <= kMaxRows;
#if VA_COMBINE_WARP
    if ((wide || VA_COMBINE_WARP_TREE) && n_splits <= 48) {
        // the instantiation with the fewest splits a lane that covers n_splits (unused load slots cost time:
        // 1K call 8.29 us with 12 a lane, 7.90 us with 3)
        pdl_config(&cfg, attr, dim3(n_rows * kH, kQuarters), dim3(32), 0, stream);
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
        const int b = (n_splits + 3) / 4;
        void (*fn)(const float*, const float*, int, const float*, int, int, __nv_bfloat16*, float*) =
            b <= 1 ? combine_warp_kernel<1> : b <= 2 ? combine_warp_kernel<2> : b <= 3 ? combine_warp_kernel<3>
            : b <= 4 ? combine_warp_kernel<4> : b <= 6 ? combine_warp_kernel<6> : b <= 9 ? combine_warp_kernel<9>
            : combine_warp_kernel<12>;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, part_o, part_lse, n_splits, sink, n_rows, n_live, o, out_lse);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
#endif
#if VA_COMBINE_SMALL
    if (wide && n_splits <= VA_COMBINE_SMALL) {
        pdl_config(&cfg, attr, dim3(n_rows * kH, kQuarters), dim3(128), 0, stream);
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel<128, 5, 10>, part_o, part_lse, n_splits, sink,
                                                 n_rows, n_live, o, out_lse);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
#endif
    const int smem = wide ? VA_COMBINE_BIG_SMEM : VA_COMBINE_TREE_SMEM;
    pdl_config(&cfg, attr, dim3(n_rows * kH, kQuarters), dim3(wide ? VA_COMBINE_BIG_THREADS : VA_COMBINE_TREE_THREADS),
               smem, stream);
    if (smem > 0) {   // (the kernel's static shared memory counts toward the 48 KB default limit too)
        const cudaError_t ea = ensure_smem_attr(wide ? (const void*)combine_kernel<VA_COMBINE_BIG_THREADS, VA_COMBINE_BIG_BATCH>
                                                     : (const void*)combine_kernel<VA_COMBINE_TREE_THREADS,
                                                                                   VA_COMBINE_TREE_BATCH>, smem);
        if (ea != cudaSuccess) return ea;
    }
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
    const cudaError_t e =
        wide ? cudaLaunchKernelEx(&cfg, combine_kernel<VA_COMBINE_BIG_THREADS, VA_COMBINE_BIG_BATCH>, part_o, part_lse,
                                  n_splits, sink, n_rows, n_live, o, out_lse)
             : cudaLaunchKernelEx(&cfg, combine_kernel<VA_COMBINE_TREE_THREADS, VA_COMBINE_TREE_BATCH>, part_o, part_lse,
                                  n_splits, sink, n_rows, n_live, o, out_lse);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
