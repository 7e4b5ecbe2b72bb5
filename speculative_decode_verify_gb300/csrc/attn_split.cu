// Split-KV verify attention: 48 matrix rows (8 verify rows x 6 query heads) against one KV head.
// IQuestRT report, "Read only the KV tiles needed by the current positions": rows and heads are
// folded into 48 matrix rows that reuse each K/V tile; the sequence is partitioned across CTAs;
// only the valid extent is read, with a causal (or window) mask at the boundary.
//
// This translation unit holds the first, CUDA-core version of the split kernel: one CTA per
// split, K/V tiles of 64 positions staged in shared memory as fp32, scores and the online
// softmax in fp32.  Keys outside the split's visible range are neither loaded nor weighted.
#include <cuda_bf16.h>

#include "va_internal.cuh"

namespace va {

namespace simple {

constexpr int kThreads = 256;
constexpr int kKStride = kD + 1;  // padded row of the fp32 K tile

struct Smem {
    float q[kMaxM][kD];
    float k[kTile][kKStride];
    float v[kTile][kD];
    float p[kMaxM][kTile];
    float m[kMaxM], l[kMaxM], alpha[kMaxM];
    long long row_lo[kMaxRows], row_hi[kMaxRows];  // visible positions of each row: [lo, hi)
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

__global__ void __launch_bounds__(kThreads) split_kernel(AttnArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int M = a.n_rows * kH;
    const int live_m = a.n_live * kH;

    const Plan P = make_plan(a.pos, a.n_live, a.window, a.slots, a.n_splits, split);
    if (P.status && tid == 0 && split == 0 && a.dev_status) atomicOr(a.dev_status, P.status);

    // positions owned by this split, clipped to the extent
    const long long own_lo = max(P.lo, P.t0 * kTile);
    const long long own_hi = min(P.hi, P.t1 * kTile);

    for (int i = tid; i < M * kD; i += kThreads) sm.q[i / kD][i % kD] = bf16_bits_to_float(a.q[i]);
    if (tid < kMaxRows) {
        long long lo = 0, hi = 0;
        if (tid < a.n_live && P.status == 0) {
            const long long p = a.pos[tid];
            lo = a.window > 0 ? max(0LL, p - a.window + 1) : 0LL;
            hi = p + 1;
            lo = max(lo, own_lo);
            hi = min(hi, own_hi);
        }
        sm.row_lo[tid] = lo;
        sm.row_hi[tid] = hi;
    }
    if (tid < kMaxM) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.0f;
        sm.alpha[tid] = 1.0f;
    }

    // O accumulator: thread owns column d of rows [r0, r0 + 24)
    const int od = tid & (kD - 1);
    const int orow0 = (tid >> 7) * (kMaxM / 2);
    float acc[kMaxM / 2];
#pragma unroll
    for (int i = 0; i < kMaxM / 2; ++i) acc[i] = 0.0f;

    const long long t_begin = P.status ? 0 : P.t0;
    const long long t_end = P.status ? 0 : P.t1;
    for (long long t = t_begin; t < t_end; ++t) {
        const long long base = t * kTile;
        __syncthreads();
        // stage K and V rows of this tile that lie in the split's owned range; zero the rest
        for (int i = tid; i < kTile * kD; i += kThreads) {
            const int j = i / kD, d = i % kD;
            const long long p = base + j;
            float kv = 0.0f, vv = 0.0f;
            if (p >= own_lo && p < own_hi) {
                const long long slot = p % a.slots;
                kv = bf16_bits_to_float(a.k[slot * kD + d]);
                vv = bf16_bits_to_float(a.v[slot * kD + d]);
            }
            sm.k[j][d] = kv;
            sm.v[j][d] = vv;
        }
        __syncthreads();
        // scores: thread -> key j, 12 matrix rows
        {
            const int j = tid & (kTile - 1);
            const int g = tid >> 6;
            const long long p = base + j;
            for (int mi = 0; mi < kMaxM / 4; ++mi) {
                const int m = g * (kMaxM / 4) + mi;
                if (m >= M) break;
                const int r = m / kH;
                float s = -INFINITY;
                if (m < live_m && p >= sm.row_lo[r] && p < sm.row_hi[r]) {
                    float dot = 0.0f;
#pragma unroll 8
                    for (int d = 0; d < kD; ++d) dot = fmaf(sm.q[m][d], sm.k[j][d], dot);
                    s = dot * a.scale;
                }
                sm.p[m][j] = s;
            }
        }
        __syncthreads();
        // online softmax per matrix row: warp w takes rows w, w + 8, ...
        {
            const int warp = tid >> 5, lane = tid & 31;
            for (int m = warp; m < M; m += kThreads / 32) {
                const float s0 = sm.p[m][lane], s1 = sm.p[m][lane + 32];
                float mx = fmaxf(s0, s1);
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = sm.m[m];
                const float m_new = fmaxf(m_old, mx);
                float p0 = 0.0f, p1 = 0.0f, alpha = 1.0f;
                if (m_new != -INFINITY) {
                    p0 = expf(s0 - m_new);
                    p1 = expf(s1 - m_new);
                    alpha = expf(m_old - m_new);
                }
                float sum = p0 + p1;
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                sm.p[m][lane] = p0;
                sm.p[m][lane + 32] = p1;
                __syncwarp();
                if (lane == 0) {
                    sm.m[m] = m_new;
                    sm.l[m] = sm.l[m] * alpha + sum;
                    sm.alpha[m] = alpha;
                }
            }
        }
        __syncthreads();
        // O update: acc[row] = acc[row] * alpha + sum_j p[row][j] * v[j][d]
        for (int i = 0; i < kMaxM / 2; ++i) {
            const int m = orow0 + i;
            if (m >= M) break;
            float o = acc[i] * sm.alpha[m];
#pragma unroll 8
            for (int j = 0; j < kTile; ++j) o = fmaf(sm.p[m][j], sm.v[j][od], o);
            acc[i] = o;
        }
    }
    __syncthreads();
    // epilogue: normalised partial and its natural-log LSE
    float* po = a.part_o + (long long)split * M * kD;
    for (int i = 0; i < kMaxM / 2; ++i) {
        const int m = orow0 + i;
        if (m >= M) break;
        const float l = sm.l[m];
        po[(long long)m * kD + od] = l > 0.0f ? acc[i] / l : 0.0f;
    }
    if (tid < M) {
        const float l = sm.l[tid];
        a.part_lse[(long long)split * M + tid] = l > 0.0f ? sm.m[tid] + logf(l) : -INFINITY;
    }
}

}  // namespace simple

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(simple::Smem);
    cudaError_t e = ensure_smem_attr((const void*)simple::split_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    simple::split_kernel<<<a.n_splits, simple::kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace va
