// Split-KV verify attention on the sm_100-family tensor cores (tcgen05 + TMA + TMEM).
//
// IQuestRT report, "Read only the KV tiles needed by the current positions": eight verify rows x six
// query heads are folded into 48 matrix rows that reuse every K/V tile; the sequence is partitioned
// across CTAs; the read extent comes from the current positions and the causal (or window) mask is
// applied at the boundary; each split writes a normalised partial and its log-sum-exp for a separate
// combine ("Expose more parallelism in attention").
//
// Design for one GB300 SM per split:
//   * Transposed products so that the 128-row MMA dimension is always full: for a tile of 128 keys,
//     S^T[128 keys x 48 rows] = K[128 x 128] . Q^T, and O^T[128 d x 48 rows] += V^T . P^T.  Both
//     accumulators live in tensor memory (TMEM); S^T is double-buffered, O^T accumulates over tiles.
//   * A TMA warp streams 64-position boxes of K and V (128-byte swizzle) into a 3-deep K ring and a
//     2-deep V ring; K and V complete separate barriers, so QK starts as soon as K has landed.
//   * One thread issues the MMAs; four softmax warps own one TMEM lane quadrant each: thread L holds
//     key L of the tile for S^T and output column d = L for O^T.
//   * Softmax keeps one reference maximum per matrix row, shared by the CTA.  Scores may exceed it by up
//     to 2^8 before it is raised (a CTA-wide vote); raising it rescales the TMEM accumulator and the
//     running sums.  The log-sum-exp stays exact: lse = ref + log2(sum) in base-2 units.
//   * P is split into bf16 hi + lo parts (two MMAs into the same accumulator), so the probabilities
//     enter the product with ~2^-17 relative error instead of bf16's 2^-9.
//   * K/V rows outside the split's owned positions (the unaligned ends of the extent: cache capacity
//     beyond the valid history, or ring slots outside the window) are zeroed in shared memory before
//     PV, so that garbage or NaN there cannot reach the accumulator through a zero probability.
//   * Every wait is bounded (VA_DEV_TIMEOUT); a timed-out CTA drains its own copies and MMAs, frees its
//     TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {
namespace tc {

constexpr int kNK = 3;                    // K ring depth (tiles of 128 positions)
constexpr int kNV = 2;                    // V ring depth
constexpr uint32_t kHalfBox = 8192;       // one TMA box: 64 positions x 64 columns x 2 B
constexpr uint32_t kDHalf = 16384;        // 128 positions x 64 columns: one column half of a stage
constexpr uint32_t kStage = 32768;        // K or V of one 128-position tile
constexpr uint32_t kQHalf = 6144;         // 48 rows x 64 columns
constexpr uint32_t kQBytes = 2 * kQHalf;
constexpr uint32_t kPBytes = 16384;       // P^T: 128 keys x 64 columns (48 used), 128-byte swizzle
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kNK * kStage;
constexpr uint32_t kOffQ = kOffV + kNV * kStage;
constexpr uint32_t kOffPhi = kOffQ + kQBytes;
constexpr uint32_t kOffPlo = kOffPhi + kPBytes;
constexpr uint32_t kOffMisc = kOffPlo + kPBytes;
constexpr int kThreads = 192;             // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 softmax
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128;
constexpr float kThresh = 8.0f;           // log2 headroom above the reference maximum
constexpr float kRefInit = -1.0e30f;      // reference maximum before any visible key
constexpr uint64_t kWaitNs = 2000000000ull;

struct Misc {
    uint64_t k_full[kNK], k_empty[kNK], v_full[kNV], v_empty[kNV];
    uint64_t s_full[2], s_free[2], p_full, pv_done, drain;
    uint32_t tmem_base;
    int abort;
    int vote[2][4];
    float red[4][kMaxM];
    float ref[kMaxM];
    float alpha[kMaxM];
    long long row_lo[kMaxRows], row_hi[kMaxRows];
};
constexpr uint32_t kSmemBytes = kOffMisc + (uint32_t)sizeof(Misc) + 1024;
static_assert(kOffQ % 1024 == 0 && kOffPhi % 1024 == 0 && kOffPlo % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

// Column base of the three columns a lane holds after warp_reduce_scatter48.
__device__ __forceinline__ int scatter_col_base(int lane) {
    return ((lane >> 4) & 1) * 24 + ((lane >> 3) & 1) * 12 + ((lane >> 2) & 1) * 6 + ((lane >> 1) & 1) * 3;
}

// Reduce 48 per-thread columns over the warp; afterwards lane holds the warp totals of columns
// [scatter_col_base(lane), +3) in v[0..2] (lanes 2i and 2i+1 hold the same three).
template <bool kMax>
__device__ __forceinline__ void warp_reduce_scatter48(float (&v)[48], int lane) {
#define VA_STAGE(W, BIT)                                                   \
    _Pragma("unroll") for (int i = 0; i < (W); ++i) {                      \
        const bool up = (lane & (BIT)) != 0;                               \
        const float send = up ? v[i] : v[i + (W)];                         \
        const float keep = up ? v[i + (W)] : v[i];                         \
        const float got = __shfl_xor_sync(0xffffffffu, send, (BIT));       \
        v[i] = kMax ? fmaxf(keep, got) : keep + got;                       \
    }
    VA_STAGE(24, 16)
    VA_STAGE(12, 8)
    VA_STAGE(6, 4)
    VA_STAGE(3, 2)
#undef VA_STAGE
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const float got = __shfl_xor_sync(0xffffffffu, v[i], 1);
        v[i] = kMax ? fmaxf(v[i], got) : v[i] + got;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    Misc& ms = *reinterpret_cast<Misc*>(base + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x;
    const int M = a.n_rows * kH;      // matrix rows present in q / the partials
    const int ML = a.n_live * kH;     // live matrix rows

    const Plan P = make_plan(a.pos, a.n_live, a.window, a.slots, a.n_splits, split);
    if (P.status && split == 0 && tid == 0 && a.dev_status) atomicOr(a.dev_status, P.status);
    const int n64 = P.status ? 0 : (int)(P.t1 - P.t0);
    const int ntiles = (n64 + 1) >> 1;
    float* part_o = a.part_o + (long long)split * M * kD;
    float* part_lse = a.part_lse + (long long)split * M;
    if (ntiles == 0) {  // empty split (or unusable positions): o = 0, lse = -inf
        for (int i = tid; i < M * kD; i += kThreads) part_o[i] = 0.0f;
        for (int i = tid; i < M; i += kThreads) part_lse[i] = -INFINITY;
        return;
    }
    const long long own_lo = max(P.lo, P.t0 * kTile);
    const long long own_hi = min(P.hi, P.t1 * kTile);

    // ---------------------------------------------------------------- one-time set-up
    if (tid < kMaxRows) {
        long long lo = 0, hi = 0;
        if (tid < a.n_live) {
            const long long p = __ldg(a.pos + tid);
            lo = a.window > 0 ? max(0LL, p - a.window + 1) : 0LL;
            hi = p + 1;
            lo = max(lo, own_lo);
            hi = min(hi, own_hi);
            if (hi < lo) hi = lo;
        }
        ms.row_lo[tid] = lo;
        ms.row_hi[tid] = hi;
    }
    if (tid < kMaxM) ms.ref[tid] = kRefInit;
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&ms.tmem_base), kTmemCols);
    if (tid == 0) {
        for (int i = 0; i < kNK; ++i) {
            ptx::mbar_init(ptx::smem_u32(&ms.k_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&ms.k_empty[i]), 1);
        }
        for (int i = 0; i < kNV; ++i) {
            ptx::mbar_init(ptx::smem_u32(&ms.v_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&ms.v_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(ptx::smem_u32(&ms.s_full[i]), 1);
            ptx::mbar_init(ptx::smem_u32(&ms.s_free[i]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&ms.p_full), 4);
        ptx::mbar_init(ptx::smem_u32(&ms.pv_done), 1);
        ptx::mbar_init(ptx::smem_u32(&ms.drain), 1);
        ms.abort = 0;
        ptx::mbar_init_fence();
    }
    if (tid == 32) {
        ptx::tma_prefetch_desc(&tmk);
        ptx::tma_prefetch_desc(&tmv);
    }
    {   // Q: 48 rows x 256 B in two 64-column halves, 128-byte swizzle; rows beyond n_rows are zero
        const uint4* q4 = reinterpret_cast<const uint4*>(a.q);
        for (int i = tid; i < kMaxM * 16; i += kThreads) {
            const int m = i >> 4, c = i & 15;
            const uint4 val = (m < M) ? __ldg(q4 + m * 16 + c) : make_uint4(0u, 0u, 0u, 0u);
            const int cc = c & 7;
            const uint32_t off = kOffQ + (uint32_t)(c >> 3) * kQHalf + (uint32_t)(m >> 3) * 1024u +
                                 (uint32_t)(m & 7) * 128u + ((uint32_t)(cc ^ (m & 7)) << 4);
            *reinterpret_cast<uint4*>(base + off) = val;
        }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    volatile int* abort_flag = &ms.abort;
    auto bar = [](const uint64_t& b) { return ptx::smem_u32(&b); };
    auto fail = [&]() {
        *abort_flag = 1;
        if (a.dev_status) atomicOr(a.dev_status, VA_DEV_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const long long t = P.t0 + 2LL * j;
                const int halves = (t + 1 < P.t1) ? 2 : 1;
                const int ks = j % kNK;
                if (!ptx::mbar_wait(bar(ms.k_empty[ks]), ((j / kNK) & 1) ^ 1, abort_flag, kWaitNs)) {
                    fail();
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(ms.k_full[ks]), (uint32_t)halves * 2u * kHalfBox);
                for (int hh = 0; hh < halves; ++hh) {
                    const int slot = (int)(((t + hh) * kTile) % a.slots);
                    for (int h = 0; h < 2; ++h)
                        ptx::tma_load_2d(base_s + kOffK + ks * kStage + h * kDHalf + hh * kHalfBox, &tmk, h * 64, slot,
                                         bar(ms.k_full[ks]));
                }
                k_issued = j + 1;
                const int vs = j % kNV;
                if (!ptx::mbar_wait(bar(ms.v_empty[vs]), ((j / kNV) & 1) ^ 1, abort_flag, kWaitNs)) {
                    fail();
                    break;
                }
                ptx::mbar_arrive_expect_tx(bar(ms.v_full[vs]), (uint32_t)halves * 2u * kHalfBox);
                for (int hh = 0; hh < halves; ++hh) {
                    const int slot = (int)(((t + hh) * kTile) % a.slots);
                    for (int h = 0; h < 2; ++h)
                        ptx::tma_load_2d(base_s + kOffV + vs * kStage + h * kDHalf + hh * kHalfBox, &tmv, h * 64, slot,
                                         bar(ms.v_full[vs]));
                }
                v_issued = j + 1;
            }
            // every issued copy has landed before this CTA may exit
            for (int j = max(0, k_issued - kNK); j < k_issued; ++j)
                ptx::mbar_wait(bar(ms.k_full[j % kNK]), (j / kNK) & 1, nullptr, kWaitNs);
            for (int j = max(0, v_issued - kNV); j < v_issued; ++j)
                ptx::mbar_wait(bar(ms.v_full[j % kNV]), (j / kNV) & 1, nullptr, kWaitNs);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 48, 0, 0);   // A = K, B = Q: both K-major
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, 48, 1, 1);   // A = V^T, B = P^T: MN-major
            bool ok = true;
            for (int j = 0; j <= ntiles && ok; ++j) {
                if (j < ntiles) {
                    const int ks = j % kNK, sb = j & 1;
                    ok = ptx::mbar_wait(bar(ms.k_full[ks]), (j / kNK) & 1, abort_flag, kWaitNs) &&
                         ptx::mbar_wait(bar(ms.s_free[sb]), ((j >> 1) & 1) ^ 1, abort_flag, kWaitNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const uint32_t d = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t h = (uint32_t)kk >> 2, off = (uint32_t)(kk & 3) * 32u;
                        ptx::mma_bf16(d, ptx::smem_desc(base_s + kOffK + ks * kStage + h * kDHalf + off, 0, 1024),
                                      ptx::smem_desc(base_s + kOffQ + h * kQHalf + off, 0, 1024), idesc_qk, kk > 0);
                    }
                    ptx::mma_commit(bar(ms.s_full[sb]));
                    ptx::mma_commit(bar(ms.k_empty[ks]));
                }
                if (j >= 1) {
                    const int i = j - 1, vs = i % kNV;
                    ok = ptx::mbar_wait(bar(ms.v_full[vs]), (i / kNV) & 1, abort_flag, kWaitNs) &&
                         ptx::mbar_wait(bar(ms.p_full), i & 1, abort_flag, kWaitNs);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    const long long t = P.t0 + 2LL * i;
                    const int nk = (t + 1 < P.t1) ? 8 : 4;
                    for (int kk = 0; kk < nk; ++kk) {
                        const uint64_t adesc = ptx::smem_desc(base_s + kOffV + vs * kStage + kk * 2048, kDHalf, 1024);
                        ptx::mma_bf16(tmem + kColO, adesc, ptx::smem_desc(base_s + kOffPhi + kk * 2048, 8192, 1024),
                                      idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                        ptx::mma_bf16(tmem + kColO, adesc, ptx::smem_desc(base_s + kOffPlo + kk * 2048, 8192, 1024),
                                      idesc_pv, 1u);
                    }
                    ptx::mma_commit(bar(ms.pv_done));
                    ptx::mma_commit(bar(ms.v_empty[vs]));
                }
            }
            if (!ok) fail();
            ptx::mma_commit(bar(ms.drain));   // all MMAs of this CTA done before TMEM is freed
            ptx::mbar_wait(bar(ms.drain), 0, nullptr, kWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / accumulator warps
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int wq = warp - 2;
        const int L = q * 32 + lane;          // key of the tile (S^T) and output column d (O^T)
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        const float c = a.scale * 1.4426950408889634f;   // scores in log2 units
        long long all_lo = own_lo, all_hi = own_hi;
        for (int r = 0; r < a.n_live; ++r) {
            all_lo = max(all_lo, ms.row_lo[r]);
            all_hi = min(all_hi, ms.row_hi[r]);
        }
        float ref[kMaxM], l[kMaxM];
#pragma unroll
        for (int n = 0; n < kMaxM; ++n) {
            ref[n] = kRefInit;
            l[n] = 0.0f;
        }
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const long long t = P.t0 + 2LL * j;
            const int nkeys = (t + 1 < P.t1) ? 128 : 64;
            const long long kbase = t * kTile;
            const long long kp = kbase + L;
            const int sb = j & 1;
            if (!ptx::mbar_wait(bar(ms.s_full[sb]), (j >> 1) & 1, abort_flag, kWaitNs)) ok = false;
            ptx::tc_fence_after();
            float x[kMaxM];
            ptx::tmem_ld48_wait(tl + (sb ? kColS1 : kColS0), x);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.s_free[sb]));

            // masked scores in log2 units
            if (kbase >= all_lo && kbase + nkeys <= all_hi) {
                // every live row sees every key of the tile; lanes past a half tile hold stale rows
                const bool key_in = L < nkeys;
#pragma unroll
                for (int n = 0; n < kMaxM; ++n) x[n] = (key_in && n < ML) ? x[n] * c : -INFINITY;
            } else {
                bool vis[kMaxRows];
#pragma unroll
                for (int r = 0; r < kMaxRows; ++r) vis[r] = (r < a.n_live) && kp >= ms.row_lo[r] && kp < ms.row_hi[r];
#pragma unroll
                for (int n = 0; n < kMaxM; ++n) x[n] = vis[n / kH] ? x[n] * c : -INFINITY;
            }
            // raise the reference maxima only when a score exceeds them by more than 2^kThresh
            float umax = -INFINITY;
#pragma unroll
            for (int n = 0; n < kMaxM; ++n) umax = fmaxf(umax, x[n] - ref[n]);
            const unsigned want = __any_sync(0xffffffffu, umax > kThresh);
            if (lane == 0) ms.vote[j & 1][wq] = want ? 1 : 0;
            ptx::named_bar_sync(1, 128);
            const bool rescale = (ms.vote[j & 1][0] | ms.vote[j & 1][1] | ms.vote[j & 1][2] | ms.vote[j & 1][3]) != 0;
            // PV(j-1) done: the P buffers may be rewritten and the accumulator is stable
            if (j > 0 && !ptx::mbar_wait(bar(ms.pv_done), (j - 1) & 1, abort_flag, kWaitNs)) ok = false;
            if (rescale) {
                float v[kMaxM];
#pragma unroll
                for (int n = 0; n < kMaxM; ++n) v[n] = x[n];
                warp_reduce_scatter48<true>(v, lane);
                const int cb = scatter_col_base(lane);
                if ((lane & 1) == 0) {
                    ms.red[wq][cb] = v[0];
                    ms.red[wq][cb + 1] = v[1];
                    ms.red[wq][cb + 2] = v[2];
                }
                ptx::named_bar_sync(1, 128);
                if (L < kMaxM) {
                    const float cm = fmaxf(fmaxf(ms.red[0][L], ms.red[1][L]), fmaxf(ms.red[2][L], ms.red[3][L]));
                    const float old = ms.ref[L];
                    const float nw = fmaxf(old, cm);
                    ms.alpha[L] = ptx::ex2(old - nw);
                    ms.ref[L] = nw;
                }
                ptx::named_bar_sync(1, 128);
#pragma unroll
                for (int n = 0; n < kMaxM; ++n) {
                    ref[n] = ms.ref[n];
                    l[n] *= ms.alpha[n];
                }
                if (j > 0) {
                    ptx::tc_fence_after();
#pragma unroll
                    for (int c16 = 0; c16 < 3; ++c16) {
                        float o[16];
                        ptx::tmem_ld16_wait(tl + kColO + 16 * c16, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] *= ms.alpha[16 * c16 + i];
                        ptx::tmem_st16(tl + kColO + 16 * c16, o);
                    }
                    ptx::tmem_wait_st();
                }
            }
            // probabilities; hi/lo bf16 split for the PV product
            uint32_t hi_w[kMaxM / 2], lo_w[kMaxM / 2];
#pragma unroll
            for (int i = 0; i < kMaxM / 2; ++i) {
                const float p0 = ptx::ex2(x[2 * i] - ref[2 * i]);
                const float p1 = ptx::ex2(x[2 * i + 1] - ref[2 * i + 1]);
                l[2 * i] += p0;
                l[2 * i + 1] += p1;
                const uint32_t hb = pack_bf16x2(p0, p1);
                hi_w[i] = hb;
                lo_w[i] = pack_bf16x2(p0 - __uint_as_float(hb << 16), p1 - __uint_as_float(hb & 0xFFFF0000u));
            }
            // V rows of positions this split does not own are zeroed before PV reads them
            const int vs = j % kNV;
            if (kbase < own_lo || kbase + nkeys > own_hi) {
                if (!ptx::mbar_wait(bar(ms.v_full[vs]), (j / kNV) & 1, abort_flag, kWaitNs)) ok = false;
                if (L < nkeys && (kp < own_lo || kp >= own_hi)) {
                    for (int h = 0; h < 2; ++h) {
                        uint4* row = reinterpret_cast<uint4*>(base + kOffV + vs * kStage + h * kDHalf +
                                                              (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u);
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) row[cc] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            // row L of P^T (keys x 48 matrix rows), 128-byte swizzle
            {
                const uint32_t roff = (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u;
#pragma unroll
                for (int cc = 0; cc < 6; ++cc) {
                    const uint32_t off = roff + ((uint32_t)(cc ^ (L & 7)) << 4);
                    *reinterpret_cast<uint4*>(base + kOffPhi + off) =
                        make_uint4(hi_w[4 * cc], hi_w[4 * cc + 1], hi_w[4 * cc + 2], hi_w[4 * cc + 3]);
                    *reinterpret_cast<uint4*>(base + kOffPlo + off) =
                        make_uint4(lo_w[4 * cc], lo_w[4 * cc + 1], lo_w[4 * cc + 2], lo_w[4 * cc + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.p_full));
        }
        // ------------------------------------------------------------ epilogue
        if (!ptx::mbar_wait(bar(ms.pv_done), (ntiles - 1) & 1, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        float o[kMaxM];
        ptx::tmem_ld48_wait(tl + kColO, o);
        warp_reduce_scatter48<false>(l, lane);
        {
            const int cb = scatter_col_base(lane);
            if ((lane & 1) == 0) {
                ms.red[wq][cb] = l[0];
                ms.red[wq][cb + 1] = l[1];
                ms.red[wq][cb + 2] = l[2];
            }
        }
        ptx::named_bar_sync(1, 128);
        if (L < kMaxM) ms.alpha[L] = (ms.red[0][L] + ms.red[1][L]) + (ms.red[2][L] + ms.red[3][L]);
        ptx::named_bar_sync(1, 128);
#pragma unroll
        for (int n = 0; n < kMaxM; ++n) {
            if (n < M) {
                const float lt = ms.alpha[n];
                part_o[n * kD + L] = lt > 0.0f ? o[n] / lt : 0.0f;
            }
        }
        if (L < M) {
            const float lt = ms.alpha[L];
            part_lse[L] = lt > 0.0f ? (ms.ref[L] + log2f(lt)) * 0.6931471805599453f : -INFINITY;
        }
        if (!ok) fail();
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// [slots][128] bf16 rows, boxes of 64 rows x 64 columns with the 128-byte swizzle; rows past the
// end read as zero.
bool encode_kv_map(CUtensorMap* map, const void* base, int slots) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)slots};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
    CUtensorMap tmk, tmv;
    if (!tc::encode_kv_map(&tmk, a.k, a.slots) || !tc::encode_kv_map(&tmv, a.v, a.slots)) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr((const void*)tc::attn_tc_kernel, (int)tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    tc::attn_tc_kernel<<<a.n_splits, tc::kThreads, tc::kSmemBytes, stream>>>(a, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace va
