// Sampling, acceptance and settlement: the steps after verification attention in a speculative round.
//
// IQuestRT report, "Include sampling and acceptance in the execution path" (top-k 20 / top-p 0.95 /
// temperature 1 over 160,000 logits; rejection sampling with min(1, p/q); replacement from
// max(0, p - q); bonus token; KV rollback inside the step) and "Parallelize the Top-K vocabulary
// scan" (8,192-logit tiles, per-tile candidates, ordered merge, tile maxima skip); "Qwen3.8-27B on one
// RTX 4090", "More tokens per round: verify trees".
//
// Top-k on GB300 (one launch; the last CTA of each row to finish its tile does the merge):
//   collect  one CTA per (8,192-logit tile, row): 256 threads x 32 logits from 128-bit loads.  Every
//            logit gets a 64-bit key (order-preserving value bits, then the complemented token id),
//            so keys are distinct and "larger key" is exactly the candidate order.  A lower bound of the
//            tile's k-th key comes from the per-thread maxima: in every warp, the j-th largest value by
//            j warp-wide max reductions (j = ceil(k / warps)), then the minimum over the warps (a tile
//            with fewer than 32 threads of logits takes the exact k-th largest thread maximum, by warp
//            bitonic sorts and binary searches); only logits at or above it are ranked.
//   merge    the row's last CTA: with m = ceil(k / tiles), the smallest of every tile's m-th key bounds
//            the row's k-th key from below (one warp's min-reduction); the keys at or above it are ranked
//            by counting; one warp then forms the float32 weights (one candidate per lane), the running
//            sums (in order, each lane reading the weights from shared memory), the top-p prefix and the
//            draw.
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_sample.h"
#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {
namespace smp {

// Each tile's logits pulled into L2 by a bulk prefetch before the launch dependency resolves (measured on
// GB300, 8 x 160,000 cold logits, graph-replayed: 11.01 -> 10.28 us per call).
#ifndef VA_SMP_PREWARM
#define VA_SMP_PREWARM 1
#endif
// The arrival of a tile: 1 one acquire-release atomic per CTA; 0 a fence, a relaxed atomic and, in the
// merging CTA, a second fence (measured on GB300, 8 x 160,000 logits: 11.28 -> 10.95 us per call).
#ifndef VA_SMP_ACQREL
#define VA_SMP_ACQREL 1
#endif

constexpr int kTileLogits = VA_SAMPLE_TILE;   // 8192
constexpr int kThreads = 256;
constexpr int kPerThread = kTileLogits / kThreads;   // 32
constexpr int kMaxK = VA_SAMPLE_MAX_K;        // 32
constexpr int kMaxCand = 256;                 // candidates ranked by counting; more take the slow path

// Order-preserving image of a float (NaN lowest, -0 == +0).
__device__ __forceinline__ uint32_t ord_bits(float f) {
    if (f != f) return 0u;
    uint32_t b = __float_as_uint(f);
    if ((b & 0x7FFFFFFFu) == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_to_float(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ uint64_t make_key(float f, int idx) {
    return ((uint64_t)ord_bits(f) << 32) | (uint32_t)(~(uint32_t)idx);
}
__device__ __forceinline__ int key_index(uint64_t key) { return (int)(~(uint32_t)(key & 0xFFFFFFFFu)); }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Sort the 32 keys of a warp, largest first (bitonic network over the lanes); returns this lane's key.
__device__ __forceinline__ uint64_t warp_sort_desc_u64(uint64_t v, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool lower = (lane & stride) == 0;           // this lane holds the lower index of the pair
            const bool desc = (lane & size) == 0;              // this block of the network sorts descending
            const bool keep_big = lower == desc;
            v = keep_big ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// k-th largest (1-based) of 256 distinct keys held one per thread.  Each warp sorts its 32 keys; the rank
// of a key is the number of larger keys in every warp's sorted list (a binary search each).
__device__ uint64_t block_kth_largest_u64(uint64_t v, int k, uint64_t* lists /*[8][32]*/, uint64_t* out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) *out = 0ull;   // the answer when it is one of several equal zero (empty-thread) keys
    const uint64_t s = warp_sort_desc_u64(v, lane);
    lists[warp * 32 + lane] = s;
    __syncthreads();
    // in every other list, the count of entries > s (lists are descending): a branchless binary search,
    // the eight searches interleaved step by step
    int cnt[kThreads / 32];
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) cnt[w] = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w)
            if (lists[w * 32 + cnt[w] + step - 1] > s) cnt[w] += step;
    }
    int rank = lane;   // larger keys in this warp's own list
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        // cnt counts entries > s among the first 31; the last entry decides the 32nd
        const int c = cnt[w] + ((cnt[w] == 31 && lists[w * 32 + 31] > s) ? 1 : 0);
        rank += (w == warp) ? 0 : c;
    }
    if (rank == k - 1) *out = s;
    __syncthreads();
    const uint64_t r = *out;
    __syncthreads();
    return r;
}

// Largest key over the block (each thread offers one).
__device__ uint64_t block_max_u64(uint64_t v, uint64_t* red /*[8]*/) {
    v = warp_max_u64(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint64_t m = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = red[w] > m ? red[w] : m;
    __syncthreads();
    return m;
}

constexpr int kMaxMerge = kMaxK * (VA_SAMPLE_MAX_VOCAB / kTileLogits);   // 32 tiles x 32 keys

struct TopkSmem {
    uint64_t cand[kMaxMerge];   // collection: candidates of the tile; merge: candidates of the row
    uint64_t all[kMaxMerge];    // merge: every tile's sorted keys
    uint64_t lists[kThreads];   // per-warp sorted thread maxima
    uint64_t red[kThreads / 32];
    uint32_t wmin[kThreads / 32];
    uint64_t top[kMaxK];
    uint64_t tau;
    float w[kMaxK], run[kMaxK];
    int n_cand;
    int last;
};

// Collection of one tile of one row, then - in the last CTA of the row to finish - the merge and the
// draw.  ws: [n_rows][n_tiles][k] sorted tile keys (largest first; 0 past the tile's logits); arrivals:
// [n_rows] arrival counters (zero between calls: the merging CTA resets its row's counter).
__global__ void __launch_bounds__(kThreads) topk_sample_kernel(const float* __restrict__ logits, int vocab, int k,
                                                               float top_p, float temperature,
                                                               const float* __restrict__ u, int32_t* __restrict__ ids,
                                                               float* __restrict__ probs, int32_t* __restrict__ counts,
                                                               int32_t* __restrict__ tokens, uint64_t* __restrict__ ws,
                                                               unsigned* __restrict__ arrivals) {
    __shared__ TopkSmem sm;
    const int tile = blockIdx.x, row = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_tiles = gridDim.x;
    ptx::griddep_launch_dependents();
#if VA_SMP_PREWARM
    // the tile's logits pulled into L2 while the kernel before may still run (a hint: the lines are read
    // again after the dependency resolves, so a prefetch of lines still being written costs nothing but
    // bandwidth)
    if (tid == 0) {
        const long long first = (long long)tile * kTileLogits;
        const long long n = min((long long)kTileLogits, (long long)vocab - first);
        if (n > 0) ptx::bulk_prefetch_l2(logits + (size_t)row * vocab + first, (uint32_t)(n * 4));
    }
#endif
    ptx::griddep_wait();
    const float4* src = reinterpret_cast<const float4*>(logits + (size_t)row * vocab);
    const int base4 = tile * (kTileLogits / 4);
    const int n4 = vocab / 4;
    uint64_t key[kPerThread];
    float4 val[kPerThread / 4];
#pragma unroll
    for (int i = 0; i < kPerThread / 4; ++i) {
        const int q = base4 + i * kThreads + tid;
        val[i] = q < n4 ? __ldcs(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kPerThread / 4; ++i) {
        const int q = base4 + i * kThreads + tid;
        const bool in = q < n4;
        const float f[4] = {val[i].x, val[i].y, val[i].z, val[i].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) key[4 * i + c] = in ? make_key(f[c], 4 * q + c) : 0ull;
    }
    uint64_t mx[kPerThread / 2];   // the thread maximum as a tree (short dependency chain)
#pragma unroll
    for (int i = 0; i < kPerThread / 2; ++i) mx[i] = key[2 * i] > key[2 * i + 1] ? key[2 * i] : key[2 * i + 1];
#pragma unroll
    for (int w = kPerThread / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) mx[i] = mx[i] > mx[i + w] ? mx[i] : mx[i + w];
    const uint64_t tmax = mx[0];
    if (tid == 0) sm.n_cand = 0;
    // threshold tau: a lower bound of the tile's k-th largest key, so that every key of the tile's top k is
    // at or above it.  With f warps whose 32 threads all hold logits, take j = ceil(k / f): in each such
    // warp, the j-th largest distinct value among its thread maxima (one warp-wide max per round, the
    // lanes at the maximum dropped), then the minimum over those warps.  Each of the f warps has at least
    // j threads whose maximum is at or above tau, so at least k distinct keys are: the k-th largest is.
    // Only the value bits are compared; all keys with the value are kept.  A tile with fewer than 32
    // threads of logits takes the exact k-th largest thread maximum (an empty thread offers key 0, below
    // every logit; a tile with fewer than k logits gets 0).
    uint64_t tau;
    const int full_warps = min(kThreads, max(0, n4 - base4)) / 32;
    if (full_warps > 0) {
        const int j = (k + full_warps - 1) / full_warps;
        uint32_t v = (uint32_t)(tmax >> 32), m = 0u;
        for (int r = 0; r < j; ++r) {
            m = __reduce_max_sync(0xffffffffu, v);
            v = (v == m) ? 0u : v;
        }
        if (lane == 0) sm.wmin[warp] = warp < full_warps ? m : 0xFFFFFFFFu;
        __syncthreads();
        uint32_t t = 0xFFFFFFFFu;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) t = min(t, sm.wmin[w]);
        tau = (uint64_t)t << 32;
    } else {
        tau = block_kth_largest_u64(tmax, k, sm.lists, &sm.tau);
    }
    // compact the keys at or above the threshold: per-thread count, warp scan, one atomic per warp
    unsigned mine = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) mine |= (key[i] != 0ull && key[i] >= tau) ? (1u << i) : 0u;
    const int cnt = __popc(mine);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    int wbase = 0;
    if (lane == 31 && incl > 0) wbase = atomicAdd(&sm.n_cand, incl);
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    int slot = wbase + incl - cnt;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        if ((mine >> i) & 1u) {
            if (slot < kMaxCand) sm.cand[slot] = key[i];
            ++slot;
        }
    }
    __syncthreads();
    const int nc = sm.n_cand;
    uint64_t* out = ws + ((size_t)row * n_tiles + tile) * k;
    if (nc <= kMaxCand) {
        // rank by counting: candidate c goes to position (number of larger candidates) if that is < k
        for (int c = tid; c < nc; c += kThreads) {
            const uint64_t kc = sm.cand[c];
            int rank = 0;
#pragma unroll 8
            for (int o = 0; o < nc; ++o) rank += sm.cand[o] > kc;
            if (rank < k) out[rank] = kc;
        }
        for (int r = nc + tid; r < k; r += kThreads) out[r] = 0ull;   // fewer than k logits in the tile
    } else {
        // many equal values at the threshold: k rounds of block-wide maximum over every logit
        uint64_t taken = ~0ull;   // keys below this one remain
        for (int r = 0; r < k; ++r) {
            uint64_t m = 0;
#pragma unroll
            for (int i = 0; i < kPerThread; ++i) m = (key[i] < taken && key[i] > m) ? key[i] : m;
            const uint64_t best = block_max_u64(m, sm.red);
            if (tid == 0) out[r] = best;
            taken = best;
        }
    }

    // ---------------------------------------------------------------- arrival: the last tile merges
    // (the block barrier orders every thread's key stores before thread 0's fence, which is cumulative:
    // they are visible before its arrival is)
    __syncthreads();
    if (tid == 0) {
#if VA_SMP_ACQREL
        // one acquire-release atomic: releases the block's key stores (ordered before it by the barrier),
        // and acquires the other tiles' for the merge below (the barrier passes that on to every thread)
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(arrivals + row) : "memory");
        sm.last = prev == (unsigned)(n_tiles - 1);
#else
        __threadfence();
        sm.last = atomicAdd(arrivals + row, 1u) == (unsigned)(n_tiles - 1);
#endif
    }
    __syncthreads();
    if (!sm.last) return;
    if (!VA_SMP_ACQREL) __threadfence();
    if (tid == 0) arrivals[row] = 0u;   // ready for the next call
    const uint64_t* rw = ws + (size_t)row * n_tiles * k;
    const int total = n_tiles * k;
    for (int e = tid; e < total; e += kThreads) sm.all[e] = __ldcg(rw + e);
    __syncthreads();
    // a lower bound of the row's k-th key: with m = ceil(k / tiles), the smallest of every tile's m-th key
    // (tiles x m >= k keys are at or above it); only keys at or above it are ranked
    if (tid < 32) {
        const int m = min(k, (k + n_tiles - 1) / n_tiles);
        uint64_t b = ~0ull;
        for (int t = lane; t < n_tiles; t += 32) {
            const uint64_t kv = sm.all[t * k + m - 1];
            b = kv < b ? kv : b;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t w = __shfl_xor_sync(0xffffffffu, b, o);
            b = w < b ? w : b;
        }
        if (lane == 0) {
            sm.tau = b;
            sm.n_cand = 0;
        }
    }
    __syncthreads();
    const uint64_t lb = sm.tau;
    for (int e = tid; e < total; e += kThreads) {
        const uint64_t kv = sm.all[e];
        if (kv >= lb && kv != 0ull) sm.cand[atomicAdd(&sm.n_cand, 1)] = kv;
    }
    __syncthreads();
    const int ncm = sm.n_cand;
    for (int c = tid; c < ncm; c += kThreads) {
        const uint64_t kc = sm.cand[c];
        int rank = 0;
#pragma unroll 8
        for (int o = 0; o < ncm; ++o) rank += sm.cand[o] > kc;
        if (rank < k) sm.top[rank] = kc;
    }
    __syncthreads();
    if (tid < 32) {
        // weights, top-p prefix and draw in float32 (IEEE division and expf, in candidate order):
        // lane j holds candidate j
        const int n = min(ncm, k);
        const float l0 = ord_to_float((uint32_t)(sm.top[0] >> 32));
        const float w = lane < n
            ? expf(__fdiv_rn(__fsub_rn(ord_to_float((uint32_t)(sm.top[lane] >> 32)), l0), temperature)) : 0.0f;
        sm.w[lane] = w;
        __syncwarp();
        // running sums in candidate order: lane j adds w_0, w_1, .. w_j one by one from shared memory (the
        // same float32 sums as one sequential pass), all lanes at once
        float run = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
            if (j <= lane && j < n) run = __fadd_rn(run, sm.w[j]);
        if (lane < n) sm.run[lane] = run;
        __syncwarp();
        const float total_w = sm.run[n - 1];
        // shortest prefix whose share reaches top_p: the first j with run_j / total >= top_p
        const unsigned reach = __ballot_sync(0xffffffffu, lane < n && __fdiv_rn(sm.run[lane], total_w) >= top_p);
        const int keep = reach ? __ffs(reach) : n;
        const float z = sm.run[keep - 1];
        const float thr = __fmul_rn(__ldcg(u + row), z);
        // the draw: the first kept j whose running sum exceeds u * z (zero weights never do first)
        const unsigned over = __ballot_sync(0xffffffffu, lane < keep && sm.run[lane] > thr && w > 0.0f);
        const unsigned pos_w = __ballot_sync(0xffffffffu, lane < keep && w > 0.0f);
        const int pick = over ? __ffs(over) - 1 : (pos_w ? 31 - __clz(pos_w) : 0);
        for (int j = lane; j < k; j += 32) {
            ids[(size_t)row * k + j] = j < keep ? key_index(sm.top[j]) : -1;
            probs[(size_t)row * k + j] = j < keep ? __fdiv_rn(sm.w[j], z) : 0.0f;
        }
        if (lane == 0) {
            counts[row] = keep;
            tokens[row] = key_index(sm.top[pick]);
        }
    }
}

// ----------------------------------------------------------------------------- chain acceptance
constexpr int kMaxChainRows = 64;

struct AcceptSmem {
    int32_t p_ids[kMaxChainRows][kMaxK];
    float p_pr[kMaxChainRows][kMaxK];
    int32_t q_ids[kMaxChainRows][kMaxK];
    float q_pr[kMaxChainRows][kMaxK];
    int32_t p_cnt[kMaxChainRows], q_cnt[kMaxChainRows], drafts[kMaxChainRows];
    float u_acc[kMaxChainRows];
};

// Probability of token t in a sparse distribution (0 if absent), found by one warp.
__device__ __forceinline__ float warp_lookup(const int32_t* ids, const float* pr, int cnt, int t, int lane) {
    const bool hit = lane < cnt && ids[lane] == t;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    return m ? pr[__ffs(m) - 1] : 0.0f;
}

__global__ void __launch_bounds__(kThreads) accept_chain_kernel(
    const int32_t* __restrict__ p_ids, const float* __restrict__ p_probs, const int32_t* __restrict__ p_counts,
    const int32_t* __restrict__ q_ids, const float* __restrict__ q_probs, const int32_t* __restrict__ q_counts,
    int ks, const int32_t* __restrict__ drafts, const int32_t* __restrict__ target_tokens, int n_drafts,
    const float* __restrict__ u_accept, const float* __restrict__ u_replace, const int32_t* __restrict__ pos,
    int32_t* __restrict__ n_accepted, int32_t* __restrict__ out_tokens, int32_t* __restrict__ next_pos) {
    __shared__ AcceptSmem sm;
    const int tid = threadIdx.x, lane = tid & 31;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    const int rows = n_drafts + 1;
    const int kk = min(ks, kMaxK);
    // stage every input once, in parallel
    for (int e = tid; e < rows * kk; e += kThreads) {
        const int r = e / kk, j = e - r * kk;
        sm.p_ids[r][j] = __ldcg(p_ids + (size_t)r * ks + j);
        sm.p_pr[r][j] = __ldcg(p_probs + (size_t)r * ks + j);
        sm.q_ids[r][j] = r > 0 ? __ldcg(q_ids + (size_t)r * ks + j) : -1;
        sm.q_pr[r][j] = r > 0 ? __ldcg(q_probs + (size_t)r * ks + j) : 0.0f;
    }
    for (int r = tid; r < rows; r += kThreads) {
        sm.p_cnt[r] = min(__ldcg(p_counts + r), kk);
        sm.q_cnt[r] = r > 0 ? min(__ldcg(q_counts + r), kk) : 0;
        sm.drafts[r] = __ldcg(drafts + r);
        sm.u_acc[r] = __ldcg(u_accept + r);
    }
    __syncthreads();
    if (tid >= 32) return;
    int a = 0, last = -1;
    for (int i = 1; i <= n_drafts; ++i) {
        const int d = sm.drafts[i];
        const float pd = warp_lookup(sm.p_ids[i - 1], sm.p_pr[i - 1], sm.p_cnt[i - 1], d, lane);
        const float qd = warp_lookup(sm.q_ids[i], sm.q_pr[i], sm.q_cnt[i], d, lane);
        // u < min(1, p/q) exactly: the sign of the fused u * q - p is the sign of the exact value
        if (fmaf(sm.u_acc[i], qd, -pd) < 0.0f) {
            ++a;
            continue;
        }
        // replacement from max(0, p_{i-1} - q_i) over p_{i-1}'s candidates (lane j: candidate j)
        const int cnt = sm.p_cnt[i - 1];
        const int tj = lane < cnt ? sm.p_ids[i - 1][lane] : -1;
        float qj = 0.0f;
        for (int c = 0; c < sm.q_cnt[i]; ++c)
            if (sm.q_ids[i][c] == tj) {
                qj = sm.q_pr[i][c];
                break;
            }
        const float r = lane < cnt ? fmaxf(0.0f, __fsub_rn(sm.p_pr[i - 1][lane], qj)) : 0.0f;
        const bool positive = __any_sync(0xffffffffu, r > 0.0f);
        const float rw = positive ? r : (lane < cnt ? sm.p_pr[i - 1][lane] : 0.0f);   // p <= q: draw from p
        // running sums in candidate order, float32, in lane 0
        float rr[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) rr[j] = __shfl_sync(0xffffffffu, rw, j);
        if (lane == 0) {
            float tot = 0.0f;
            for (int j = 0; j < cnt; ++j) tot = __fadd_rn(tot, rr[j]);
            const float thr = __fmul_rn(__ldcg(u_replace), tot);
            float run = 0.0f;
            int pick = -1;
            for (int j = 0; j < cnt; ++j) {
                if (!(rr[j] > 0.0f)) continue;
                run = __fadd_rn(run, rr[j]);
                pick = j;
                if (run > thr) break;
            }
            last = pick >= 0 ? sm.p_ids[i - 1][pick] : sm.p_ids[i - 1][0];
        }
        break;
    }
    if (lane == 0) {
        if (a == n_drafts) last = __ldcg(target_tokens + n_drafts);
        for (int j = 0; j <= n_drafts; ++j) out_tokens[j] = j < a ? sm.drafts[j + 1] : (j == a ? last : -1);
        *n_accepted = a;
        if (next_pos) *next_pos = __ldcg(pos) + a + 1;
    }
}

// ----------------------------------------------------------------------------- tree acceptance + settlement
constexpr int kSettleWarps = VA_MAX_TREE_NODES;   // one warp per path depth

__global__ void __launch_bounds__(32 * kSettleWarps) tree_accept_settle_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int slots, const int32_t* __restrict__ tree, int n_nodes,
    const int32_t* __restrict__ node_tokens, const int32_t* __restrict__ target_tokens, int32_t* __restrict__ path_out,
    int32_t* __restrict__ emitted_out, int32_t* __restrict__ n_accepted, int32_t* __restrict__ next_pos,
    int32_t* dev_status) {
    __shared__ int s_mask[VA_MAX_TREE_NODES], s_tok[VA_MAX_TREE_NODES], s_tgt[VA_MAX_TREE_NODES];
    __shared__ int s_parent[VA_MAX_TREE_NODES], s_path[VA_MAX_TREE_NODES];
    __shared__ int s_len, s_base, s_bad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    if (tid < n_nodes) {
        s_mask[tid] = __ldcg(tree + 1 + tid);
        s_tok[tid] = __ldcg(node_tokens + tid);
        s_tgt[tid] = __ldcg(target_tokens + tid);
    }
    if (tid == 0) s_base = __ldcg(tree);
    __syncthreads();
    if (tid == 0) {
        int bad = 0;
        for (int c = 0; c < n_nodes; ++c) {
            const unsigned m = (unsigned)s_mask[c];
            const unsigned anc = m & ~(1u << c);
            if (!((m >> c) & 1u) || (m >> n_nodes) != 0u) bad = 1;
            const int par = anc ? 31 - __clz(anc) : -1;   // the deepest ancestor
            s_parent[c] = par;
            if (c == 0 ? (par != -1) : (par < 0 || (unsigned)s_mask[par] != anc)) bad = 1;
        }
        int status = bad ? VA_DEV_BAD_PATH : 0;
        if (s_base < 0) status |= VA_DEV_NEGATIVE_POS;
        s_bad = status;
        int len = 1;
        s_path[0] = 0;
        int v = 0;
        if (!status) {
            for (;;) {
                const int t = s_tgt[v];
                int nxt = -1;
                for (int c = v + 1; c < n_nodes; ++c)
                    if (s_parent[c] == v && s_tok[c] == t) {
                        nxt = c;
                        break;
                    }
                emitted_out[len - 1] = t;
                if (nxt < 0) break;
                s_path[len++] = nxt;
                v = nxt;
            }
        }
        s_len = status ? 0 : len;
        for (int j = 0; j < n_nodes; ++j) {
            path_out[j] = j < s_len ? s_path[j] : -1;
            if (j >= s_len) emitted_out[j] = -1;
        }
        *n_accepted = status ? 0 : len - 1;
        if (next_pos) *next_pos = status ? s_base : s_base + len;
        if (status && dev_status) atomicOr(dev_status, status);
    }
    __syncthreads();
    if (!k_cache || s_bad) return;
    // settlement: warp d moves the path node at depth d; every row is read before any is written
    constexpr int kChunks = kD * 2 / 16;   // 16-byte chunks per row
    const int len = s_len;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    long long dst = 0;
    bool move = false;
    if (warp < len) {
        const int node = s_path[warp];
        move = node != warp;
        const long long src = ((long long)s_base + node) % slots;
        dst = ((long long)s_base + warp) % slots;
        const int c = lane & (kChunks - 1);
        if (move) val = lane < kChunks ? __ldcg(k_cache + src * kChunks + c) : __ldcg(v_cache + src * kChunks + c);
    }
    __syncthreads();
    if (move) {
        const int c = lane & (kChunks - 1);
        if (lane < kChunks)
            k_cache[dst * kChunks + c] = val;
        else
            v_cache[dst * kChunks + c] = val;
    }
}

}  // namespace smp
}  // namespace va

// ------------------------------------------------------------------------------- C ABI
namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
va_status launched(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? VA_OK : VA_CUDA_ERROR;
}
int n_tiles_of(int vocab) { return (vocab + VA_SAMPLE_TILE - 1) / VA_SAMPLE_TILE; }
}  // namespace

extern "C" {

size_t va_sample_workspace_bytes(int n_rows, int vocab, int top_k) {
    if (n_rows < 1 || n_rows > VA_SAMPLE_MAX_ROWS || top_k < 1 || top_k > VA_SAMPLE_MAX_K || vocab < top_k ||
        vocab > VA_SAMPLE_MAX_VOCAB)
        return 0;
    // the arrival counters first, at a place that does not depend on the shape (room for the largest
    // row count), so that one workspace serves calls of different shapes; then the tile keys
    const size_t keys = sizeof(uint64_t) * (size_t)n_rows * n_tiles_of(vocab) * top_k;
    return VA_SAMPLE_COUNTER_BYTES + keys;
}

va_status va_sample_topk_topp(const float* logits, int n_rows, int vocab, int top_k, float top_p, float temperature,
                              const float* u, int32_t* ids, float* probs, int32_t* counts, int32_t* tokens,
                              void* workspace, size_t workspace_bytes, va_stream stream) {
    const size_t need = va_sample_workspace_bytes(n_rows, vocab, top_k);
    if (need == 0 || vocab % 4 != 0) return VA_INVALID_ARG;
    if (!logits || !u || !ids || !probs || !counts || !tokens || !workspace) return VA_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(workspace) || workspace_bytes < need) return VA_INVALID_ARG;
    if (!(top_p > 0.0f && top_p <= 1.0f) || !(temperature > 0.0f) || temperature == INFINITY) return VA_INVALID_ARG;
    const int n_tiles = n_tiles_of(vocab);
    unsigned* arrivals = static_cast<unsigned*>(workspace);
    uint64_t* ws = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(workspace) + VA_SAMPLE_COUNTER_BYTES);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    va::pdl_config(&cfg, attr, dim3(n_tiles, n_rows), dim3(va::smp::kThreads), 0, (cudaStream_t)stream);
    return launched(cudaLaunchKernelEx(&cfg, va::smp::topk_sample_kernel, logits, vocab, top_k, top_p, temperature, u,
                                       ids, probs, counts, tokens, ws, arrivals));
}

va_status va_accept_chain(const int32_t* p_ids, const float* p_probs, const int32_t* p_counts, const int32_t* q_ids,
                          const float* q_probs, const int32_t* q_counts, int k_stride, const int32_t* drafts,
                          const int32_t* target_tokens, int n_drafts, const float* u_accept, const float* u_replace,
                          const int32_t* pos, int32_t* n_accepted, int32_t* out_tokens, int32_t* next_pos,
                          va_stream stream) {
    if (!p_ids || !p_probs || !p_counts || !drafts || !target_tokens || !u_accept || !u_replace || !pos ||
        !n_accepted || !out_tokens)
        return VA_INVALID_ARG;
    if (n_drafts < 0 || n_drafts >= va::smp::kMaxChainRows || k_stride < 1 || k_stride > VA_SAMPLE_MAX_K)
        return VA_INVALID_ARG;
    if (n_drafts > 0 && (!q_ids || !q_probs || !q_counts)) return VA_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    va::pdl_config(&cfg, attr, dim3(1), dim3(va::smp::kThreads), 0, (cudaStream_t)stream);
    return launched(cudaLaunchKernelEx(&cfg, va::smp::accept_chain_kernel, p_ids, p_probs, p_counts, q_ids, q_probs,
                                       q_counts, k_stride, drafts, target_tokens, n_drafts, u_accept, u_replace, pos,
                                       n_accepted, out_tokens, next_pos));
}

va_status va_tree_accept_settle(va_bf16* k_cache, va_bf16* v_cache, int slots, const int32_t* tree, int n_nodes,
                                const int32_t* node_tokens, const int32_t* target_tokens, int32_t* path,
                                int32_t* emitted, int32_t* n_accepted, int32_t* next_pos, int32_t* dev_status,
                                va_stream stream) {
    if (!tree || !node_tokens || !target_tokens || !path || !emitted || !n_accepted) return VA_INVALID_ARG;
    if (n_nodes < 1 || n_nodes > VA_MAX_TREE_NODES) return VA_INVALID_ARG;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return VA_INVALID_ARG;
    if (k_cache && (slots < 1 || !aligned16(k_cache) || !aligned16(v_cache))) return VA_INVALID_ARG;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    va::pdl_config(&cfg, attr, dim3(1), dim3(32 * va::smp::kSettleWarps), 0, (cudaStream_t)stream);
    return launched(cudaLaunchKernelEx(&cfg, va::smp::tree_accept_settle_kernel, reinterpret_cast<uint4*>(k_cache),
                                       reinterpret_cast<uint4*>(v_cache), slots, tree, n_nodes, node_tokens,
                                       target_tokens, path, emitted, n_accepted, next_pos, dev_status));
}

}  // extern "C"
