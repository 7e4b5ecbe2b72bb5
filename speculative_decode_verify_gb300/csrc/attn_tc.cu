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
//   * Two TMA warps stream 64-position boxes of K and V (128-byte swizzle) into 3-deep K and V
//     rings; K and V complete separate barriers, so QK starts as soon as K has landed.  Q and the first
//     stages are requested before the CTA's own set-up, and every load also asks L2 for the tile
//     kPrefetch tiles further on, so the rings refill from L2 rather than from DRAM.  P^T of a tile is written over that tile's K
//     once QK has consumed it, so the P buffers cost no extra shared memory and are double-buffered.
//   * One warp each issues the K loads, the V loads and the MMAs (one thread per role, so that a role
//     waiting on a barrier never holds up another); eight softmax warps, two per TMEM lane quadrant (one
//     per half of the 48 matrix rows): thread L holds key L of the tile for S^T and output column d = L
//     for O^T.
//   * Softmax keeps one reference per matrix row, shared by the CTA: initially the scaled score of the
//     split's first key.  Scores may exceed it by up to 2^8 before it is raised to the exact running
//     maximum (a CTA-wide vote); raising it rescales the TMEM accumulator and the running sums.  The
//     log-sum-exp stays exact: lse = ref + log2(sum) in base-2 units.
//   * P is split into bf16 hi + lo parts (two MMAs into the same accumulator), so the probabilities
//     enter the product with ~2^-17 relative error instead of bf16's 2^-9.
//   * K/V rows outside the split's owned positions (the unaligned ends of the extent: cache capacity
//     beyond the valid history, or ring slots outside the window) are zeroed in shared memory before
//     PV, so that garbage or NaN there cannot reach the accumulator through a zero probability.
//   * Every wait is bounded (VA_DEV_TIMEOUT); a timed-out CTA drains its own copies and MMAs, frees its
//     TMEM and returns.
//   * Draft trees ("Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees"): the
//     same kernel with the node region masked by each node's ancestor bitmask instead of the causal
//     tail.  Up to 16 nodes run as two groups of 8 rows (grid.y); the two CTAs of a split read the
//     same tiles at about the same time, so the second read is served by L2.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {
namespace tc {

#ifndef VA_NK
#define VA_NK 4
#endif
#ifndef VA_NV
#define VA_NV 2
#endif
// Start-up shaping: every CTA asks for its first tiles at the same moment and the DRAM serves all of
// them interleaved, so tile 0 lands no earlier than the rest and no stage frees up for several us.
// Requesting tile j of the first ring fill j * VA_STAGGER_NS after tile 0 lets tile 0 land first
// (0: no stagger).  Measured on GB300 per 192K verify call with the L2 pre-warm and the one-barrier start:
// 1,600 ns +0.90 us against 1,200 ns; 800 ns -0.23 us, 600 ns -0.27 us, 400 ns -0.32 us (-0.64 us per
// launch back to back), 200 ns -0.05 us against 400 ns; 0 +0.52 us against 400 ns.  (Before the pre-warm
// 1,200 ns was best.)
// Tiles pulled into L2 ahead of the rings by the softmax warps with plain loads (0: none).
#ifndef VA_L2AHEAD
#define VA_L2AHEAD 0
#endif
#ifndef VA_HINT_KV
#define VA_HINT_KV 1
#endif
#ifndef VA_HINT_POS
#define VA_HINT_POS 1
#endif
#ifndef VA_HINT_Q
#define VA_HINT_Q 1
#endif
#ifndef VA_STAGGER_NS
#define VA_STAGGER_NS 200
#endif

#ifndef VA_POLL_EVERY
#define VA_POLL_EVERY 64
#endif
// VA_POLL_EVERY: the MMA issuer's poll loop reads the timer and the abort flag (its give-up checks) once
// every VA_POLL_EVERY rounds that find nothing ready, which shortens a round (64 against 1 per 192K verify
// call: -0.10 and -0.11 us in two A/Bs, +0.01 us in a third).

// Tiles of a chain call's split pulled into L2 before the launch dependency resolves (0: none), from the
// plan of positions read at that time (a hint only: the kernel before may still be writing them; an L2
// prefetch of the wrong tiles costs bandwidth, never a result).  It also warms the address translations of
// the split's first pages.  Measured on GB300 (192K verify call, five rotating caches): 25.3 -> 24.0 us per
// call and 21.8 -> 20.2 us per launch back to back with 2 tiles (1 tile 24.8, 3 tiles 24.2, 4 tiles 24.6).
#ifndef VA_PREWARM
#define VA_PREWARM 2
#endif
// Speculative start of chain calls: the thread that warms L2 also requests tile 0 of the plan given by the
// positions it read before the launch dependency resolved, as soon as it resolves, and only then reads the
// positions again; if they differ (the kernel before was still writing them), it waits for those copies
// and re-arms tile 0's barriers before any role uses them, and tile 0 is requested again with the rest.
// VA_SPEC_SKEW (test builds only) shifts the early positions by one tile so that every launch whose tile 0
// was requested early takes that path.
#ifndef VA_SPEC
#define VA_SPEC 0
#endif
#ifndef VA_SPEC_SKEW
#define VA_SPEC_SKEW 0
#endif
// Start: 0 two block barriers after the launch dependency (warp 0's plan, then the set-up); 1 one block
// barrier before it (barriers and TMEM), a named barrier on which warp 0 only arrives once its plan is
// published (it then requests q and the first K stages at once), the V producer requesting its own first
// stages, and the row set-up by the softmax warps behind their own barrier.  Measured on GB300 (per
// verify call, outputs bit-identical): 1K 9.30 -> 8.62 us, the 4,103-position window 9.61 -> 8.92 us,
// 192K 24.03 -> 23.83 us; the split launch alone back to back and the 16-node tree within 0.1 us.  (The row
// set-up by warp 0 behind a third named barrier: -0.64, -0.67 and -0.10 us.)
#ifndef VA_EARLY
#define VA_EARLY 1
#endif
static_assert(!(VA_EARLY && VA_SPEC), "the speculative start assumes the two-barrier start");
// The same for draft trees (from the tree descriptor): measured ±0 on the 16-node tree at 192K, so off.
#ifndef VA_PREWARM_TREE
#define VA_PREWARM_TREE 0
#endif
constexpr int kNK = VA_NK;                // K ring depth (tiles of 128 positions); P of tile j reuses K's stage
constexpr int kNV = VA_NV;                // V ring depth
#ifndef VA_PREFETCH
#define VA_PREFETCH 0
#endif
// Tiles requested into L2 ahead of the rings.  Off: the per-SM TMA engine that serves the rings also
// serves the prefetches, and measured on GB300 every prefetch distance (2, 4, 6) made the kernel slower.
constexpr int kPrefetch = VA_PREFETCH;
constexpr uint32_t kHalfBox = 8192;       // one TMA box: 64 positions x 64 columns x 2 B
constexpr uint32_t kDHalf = 16384;        // 128 positions x 64 columns: one column half of a stage
constexpr uint32_t kStage = 32768;        // K or V of one 128-position tile
constexpr uint32_t kQHalf = 6144;         // 48 rows x 64 columns
constexpr uint32_t kQBytes = 2 * kQHalf;
constexpr uint32_t kPBytes = 16384;       // P^T: 128 keys x 64 columns (48 used), 128-byte swizzle
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kNK * kStage;
constexpr uint32_t kOffQ = kOffV + kNV * kStage;
constexpr uint32_t kOffMisc = kOffQ + kQBytes;
// Once QK(j) has read K(j), its stage holds P^T of tile j: the hi part in the first 16 KB, the lo part
// in the second.  The stage returns to the K ring when PV(j) has read P.
constexpr uint32_t kPhiInStage = 0, kPloInStage = kPBytes;
constexpr int kSoftWarps = 8;            // two per SM sub-partition: (lane quadrant, column half)
constexpr int kSoftWarp0 = 3;                    // warp 0 K loads, warp 1 MMA + TMEM owner, warp 2 V loads
constexpr int kThreads = 32 * (kSoftWarp0 + kSoftWarps);
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kCols = kMaxM / 2;          // matrix rows (accumulator columns) per softmax thread
constexpr uint32_t kTmemCols = 256;
// S^T of two tiles (48 columns each), O^T = P_hi V (columns 128..175) and P_lo V (192..239): the PV
// product runs with N = 128 over [P_hi | P_lo], and columns 176..191 and 240..255 receive the products
// of the unused P columns (never read).
constexpr uint32_t kColS0 = 0, kColS1 = 64, kColO = 128, kColLo = 64;
constexpr float kThresh = 256.0f;         // a probability may reach 2^8 before the reference is raised
constexpr float kRefInit = -1.0e30f;      // reference maximum before any visible key
constexpr uint64_t kWaitNs = 2000000000ull;

struct Misc {
    uint64_t k_full[kNK], k_empty[kNK], v_full[kNV], v_empty[kNV];
    uint64_t q_full, s_full[2], s_free[2], p_full[2], pv_done, o_ready, drain;
    uint64_t app_done;               // verify_attn_step: this split's share of the append is written
    uint32_t tmem_base;
    int abort;
    unsigned long long t_first_v;    // VA_EARLY: globaltimer when the V producer requested tile 0
    int vote[2][kSoftWarps];
    unsigned long long t_first;      // globaltimer when tile 0 was requested
    float red[4][kMaxM];
    float ref[kMaxM];
    float alpha[kMaxM];
    float inv_l[kMaxM];
    long long row_lo[kMaxRows], row_hi[kMaxRows];
    long long tree_base;             // tree calls: slot of node 0; chain calls: no node region (LLONG_MAX)
    Plan plan;                       // this split's extent and tiles (derived by warp 0)
    unsigned row_anc[kMaxRows];      // ancestor-or-self mask of each row of this CTA's group
    int pos[kMaxRows];
    int hint[kMaxRows];              // VA_SPEC: the positions as read before the launch dependency resolved
    int spec_tile[3];                // VA_SPEC: tile 0 of the plan they give (halves, first slot, second slot)
    int spec;                        // VA_SPEC: 2 when tile 0 was requested early from valid positions
    int anc[kMaxNodes];              // tree calls: every node's mask              // tree calls: every node's mask
    int base;
};
constexpr uint32_t kSmemBytes = kOffMisc + (uint32_t)sizeof(Misc) + 1024;
static_assert(kOffQ % 1024 == 0 && kStage % 1024 == 0 && 2 * kPBytes <= kStage, "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

// L2 prefetch of the K and V boxes of the first n tiles of plan Q (the loads' own boxes, see load_tile).
__device__ __forceinline__ void prewarm_tiles(const Plan& Q, int n, int slots, const CUtensorMap* k64,
                                              const CUtensorMap* k128, const CUtensorMap* v64, const CUtensorMap* v128) {
    const long long n64 = Q.t1 - Q.t0;
    const bool odd = (n64 & 1) != 0;
    const int nt = (int)((n64 + 1) >> 1);
    const unsigned slot_t0 = nt > 0 ? (unsigned)((Q.t0 * kTile) % slots) : 0u;   // then 32-bit offsets
    auto wrap_slot = [&](unsigned s) {
        while (s >= (unsigned)slots) s -= (unsigned)slots;
        return (int)s;
    };
    for (int j = 0; j < n && j < nt; ++j) {
        const unsigned dt = odd ? (j > 0 ? 2u * j - 1u : 0u) : 2u * j;
        const int halves = (odd && j == 0) ? 1 : 2;
        const int s0 = wrap_slot(slot_t0 + dt * kTile), s1 = wrap_slot(slot_t0 + (dt + 1u) * kTile);
        if (halves == 2 && s1 == s0 + kTile) {
            for (int h = 0; h < 2; ++h) {
                ptx::tma_prefetch_l2_2d(k128, h * 64, s0);
                ptx::tma_prefetch_l2_2d(v128, h * 64, s0);
            }
        } else {
            for (int hh = 0; hh < halves; ++hh)
                for (int h = 0; h < 2; ++h) {
                    ptx::tma_prefetch_l2_2d(k64, h * 64, hh ? s1 : s0);
                    ptx::tma_prefetch_l2_2d(v64, h * 64, hh ? s1 : s0);
                }
        }
    }
}

// The boxes of one K or V tile (those of load_tile): `halves` 64-row halves from slots s0 and s1.
__device__ __forceinline__ void issue_tile(const CUtensorMap* m64, const CUtensorMap* m128, uint32_t stage,
                                           uint32_t full, int halves, int s0, int s1) {
    const uint64_t pol = ptx::policy_evict_first();
    ptx::mbar_arrive_expect_tx(full, (uint32_t)halves * 2u * kHalfBox);
    if (halves == 2 && s1 == s0 + kTile) {
        for (int h = 0; h < 2; ++h) ptx::tma_load_2d_hint(stage + h * kDHalf, m128, h * 64, s0, full, pol);
    } else {
        for (int hh = 0; hh < halves; ++hh)
            for (int h = 0; h < 2; ++h)
                ptx::tma_load_2d_hint(stage + h * kDHalf + hh * kHalfBox, m64, h * 64, hh ? s1 : s0, full, pol);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

// Column base of the three columns a lane holds after warp_reduce_scatter24.
__device__ __forceinline__ int scatter_col_base(int lane) {
    return ((lane >> 4) & 1) * 12 + ((lane >> 3) & 1) * 6 + ((lane >> 2) & 1) * 3;
}

// Reduce 24 per-thread columns over the warp; afterwards the lane holds the warp totals of columns
// [scatter_col_base(lane), +3) in v[0..2] (the four lanes 4i..4i+3 hold the same three).
template <bool kMax>
__device__ __forceinline__ void warp_reduce_scatter24(float (&v)[kCols], int lane) {
#define VA_STAGE(W, BIT)                                                   \
    _Pragma("unroll") for (int i = 0; i < (W); ++i) {                      \
        const bool up = (lane & (BIT)) != 0;                               \
        const float send = up ? v[i] : v[i + (W)];                         \
        const float keep = up ? v[i + (W)] : v[i];                         \
        const float got = __shfl_xor_sync(0xffffffffu, send, (BIT));       \
        v[i] = kMax ? fmaxf(keep, got) : keep + got;                       \
    }
    VA_STAGE(12, 16)
    VA_STAGE(6, 8)
    VA_STAGE(3, 4)
#undef VA_STAGE
#pragma unroll
    for (int b = 2; b >= 1; b >>= 1)
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const float got = __shfl_xor_sync(0xffffffffu, v[i], b);
            v[i] = kMax ? fmaxf(v[i], got) : v[i] + got;
        }
}

#ifdef VA_TRACE
// Timeline probe of the debug build: per CTA, 256 globaltimer stamps (ns).  [0] start, [1] set-up
// done, [2] end, [3] tile count; tile j (j < 31) at 8 + 8 j: K requested, V requested, K seen by the
// MMA thread, V seen by the MMA thread, S seen by softmax, P published, P seen by the MMA thread.
__device__ unsigned long long* g_trace = nullptr;
#define VA_TRACE_AT(slot) \
    do { if (g_trace && (slot) < 256) g_trace[(size_t)blockIdx.x * 256 + (slot)] = ptx::globaltimer_ns(); } while (0)
#define VA_TRACE_TILE(j, k) do { if ((j) < 31) VA_TRACE_AT(8 + 8 * (j) + (k)); } while (0)
#else
#define VA_TRACE_AT(slot) do { } while (0)
#define VA_TRACE_TILE(j, k) do { } while (0)
#endif

#ifdef VA_DEBUG_VISIT
// Visit map of the debug build: [n_rows][slots] counts, one per (live row, key) let into the softmax,
// for an exact comparison with the visible-slot sets of the positions.
__device__ unsigned* g_visit = nullptr;
#endif

// kAppend: the verify_attn_step instantiation, which writes the live rows itself (a.k_new / a.v_new);
// the instantiation without it carries none of that code.
// kTree (with VA_TREE_TEMPLATE): the instantiation for tree calls (a.tree set); the chain instantiations
// carry none of the tree code, nor the tree instantiation the chain plan.
template <bool kAppend, bool kTree>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
               const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmk2,
               const __grid_constant__ CUtensorMap tmv2) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    Misc& ms = *reinterpret_cast<Misc*>(base + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x;
    const int group = blockIdx.y;     // rows [8 group, 8 group + 8) of the call
    const bool is_tree = VA_TREE_TEMPLATE ? kTree : a.tree != nullptr;
    const int M = min(kMaxM, a.n_rows * kH - kMaxM * group);             // matrix rows of this group
    const int n_live_g = max(0, min(kMaxRows, a.n_live - kMaxRows * group));   // live rows of this group
    const int ML = n_live_g * kH;     // live matrix rows of this group
    if (tid == 0) VA_TRACE_AT(0);
    auto bar = [](const uint64_t& b) { return ptx::smem_u32(&b); };

    // ---------------------------------------------------------------- set-up without global memory
    if (tid == 0) {
        ptx::mbar_init(bar(ms.q_full), 1);
        for (int i = 0; i < kNK; ++i) {
            ptx::mbar_init(bar(ms.k_full[i]), 1);
            ptx::mbar_init(bar(ms.k_empty[i]), 1);
        }
        for (int i = 0; i < kNV; ++i) {
            ptx::mbar_init(bar(ms.v_full[i]), 1);
            ptx::mbar_init(bar(ms.v_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(ms.s_full[i]), 1);
            ptx::mbar_init(bar(ms.s_free[i]), kSoftWarps);
        }
        ptx::mbar_init(bar(ms.p_full[0]), kSoftWarps);
        ptx::mbar_init(bar(ms.p_full[1]), kSoftWarps);
        ptx::mbar_init(bar(ms.pv_done), 1);
        ptx::mbar_init(bar(ms.o_ready), 1);
        ptx::mbar_init(bar(ms.drain), 1);
        if (kAppend) ptx::mbar_init(bar(ms.app_done), 1);
        ms.abort = 0;
        if (VA_SPEC) ms.spec = 0;
        ptx::mbar_init_fence();
        VA_TRACE_AT(240);
    }
    if (VA_SPEC && warp == 0) ptx::named_bar_arrive(2, 64);   // the barriers, to the early requester's warp
    if (tid == 32) {
        ptx::tma_prefetch_desc(&tmq);
        ptx::tma_prefetch_desc(&tmk);
        ptx::tma_prefetch_desc(&tmv);
        ptx::tma_prefetch_desc(&tmk2);
        ptx::tma_prefetch_desc(&tmv2);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&ms.tmem_base), kTmemCols);
    if (tid == 32) VA_TRACE_AT(241);
#if VA_EARLY
    ptx::tc_fence_before();
    __syncthreads();   // barriers initialised, TMEM allocated: no block barrier is needed after the dependency
    ptx::tc_fence_after();
#endif

    // Programmatic dependent launch: every global access of this kernel comes after griddep_wait (the
    // prefetches above only pick lines for L2).
    ptx::griddep_launch_dependents();
#if VA_SPEC
    bool sp_planned = false;   // thread kThreads - 1: ms.hint and ms.spec_tile hold an early tile 0
#endif
#if VA_PREWARM || VA_SPEC
    // a thread off the start's critical path warms L2 (and the address translations) for this split's first
    // tiles while the kernel before may still run
    if (tid == kThreads - 1 && n_live_g > 0 && (!is_tree || VA_PREWARM_TREE)) {
        Plan Q;
        if (!is_tree) {
            int sp[kMaxRows];
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r)
                sp[r] = (r < a.n_live) ? ptx::ld_relaxed_int(a.pos + r) - (VA_SPEC_SKEW ? kTile : 0) : 0;
            Q = make_plan(sp, a.n_live, a.window, a.slots, a.n_splits, split);
#if VA_SPEC
            const long long n64 = Q.t1 - Q.t0;
            const int h0 = (n64 & 1) ? 1 : 2;
            const bool new0 = kAppend && (long long)sp[0] < (Q.t0 + h0) * kTile && Q.hi > Q.t0 * kTile;
            if (!Q.status && n64 > 0 && !new0) {   // (a tile 0 that holds new rows waits for the append)
#pragma unroll
                for (int r = 0; r < kMaxRows; ++r) ms.hint[r] = sp[r];
                ms.spec_tile[0] = h0;
                ms.spec_tile[1] = (int)((Q.t0 * kTile) % a.slots);
                ms.spec_tile[2] = (int)(((Q.t0 + 1) * kTile) % a.slots);
                sp_planned = true;
            }
#endif
        } else {
            int anc[kMaxNodes];
#pragma unroll
            for (int i = 0; i < kMaxNodes; ++i) anc[i] = (i < a.n_live) ? ptx::ld_relaxed_int(a.tree + 1 + i) : 0;
            Q = make_tree_plan(ptx::ld_relaxed_int(a.tree), anc, a.n_live, a.window, a.slots, a.n_splits, split);
        }
        if (VA_PREWARM && !Q.status) prewarm_tiles(Q, VA_PREWARM, a.slots, &tmk, &tmk2, &tmv, &tmv2);
    }
#endif
    ptx::griddep_wait();
    if (tid == 0) VA_TRACE_AT(242);
#if VA_SPEC
    if (warp == kThreads / 32 - 1) {
        ptx::named_bar_sync(2, 64);   // thread 0's barrier initialisation is visible from here on
        if (tid == kThreads - 1 && sp_planned) {
            ms.t_first = ptx::globaltimer_ns();
            VA_TRACE_TILE(0, 0);
            issue_tile(&tmk, &tmk2, base_s + kOffK, bar(ms.k_full[0]), ms.spec_tile[0], ms.spec_tile[1], ms.spec_tile[2]);
            VA_TRACE_TILE(0, 1);
            issue_tile(&tmv, &tmv2, base_s + kOffV, bar(ms.v_full[0]), ms.spec_tile[0], ms.spec_tile[1], ms.spec_tile[2]);
            int now[kMaxRows];
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) now[r] = (r < a.n_live) ? __ldcg(a.pos + r) : 0;
            bool same = true;
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) same &= r >= a.n_live || now[r] == ms.hint[r];
            if (same) {
                ms.spec = 2;
            } else if (ptx::mbar_wait(bar(ms.k_full[0]), 0, nullptr, kWaitNs) &&
                       ptx::mbar_wait(bar(ms.v_full[0]), 0, nullptr, kWaitNs)) {
                // a stale hint: its copies have landed; tile 0's barriers start over at phase 0
                ptx::mbar_inval(bar(ms.k_full[0]));
                ptx::mbar_init(bar(ms.k_full[0]), 1);
                ptx::mbar_inval(bar(ms.v_full[0]));
                ptx::mbar_init(bar(ms.v_full[0]), 1);
                ptx::mbar_init_fence();
            } else {   // never re-armed: nothing more is requested into it and every role gives up
                ms.spec = 2;
                ms.abort = 1;
                if (a.dev_status) atomicOr(a.dev_status, VA_DEV_TIMEOUT);
            }
        }
    }
#endif

    // the positions (or the tree): one request per CTA; warp 0 derives the plan and shares it through
    // shared memory (the other warps would only compete with it for issue slots)
    int row_pos[kMaxRows];
    Plan P;
    if (warp == 0) {
        if (!is_tree) {
            if (lane < a.n_live)
                ms.pos[lane] =
                    VA_HINT_POS ? ptx::ld_int_policy(a.pos + lane, ptx::policy_evict_last()) : __ldcg(a.pos + lane);
        } else if (lane <= a.n_live) {
            const int w = ptx::ld_int_policy(a.tree + lane, ptx::policy_evict_last());
            if (lane == 0) ms.base = w;
            else ms.anc[lane - 1] = w;
        }
        __syncwarp();
        if (!is_tree) {
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) row_pos[r] = (r < a.n_live) ? ms.pos[r] : 0;
            P = make_plan(row_pos, a.n_live, a.window, a.slots, a.n_splits, split);
        } else {
            int anc[kMaxNodes];
#pragma unroll
            for (int i = 0; i < kMaxNodes; ++i) anc[i] = (i < a.n_live) ? ms.anc[i] : 0;
            P = make_tree_plan(ms.base, anc, a.n_live, a.window, a.slots, a.n_splits, split);
        }
        if (lane == 0) ms.plan = P;
        if (P.status && split == 0 && group == 0 && lane == 0 && a.dev_status) atomicOr(a.dev_status, P.status);
    }
#if VA_EARLY
    if (warp == 0) ptx::named_bar_arrive(2, kThreads);   // the plan and positions are published
    else ptx::named_bar_sync(2, kThreads);
#else
    __syncthreads();
#endif
    if (warp != 0) P = ms.plan;
    if (!is_tree) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) row_pos[r] = (r < a.n_live) ? ms.pos[r] : 0;
    }
    if (tid == 0) VA_TRACE_AT(243);
    const int n64 = (P.status || n_live_g == 0) ? 0 : (int)(P.t1 - P.t0);
    const int ntiles = (n64 + 1) >> 1;
    const int M_all = a.n_rows * kH;
    float* part_o = a.part_o + ((long long)split * M_all + kMaxM * group) * kD;
    float* part_lse = a.part_lse + (long long)split * M_all + kMaxM * group;
    const long long own_lo = max(P.lo, P.t0 * kTile);
    const long long own_hi = min(P.hi, P.t1 * kTile);

    // Tile j covers one or two 64-position tiles from t = tile_t(j).  A split with an odd number of them
    // takes the single one first: at the start the softmax warps wait for data anyway, whereas a short
    // last tile would add a whole QK / softmax / PV round after the split's last byte has arrived.
    // The cache rows of tile j start at slot(t); the two halves are contiguous unless a ring wraps between
    // them.
    const bool odd = (n64 & 1) != 0;
    auto tile_t = [&](int j) { return P.t0 + (odd ? (j > 0 ? 2LL * j - 1 : 0LL) : 2LL * j); };
    auto tile_halves = [&](int j) { return (odd && j == 0) ? 1 : 2; };
    // Slot of the split's first 64-position tile: one 64-bit remainder per producer; a tile's slots are then
    // 32-bit offsets from it.  A tile lies less than 2 slots + 192 positions past it (the plan rejects
    // extents wider than the cache), so a few subtractions wrap it.  (Two 64-bit remainders per request,
    // on the path from a freed V stage to its refill, cost 0.26 us per 192K verify call.)
    unsigned slot_t0 = 0u;   // set by the threads that call tile_slots, before their first call
    auto set_slot_t0 = [&]() { slot_t0 = n64 > 0 ? (unsigned)((P.t0 * kTile) % a.slots) : 0u; };
    auto wrap_slot = [&](unsigned s) {
        while (s >= (unsigned)a.slots) s -= (unsigned)a.slots;
        return (int)s;
    };
    auto tile_slots = [&](int j, int& slot0, int& slot1, int& halves) {
        const long long t = tile_t(j);
        halves = tile_halves(j);
        const unsigned off = slot_t0 + (unsigned)(t - P.t0) * (unsigned)kTile;
        slot0 = wrap_slot(off);
        slot1 = wrap_slot(off + (unsigned)kTile);
    };
    // L2 prefetch of K or V of tile j (same boxes as the loads)
    auto prefetch_tile = [&](const CUtensorMap* m64, const CUtensorMap* m128, int j) {
        int s0, s1, halves;
        tile_slots(j, s0, s1, halves);
        if (halves == 2 && s1 == s0 + kTile) {
            for (int h = 0; h < 2; ++h) ptx::tma_prefetch_l2_2d(m128, h * 64, s0);
        } else {
            for (int hh = 0; hh < halves; ++hh)
                for (int h = 0; h < 2; ++h) ptx::tma_prefetch_l2_2d(m64, h * 64, hh ? s1 : s0);
        }
    };
    // K/V of tile j into its ring stage: per 64-column half one 128-row box (contiguous halves) or one
    // 64-row box per half.  A load also prefetches tile j + kPrefetch into L2.
    // K/V are read once: evict-first, so that they do not push the small per-call inputs out of L2
    auto load_tile = [&](const CUtensorMap* m64, const CUtensorMap* m128, uint32_t stage, uint64_t& full, int j) {
        int s0, s1, halves;
        tile_slots(j, s0, s1, halves);
        const uint64_t pol = ptx::policy_evict_first();
        ptx::mbar_arrive_expect_tx(bar(full), (uint32_t)halves * 2u * kHalfBox);
        if (halves == 2 && s1 == s0 + kTile) {
            for (int h = 0; h < 2; ++h) {
                if (VA_HINT_KV) ptx::tma_load_2d_hint(stage + h * kDHalf, m128, h * 64, s0, bar(full), pol);
                else ptx::tma_load_2d(stage + h * kDHalf, m128, h * 64, s0, bar(full));
            }
        } else {
            for (int hh = 0; hh < halves; ++hh)
                for (int h = 0; h < 2; ++h) {
                    if (VA_HINT_KV)
                        ptx::tma_load_2d_hint(stage + h * kDHalf + hh * kHalfBox, m64, h * 64, hh ? s1 : s0, bar(full), pol);
                    else
                        ptx::tma_load_2d(stage + h * kDHalf + hh * kHalfBox, m64, h * 64, hh ? s1 : s0, bar(full));
                }
        }
    };
    auto load_k = [&](int j) {
        VA_TRACE_TILE(j, 0);
        load_tile(&tmk, &tmk2, base_s + kOffK + (uint32_t)(j % kNK) * kStage, ms.k_full[j % kNK], j);
        if (kPrefetch > 0 && j >= kNK && j + kPrefetch < ntiles) prefetch_tile(&tmk, &tmk2, j + kPrefetch);
    };
    auto load_v = [&](int j) {
        VA_TRACE_TILE(j, 1);
        load_tile(&tmv, &tmv2, base_s + kOffV + (uint32_t)(j % kNV) * kStage, ms.v_full[j % kNV], j);
        if (kPrefetch > 0 && j >= kNV && j + kPrefetch < ntiles) prefetch_tile(&tmv, &tmv2, j + kPrefetch);
    };
    // verify_attn_step: a tile holding a live row's position is loaded only after the MMA warp, which
    // appends this split's live rows first, has written them (app_done).  Positions never decrease, so the
    // live rows are the positions [pos[0], hi).
    constexpr bool step = kAppend;
    auto tile_has_new = [&](int j) {
        if (!step) return false;
        const long long t = tile_t(j);
        return (long long)row_pos[0] < (t + tile_halves(j)) * kTile && P.hi > t * kTile;
    };
    // Initial fill: with VA_STAGGER_NS, only tile 0 is requested at once and the producers request
    // tile j of the first ring fill j * VA_STAGGER_NS after it.  (A tile 0 that waits for the append is
    // requested by the producers.)
    const bool defer0 = ntiles > 0 && tile_has_new(0);
    const int k_first = defer0 ? 0 : VA_STAGGER_NS ? min(1, ntiles) : min(kNK, ntiles);
    const int v_first = defer0 ? 0 : VA_STAGGER_NS ? min(1, ntiles) : min(kNV, ntiles);
    auto stagger = [&](int j) {
        if (VA_STAGGER_NS == 0) return;
        const unsigned long long due =
            (VA_EARLY && warp == 2 ? ms.t_first_v : ms.t_first) + (unsigned long long)j * VA_STAGGER_NS;
        for (int spin = 0; spin < 1000000 && ptx::globaltimer_ns() < due; ++spin) __nanosleep(64);
    };

    // row u of this group: the positions it sees inside this split, [lo, hi), and its mask of the node
    // region [tree_base, hi); the reference of matrix row u (padding rows never weigh anything).  Compact
    // code: it runs once per launch, from a cold instruction cache, on the softmax warps' way to their first
    // tile.
    auto row_setup = [&](int u) {
        if (u < kMaxRows) {
            long long lo = 0, hi = 0;
            unsigned m = 0xFFFFFFFFu;
            if (u < n_live_g) {
                long long p;   // the row's own position
                if (!is_tree) {
                    p = ms.pos[u];
                    hi = min(p + 1, own_hi);
                } else {
                    m = (unsigned)ms.anc[kMaxRows * group + u];
                    p = (long long)ms.base + tree_depth((int)m);
                    hi = min(P.hi, own_hi);
                }
                lo = max(a.window > 0 ? max(0LL, p - a.window + 1) : 0LL, own_lo);
            }
            if (hi < lo) hi = lo;
            ms.row_lo[u] = lo;
            ms.row_hi[u] = hi;
            ms.row_anc[u] = m;
            if (u == 0) ms.tree_base = is_tree ? (long long)ms.base : LLONG_MAX;
        }
        if (u < kMaxM) ms.ref[u] = u < ML ? kRefInit : INFINITY;
    };
    // ---------------------------------------------------------------- set-up with global memory
    if (ntiles > 0) {
        if (tid == 0) {
            // Q, then the first stages
            set_slot_t0();
            ptx::mbar_arrive_expect_tx(bar(ms.q_full), kQBytes);
            const uint64_t keep = ptx::policy_evict_last();   // every CTA reads the same q
            if (VA_HINT_Q) {
                ptx::tma_load_2d_hint(base_s + kOffQ, &tmq, 0, kMaxM * group, bar(ms.q_full), keep);
                ptx::tma_load_2d_hint(base_s + kOffQ + kQHalf, &tmq, 64, kMaxM * group, bar(ms.q_full), keep);
            } else {
                ptx::tma_load_2d(base_s + kOffQ, &tmq, 0, kMaxM * group, bar(ms.q_full));
                ptx::tma_load_2d(base_s + kOffQ + kQHalf, &tmq, 64, kMaxM * group, bar(ms.q_full));
            }
#if VA_SPEC
            const int j0 = ms.spec == 2 ? 1 : 0;   // tile 0 requested early
#else
            constexpr int j0 = 0;
#endif
            if (!j0) ms.t_first = ptx::globaltimer_ns();
            for (int j = j0; j < k_first; ++j) load_k(j);
            if (!VA_EARLY)
                for (int j = j0; j < v_first; ++j) load_v(j);
        }
#if !VA_EARLY
        row_setup(tid);
#endif
    }
#if !VA_EARLY
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
#endif
    const uint32_t tmem = ms.tmem_base;
    volatile int* abort_flag = &ms.abort;
    if (tid == 0) {
        VA_TRACE_AT(1);
#ifdef VA_TRACE
        if (g_trace) g_trace[(size_t)blockIdx.x * 256 + 3] = (unsigned long long)ntiles;
#endif
    }
    auto fail = [&]() {
        *abort_flag = 1;
        if (a.dev_status) atomicOr(a.dev_status, VA_DEV_TIMEOUT);
    };

    if (ntiles == 0) {
        // empty split (or unusable positions): o = 0, lse = -inf
        for (int i = tid; i < M * kD; i += kThreads) part_o[i] = 0.0f;
        for (int i = tid; i < M; i += kThreads) part_lse[i] = -INFINITY;
    } else if (warp == 0) {
        // ------------------------------------------------------------ K producer
        if (lane == 0) {
            if (kPrefetch > 0)
                for (int j = k_first; j < min(kNK + kPrefetch, ntiles); ++j) prefetch_tile(&tmk, &tmk2, j);
            int issued = k_first;
            for (int j = k_first; j < ntiles; ++j) {
                if (j < kNK) stagger(j);
                if ((tile_has_new(j) && !ptx::mbar_wait(bar(ms.app_done), 0, abort_flag, kWaitNs)) ||
                    !ptx::mbar_wait(bar(ms.k_empty[j % kNK]), ((j / kNK) & 1) ^ 1, abort_flag, kWaitNs)) {
                    fail();
                    break;
                }
                load_k(j);
                issued = j + 1;
            }
            for (int j = max(0, issued - kNK); j < issued; ++j)   // every issued copy lands before exit
                ptx::mbar_wait(bar(ms.k_full[j % kNK]), (j / kNK) & 1, nullptr, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ V producer
        if (lane == 0) {
            set_slot_t0();
            if (VA_EARLY) {   // the V producer requests its own first stages
                ms.t_first_v = ptx::globaltimer_ns();
                for (int j = 0; j < v_first; ++j) load_v(j);
            }
            if (kPrefetch > 0)
                for (int j = v_first; j < min(kNV + kPrefetch, ntiles); ++j) prefetch_tile(&tmv, &tmv2, j);
            int issued = v_first;
            for (int j = v_first; j < ntiles; ++j) {
                if (j < kNV) stagger(j);
                if ((tile_has_new(j) && !ptx::mbar_wait(bar(ms.app_done), 0, abort_flag, kWaitNs)) ||
                    !ptx::mbar_wait(bar(ms.v_empty[j % kNV]), ((j / kNV) & 1) ^ 1, abort_flag, kWaitNs)) {
                    fail();
                    break;
                }
                load_v(j);
                issued = j + 1;
            }
            for (int j = max(0, issued - kNV); j < issued; ++j)
                ptx::mbar_wait(bar(ms.v_full[j % kNV]), (j / kNV) & 1, nullptr, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (step) {
            // verify_attn_step: this split's share of the append (IQuestRT report, "Read only the KV tiles
            // needed by the current positions": the new rows are written before they are read).  The live
            // rows whose positions lie in this split's tiles go to slot pos mod slots; a row whose slot a
            // later row also writes is skipped, so the rows land as if written in row order.  Every other
            // split reads none of these rows (in a ring, a stale row of the same slot lies below every
            // window and is zeroed or masked).  Only a split that owns live rows waits for its stores
            // (the proxy fence) before its first product.
            const uint4* src = reinterpret_cast<const uint4*>(lane < 16 ? a.k_new : a.v_new) + (lane & 15);
            uint4* dst = reinterpret_cast<uint4*>(const_cast<uint16_t*>(lane < 16 ? a.k : a.v)) + (lane & 15);
            const long long tlo = P.t0 * kTile, thi = P.t1 * kTile;
            bool mine[kMaxRows];
            uint4 val[kMaxRows];
            bool any = false;
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                // the plan accepted the positions: they never decrease and span less than the slots, so
                // rows share a slot only when they share a position, and then they are adjacent
                mine[r] = r < a.n_live && row_pos[r] >= tlo && row_pos[r] < thi &&
                          !(r + 1 < kMaxRows && r + 1 < a.n_live && row_pos[r + 1] == row_pos[r]);
                if (mine[r]) val[r] = __ldcg(src + r * (kD / 8));
                any |= mine[r];
            }
            if (any) {   // (most splits own no live row and skip the stores and the fence)
#pragma unroll
                for (int r = 0; r < kMaxRows; ++r)
                    if (mine[r]) dst[(size_t)(row_pos[r] % a.slots) * (kD / 8)] = val[r];
                ptx::fence_proxy_async_global();   // the TMA loads of these rows come after
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.app_done));
        }
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(128, 48, 0, 0);   // A = K, B = Q: both K-major
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, 128, 1, 1);  // A = V^T, B = [P_hi | P_lo]^T: MN-major
            bool ok = ptx::mbar_wait(bar(ms.q_full), 0, abort_flag, kWaitNs);
            // Issue whichever product is ready: QK(qk) once K(qk) has landed and its S buffer is free, and
            // PV(pv) once V(pv) has landed and P(pv) is published.  PV never waits for a later K, so the
            // stages of tile pv return to the rings as soon as possible.  QK(j) is issued only after PV(j-2):
            // the commit after QK(j) then covers PV(j-2), which keeps every parity wait at most one phase
            // behind its barrier.
            int qk = 0, pv = 0;
            uint64_t idle_since = 0;
            unsigned idle_polls = 0;
            while (ok && pv < ntiles) {
                bool progressed = false;
                if (qk < ntiles && qk <= pv + 1 &&
                    ptx::mbar_test_wait(bar(ms.k_full[qk % kNK]), (qk / kNK) & 1) &&
                    ptx::mbar_test_wait(bar(ms.s_free[qk & 1]), ((qk >> 1) & 1) ^ 1)) {
                    const int ks = qk % kNK, sb = qk & 1;
                    VA_TRACE_TILE(qk, 2);
                    ptx::tc_fence_after();
                    const uint32_t d = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t h = (uint32_t)kk >> 2, off = (uint32_t)(kk & 3) * 32u;
                        ptx::mma_bf16(d, ptx::smem_desc(base_s + kOffK + ks * kStage + h * kDHalf + off, 0, 1024),
                                      ptx::smem_desc(base_s + kOffQ + h * kQHalf + off, 0, 1024), idesc_qk, kk > 0);
                    }
                    ptx::mma_commit(bar(ms.s_full[sb]));
                    ++qk;
                    progressed = true;
                }
                if (pv < qk && ptx::mbar_test_wait(bar(ms.v_full[pv % kNV]), (pv / kNV) & 1) &&
                    ptx::mbar_test_wait(bar(ms.p_full[pv & 1]), (pv >> 1) & 1)) {
                    const int i = pv, vs = i % kNV, ps = i % kNK;
                    VA_TRACE_TILE(i, 3);
                    VA_TRACE_TILE(i, 6);
                    ptx::tc_fence_after();
                    const int nk = tile_halves(i) == 2 ? 8 : 4;
                    for (int kk = 0; kk < nk; ++kk) {
                        // one MMA for both parts of P: B columns 0..63 are P_hi (48 used), 64..127 P_lo, one
                        // 128-byte swizzle atom apart (the leading byte offset), so V is read once
                        const uint64_t adesc = ptx::smem_desc(base_s + kOffV + vs * kStage + kk * 2048, kDHalf, 1024);
                        const uint32_t pbase = base_s + kOffK + ps * kStage + kk * 2048;
                        ptx::mma_bf16(tmem + kColO, adesc, ptx::smem_desc(pbase + kPhiInStage, kPloInStage - kPhiInStage, 1024),
                                      idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(bar(ms.pv_done));
                    ptx::mma_commit(bar(ms.v_empty[vs]));
                    ptx::mma_commit(bar(ms.k_empty[ps]));
                    if (i == ntiles - 1) ptx::mma_commit(bar(ms.o_ready));   // the accumulator is final
                    ++pv;
                    progressed = true;
                }
                if (progressed) {
                    idle_since = 0;
                    idle_polls = 0;
                } else if (VA_POLL_EVERY <= 1 || ++idle_polls % VA_POLL_EVERY == 0) {
                    // bounded: give up after kWaitNs without progress, or when another role aborted
                    const uint64_t now = ptx::globaltimer_ns();
                    if (idle_since == 0) idle_since = now;
                    if (*abort_flag || now - idle_since > kWaitNs) ok = false;
                }
            }
            if (!ok) fail();
            ptx::mma_commit(bar(ms.drain));   // all MMAs of this CTA done before TMEM is freed
            ptx::mbar_wait(bar(ms.drain), 0, nullptr, kWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / accumulator warps
        const int sw = warp - kSoftWarp0;     // 0..7
#if defined(VA_DEBUG_VISIT) || VA_L2AHEAD > 0
        set_slot_t0();
#endif
#if VA_EARLY
        row_setup(sw * 32 + lane);
        ptx::named_bar_sync(1, kSoftThreads);   // the rows' extents and references are published
#endif
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int ch = sw >> 2;               // column half: matrix rows [24 ch, 24 ch + 24)
        const int n0 = ch * kCols;
        const int L = q * 32 + lane;          // key of the tile (S^T) and output column d (O^T)
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        const float c = a.scale * 1.4426950408889634f;   // scores in log2 units
        long long all_lo = own_lo, all_hi = own_hi;
        for (int r = 0; r < n_live_g; ++r) {
            all_lo = max(all_lo, ms.row_lo[r]);
            all_hi = min(all_hi, ms.row_hi[r]);
        }
        const long long tree_base = ms.tree_base;
        all_hi = min(all_hi, tree_base);   // the node region of a tree is never interior
        float ref[kCols], l[kCols];
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
            ref[i] = ms.ref[n0 + i];
            l[i] = 0.0f;
        }
        // L2 warm-up of tile jt: softmax thread st touches one 256-byte row of K (st < 128) or V
        auto l2_touch_tile = [&](int jt) {
            if (jt >= ntiles) return;
            int s0, s1, halves;
            tile_slots(jt, s0, s1, halves);
            const int st = sw * 32 + lane, r = st & 127, hh = r >> 6;
            if (hh < halves) {
                const int row = (hh ? s1 : s0) + (r & 63);
                if (row < a.slots) ptx::touch_l2_256((st < 128 ? a.k : a.v) + (size_t)row * kD);
            }
        };
        if (VA_L2AHEAD > 0)
            for (int jt = 1; jt <= VA_L2AHEAD; ++jt) l2_touch_tile(jt);
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const long long t = tile_t(j);
            const int nkeys = tile_halves(j) == 2 ? 128 : 64;
            const long long kbase = t * kTile;
            const long long kp = kbase + L;
            const int sb = j & 1;
            if (VA_L2AHEAD > 0 && j > 0) l2_touch_tile(j + VA_L2AHEAD);
            if (!ptx::mbar_wait(bar(ms.s_full[sb]), (j >> 1) & 1, abort_flag, kWaitNs)) ok = false;
            if (sw == 0 && lane == 0) VA_TRACE_TILE(j, 4);
            ptx::tc_fence_after();
            float x[kCols];
            ptx::tmem_ld24_wait(tl + (sb ? kColS1 : kColS0) + n0, x);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.s_free[sb]));

            // visibility: interior tiles need only the half-tile check; padding rows have ref = +inf
            const bool interior = kbase >= all_lo && kbase + nkeys <= all_hi;
            bool vis[kCols];
            {   // this column half holds verify rows 4 ch .. 4 ch + 3
                bool rv[kMaxRows / 2];
                const long long dk = kp - tree_base;   // node index of key kp in a tree's node region
#pragma unroll
                for (int k = 0; k < kMaxRows / 2; ++k) {
                    const int r = (kMaxRows / 2) * ch + k;
                    const bool in_mask = dk < 0 || (dk < 32 && ((ms.row_anc[r] >> (int)dk) & 1u));
                    rv[k] = (L < nkeys) &&
                            (interior || ((r < n_live_g) && kp >= ms.row_lo[r] && kp < ms.row_hi[r] && in_mask));
                }
#pragma unroll
                for (int i = 0; i < kCols; ++i) vis[i] = rv[i / kH];
#ifdef VA_DEBUG_VISIT
                if (g_visit) {
                    int s0, s1, halves;
                    tile_slots(j, s0, s1, halves);
                    const int slot = ((L >> 6) ? s1 : s0) + (L & 63);
                    for (int k = 0; k < kMaxRows / 2; ++k) {
                        const int r = (kMaxRows / 2) * ch + k;
                        if (rv[k] && r < n_live_g) atomicAdd(g_visit + (size_t)(kMaxRows * group + r) * a.slots + slot, 1u);
                    }
                }
#endif
            }
            if (j == 0) {
                // Initial reference of each row: the scaled score of the split's first key when that key
                // is visible to the row (thread L = 0 holds it), else -inf-like, which forces the exact
                // rescale below.  Any later score more than 2^8 above the reference raises it.
                if (L == 0) {
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        if (n0 + i < ML) ms.ref[n0 + i] = vis[i] ? x[i] * c : kRefInit;
                }
                ptx::named_bar_sync(1, kSoftThreads);
#pragma unroll
                for (int i = 0; i < kCols; ++i) ref[i] = ms.ref[n0 + i];
            }
            float p[kCols];
            float pmax = 0.0f;
#pragma unroll
            for (int i = 0; i < kCols; ++i) {
                p[i] = vis[i] ? ptx::ex2(fmaf(x[i], c, -ref[i])) : 0.0f;
                pmax = fmaxf(pmax, p[i]);
            }
            // raise the reference maxima only when a probability exceeds 2^8 (CTA-wide vote)
            const unsigned want = __any_sync(0xffffffffu, !(pmax <= kThresh));
            if (lane == 0) ms.vote[j & 1][sw] = want ? 1 : 0;
            ptx::named_bar_sync(1, kSoftThreads);
            if (j == 0 && sw == 0 && lane == 0) VA_TRACE_AT(250);
            int any = 0;
#pragma unroll
            for (int w = 0; w < kSoftWarps; ++w) any |= ms.vote[j & 1][w];
            if (any) {
                // PV(j-1) must be done before the accumulator is rescaled.  (s_full(j) was committed after
                // PV(j-2), so pv_done can be at most one phase behind here.)
                if (j > 0 && !ptx::mbar_wait(bar(ms.pv_done), (j - 1) & 1, abort_flag, kWaitNs)) ok = false;
                float v[kCols];
#pragma unroll
                for (int i = 0; i < kCols; ++i) v[i] = vis[i] ? x[i] * c : -INFINITY;
                warp_reduce_scatter24<true>(v, lane);
                const int cb = n0 + scatter_col_base(lane);
                if ((lane & 3) == 0) {
                    ms.red[q][cb] = v[0];
                    ms.red[q][cb + 1] = v[1];
                    ms.red[q][cb + 2] = v[2];
                }
                ptx::named_bar_sync(1, kSoftThreads);
                if (ch == 0 && L < kMaxM) {
                    const float cm = fmaxf(fmaxf(ms.red[0][L], ms.red[1][L]), fmaxf(ms.red[2][L], ms.red[3][L]));
                    const float old = ms.ref[L];
                    const float nw = fmaxf(old, cm);
                    ms.alpha[L] = (nw == old) ? 1.0f : ptx::ex2(old - nw);
                    ms.ref[L] = nw;
                }
                ptx::named_bar_sync(1, kSoftThreads);
                if (j == 0 && sw == 0 && lane == 0) VA_TRACE_AT(251);
#pragma unroll
                for (int i = 0; i < kCols; ++i) {
                    ref[i] = ms.ref[n0 + i];
                    l[i] *= ms.alpha[n0 + i];
                    p[i] = vis[i] ? ptx::ex2(fmaf(x[i], c, -ref[i])) : 0.0f;
                }
                if (j > 0) {
                    ptx::tc_fence_after();
#pragma unroll
                    for (int part = 0; part < 2; ++part) {   // the accumulators of P_hi V and P_lo V
                        const uint32_t col = tl + kColO + kColLo * part + n0;
                        float o[kCols];
                        ptx::tmem_ld24_wait(col, o);
#pragma unroll
                        for (int i = 0; i < kCols; ++i) o[i] *= ms.alpha[n0 + i];
                        ptx::tmem_st16(col, o);
                        ptx::tmem_st8(col + 16, o + 16);
                    }
                    ptx::tmem_wait_st();
                }
            }
            // running sums; hi/lo bf16 split of P for the PV product
            uint32_t hi_w[kCols / 2], lo_w[kCols / 2];
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) {
                const float p0 = p[2 * i], p1 = p[2 * i + 1];
                l[2 * i] += p0;
                l[2 * i + 1] += p1;
                const uint32_t hb = pack_bf16x2(p0, p1);
                hi_w[i] = hb;
                lo_w[i] = pack_bf16x2(p0 - __uint_as_float(hb << 16), p1 - __uint_as_float(hb & 0xFFFF0000u));
            }
            if (j == 0 && sw == 0 && lane == 0) VA_TRACE_AT(252);
            // V rows of positions this split does not own are zeroed before PV reads them (column half ch)
            const int vs = j % kNV;
            if (kbase < own_lo || kbase + nkeys > own_hi) {
                if (!ptx::mbar_wait(bar(ms.v_full[vs]), (j / kNV) & 1, abort_flag, kWaitNs)) ok = false;
                if (L < nkeys && (kp < own_lo || kp >= own_hi)) {
                    uint4* row = reinterpret_cast<uint4*>(base + kOffV + vs * kStage + ch * kDHalf +
                                                          (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) row[cc] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // row L of P^T (keys x 48 matrix rows), columns [n0, n0 + 24): 16-byte chunks 3 ch .. 3 ch + 2,
            // written over K of this tile (QK(j) has completed: S^T(j) was read above)
            {
                const uint32_t roff = kOffK + (uint32_t)(j % kNK) * kStage + (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const uint32_t off = roff + ((uint32_t)((3 * ch + k) ^ (L & 7)) << 4);
                    *reinterpret_cast<uint4*>(base + kPhiInStage + off) =
                        make_uint4(hi_w[4 * k], hi_w[4 * k + 1], hi_w[4 * k + 2], hi_w[4 * k + 3]);
                    *reinterpret_cast<uint4*>(base + kPloInStage + off) =
                        make_uint4(lo_w[4 * k], lo_w[4 * k + 1], lo_w[4 * k + 2], lo_w[4 * k + 3]);
                }
            }
            if (j == 0 && sw == 0 && lane == 0) VA_TRACE_AT(253);
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.p_full[j & 1]));
            if (sw == 0 && lane == 0) VA_TRACE_TILE(j, 5);
        }
        // ------------------------------------------------------------ epilogue
        // row sums first: they do not depend on the last PV, which is still running
        warp_reduce_scatter24<false>(l, lane);
        {
            const int cb = n0 + scatter_col_base(lane);
            if ((lane & 3) == 0) {
                ms.red[q][cb] = l[0];
                ms.red[q][cb + 1] = l[1];
                ms.red[q][cb + 2] = l[2];
            }
        }
        ptx::named_bar_sync(1, kSoftThreads);
        if (ch == 0 && L < kMaxM) {
            const float lt = (ms.red[0][L] + ms.red[1][L]) + (ms.red[2][L] + ms.red[3][L]);
            ms.alpha[L] = lt;
            ms.inv_l[L] = lt > 0.0f ? 1.0f / lt : 0.0f;
        }
        ptx::named_bar_sync(1, kSoftThreads);
        if (!ptx::mbar_wait(bar(ms.o_ready), 0, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        float o[kCols], o_lo[kCols];
        ptx::tmem_ld24_wait(tl + kColO + n0, o);
        ptx::tmem_ld24_wait(tl + kColO + kColLo + n0, o_lo);
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
            const int n = n0 + i;
            if (n < M) part_o[n * kD + L] = (o[i] + o_lo[i]) * ms.inv_l[n];
        }
        if (ch == 0 && L < M) {
            const float lt = ms.alpha[L];
            part_lse[L] = lt > 0.0f ? (ms.ref[L] + log2f(lt)) * 0.6931471805599453f : -INFINITY;
        }
        if (!ok) fail();
    }

    // ---------------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) VA_TRACE_AT(2);
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

// [rows][128] bf16, boxes of box_rows rows x 64 columns with the 128-byte swizzle; rows past the end
// read as zero.
bool encode_rows_map(CUtensorMap* map, const void* base, int rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps already encoded by this host thread.  A map is a function of (address, rows, box, format)
// alone, so a caller that passes the same cache or q buffer again reuses its encoding instead of paying
// for cuTensorMapEncodeTiled on every call; a new address is a new key (no invalidation is needed).
bool cached_map(CUtensorMap* map, MapEncodeFn encode, const void* base, int rows, int box_rows) {
    struct Key {
        MapEncodeFn encode;
        const void* base;
        int rows, box_rows;
    };
    constexpr int kEntries = 32;
    thread_local Key keys[kEntries];
    thread_local CUtensorMap maps[kEntries];
    thread_local int used = 0, next = 0;
    for (int i = 0; i < used; ++i) {
        const Key& k = keys[i];
        if (k.encode == encode && k.base == base && k.rows == rows && k.box_rows == box_rows) {
            *map = maps[i];
            return true;
        }
    }
    if (!encode(map, base, rows, box_rows)) return false;
    const int slot = used < kEntries ? used++ : next;
    next = (slot + 1) % kEntries;
    keys[slot] = Key{encode, base, rows, box_rows};
    maps[slot] = *map;
    return true;
}

}  // namespace tc

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream) {
    if (a.n_groups < 1 || a.n_groups * kMaxRows < a.n_rows || (a.n_groups > 1 && !a.tree)) return cudaErrorInvalidValue;
    CUtensorMap tmq, tmk, tmv, tmk2, tmv2;
    const tc::MapEncodeFn enc = tc::encode_rows_map;
    if (!tc::cached_map(&tmq, enc, a.q, a.n_rows * kH, 48) || !tc::cached_map(&tmk, enc, a.k, a.slots, 64) ||
        !tc::cached_map(&tmv, enc, a.v, a.slots, 64) || !tc::cached_map(&tmk2, enc, a.k, a.slots, 128) ||
        !tc::cached_map(&tmv2, enc, a.v, a.slots, 128))
        return cudaErrorInvalidValue;
    const bool append = a.k_new != nullptr;
    const bool tree = VA_TREE_TEMPLATE && a.tree != nullptr;
    const void* fn = append ? (const void*)tc::attn_tc_kernel<true, false>
                            : tree ? (const void*)tc::attn_tc_kernel<false, true> : (const void*)tc::attn_tc_kernel<false, false>;
    cudaError_t e = ensure_smem_attr(fn, (int)tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3(a.n_splits, a.n_groups), dim3(tc::kThreads), tc::kSmemBytes, stream);
    e = append ? cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<true, false>, a, tmq, tmk, tmv, tmk2, tmv2)
        : tree ? cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<false, true>, a, tmq, tmk, tmv, tmk2, tmv2)
               : cudaLaunchKernelEx(&cfg, tc::attn_tc_kernel<false, false>, a, tmq, tmk, tmv, tmk2, tmv2);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va

#ifdef VA_DEBUG_VISIT
// Debug build only: point the split kernel's visit map at a device buffer of n_rows x slots unsigned
// counts, zeroed by the caller (NULL turns it off).
extern "C" VA_API int va_debug_set_visit(void* device_buffer) {
    unsigned* p = static_cast<unsigned*>(device_buffer);
    return cudaMemcpyToSymbol(va::tc::g_visit, &p, sizeof p) == cudaSuccess ? VA_OK : VA_CUDA_ERROR;
}
#endif

#ifdef VA_TRACE
// Debug build only: point the split kernel's timeline probe at a device buffer of n_splits x 256
// unsigned 64-bit words (NULL turns it off).
extern "C" VA_API int va_debug_set_trace(void* device_buffer) {
    unsigned long long* p = static_cast<unsigned long long*>(device_buffer);
    return cudaMemcpyToSymbol(va::tc::g_trace, &p, sizeof p) == cudaSuccess ? VA_OK : VA_CUDA_ERROR;
}
#endif
