// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "verify_attn.h"

// VA_Q8_FUSED_APPEND: verify_attn_q8_step codes its live rows inside the attention launch (the split
// that owns them, before it loads their tile) instead of in a separate append launch before it.
#ifndef VA_Q8_FUSED_APPEND
#define VA_Q8_FUSED_APPEND 1
#endif
// VA_TREE_TEMPLATE: tree calls launch their own instantiation of the split kernels (0: one instantiation
// tests a.tree at run time), so that each instantiation carries less code: a launch runs from a cold
// instruction cache.
#ifndef VA_TREE_TEMPLATE
#define VA_TREE_TEMPLATE 1
#endif

namespace va {

constexpr int kD = VA_HEAD_DIM;        // 128
constexpr int kH = VA_Q_HEADS;         // 6
constexpr int kMaxRows = VA_MAX_ROWS;  // 8
constexpr int kTile = VA_TILE;         // 64
constexpr int kMaxM = kH * kMaxRows;   // 48 matrix rows
constexpr int kMaxNodes = VA_MAX_TREE_NODES;   // 16: two groups of kMaxRows rows

// Arguments of one split-KV attention launch (full attention: window == 0).
struct AttnArgs {
    const uint16_t* q;       // [n_rows][6][128] bf16
    const uint16_t* k;       // [slots][128] bf16
    const uint16_t* v;       // [slots][128] bf16
    const int32_t* pos;      // [n_rows] (chain calls)
    const int32_t* tree;     // tree calls: [1 + n_live] base, then ancestor-or-self masks; nullptr for chains
    float* part_o;           // [S][n_rows][6][128]
    float* part_lse;         // [S][n_rows][6]
    int32_t* dev_status;     // optional
    float scale;
    int n_rows, n_live, slots, window, n_splits;
    int n_groups;            // groups of kMaxRows rows (grid.y); 1 for chain calls
    // verify_attn_step (chain calls only, null otherwise): the split owning a live row's position
    // writes that row of k_new / v_new to its slot before loading the row's tile.
    const uint16_t* k_new = nullptr;   // [n_live][128] bf16
    const uint16_t* v_new = nullptr;
};

// Extent and split ownership derived on the device from the positions.
// IQuestRT report, "Read only the KV tiles needed by the current positions": the current
// positions determine the read extent; the sequence is partitioned across CTAs.
struct Plan {
    long long lo, hi;      // visible extent [lo, hi) of the live rows
    long long t0, t1;      // this split's 64-position tiles [t0, t1)
    int status;            // VA_DEV_* bits, 0 if the positions are usable
};

// Split s of S owns tiles [t_lo + floor(s T / S), t_lo + floor((s + 1) T / S)) of the extent's T tiles.
// 0 <= lo < hi here.  floor(s T / S) = s q + floor(s r / S) with T = q S + r: 32-bit arithmetic only,
// since s r < S^2 <= VA_MAX_SPLITS^2 = 2^24 and T < 2^31 (64-bit divisions cost a warp ~0.1 us each).
__device__ __forceinline__ void deal_tiles(Plan& P, int n_splits, int split) {
    const long long tlo = P.lo / kTile;
    const long long thi = (P.hi + kTile - 1) / kTile - 1;
    const unsigned T = (unsigned)(thi - tlo + 1), S = (unsigned)n_splits, s = (unsigned)split;
    const unsigned q = T / S, r = T % S;
    P.t0 = tlo + (long long)(s * q + (s * r) / S);
    P.t1 = tlo + (long long)((s + 1) * q + ((s + 1) * r) / S);
}

// row_pos[] holds the live rows' positions (entries past n_live are ignored).  Callers load them once
// per CTA (one request) and share them: every thread of every CTA loading the same eight integers
// turns one L2 line into a hot spot that costs microseconds.
__device__ __forceinline__ Plan make_plan(const int (&row_pos)[kMaxRows], int n_live, int window, int slots,
                                          int n_splits, int split) {
    Plan P;
    P.lo = P.hi = P.t0 = P.t1 = 0;
    P.status = 0;
    if (n_live <= 0) return P;
    const int p0 = row_pos[0];
    int prev = p0, last = p0;
    if (p0 < 0) P.status |= VA_DEV_NEGATIVE_POS;
#pragma unroll
    for (int r = 1; r < kMaxRows; ++r) {
        if (r >= n_live) break;
        const int p = row_pos[r];
        if (p < 0) P.status |= VA_DEV_NEGATIVE_POS;
        if (p < prev) P.status |= VA_DEV_NOT_MONOTONE;
        prev = p;
        last = p;
    }
    if (window == 0 && (long long)last >= (long long)slots) P.status |= VA_DEV_BEYOND_CACHE;
    if (window > 0 && (long long)last - p0 > (long long)slots - window) P.status |= VA_DEV_RING_SPAN;
    if (P.status) return P;
    P.hi = (long long)last + 1;
    P.lo = window > 0 ? max(0LL, (long long)p0 - window + 1) : 0LL;
    deal_tiles(P, n_splits, split);
    return P;
}

// Depth of a tree node: the number of its strict ancestors.
__device__ __forceinline__ int tree_depth(int mask) { return __popc((unsigned)mask) - 1; }

// Extent and split ownership of a tree call ("Qwen3.8-27B on one RTX 4090", section "More tokens per
// round: verify trees").  Node i sits at slot base + i and sees the prefix from its window start
// base + depth_i - window + 1 (0 for full attention) and the nodes of its ancestor-or-self mask.
// The extent is [lo, base + n_nodes) with lo the earliest window start over the nodes.
__device__ __forceinline__ Plan make_tree_plan(int base, const int (&anc)[kMaxNodes], int n_nodes, int window,
                                               int slots, int n_splits, int split) {
    Plan P;
    P.lo = P.hi = P.t0 = P.t1 = 0;
    P.status = 0;
    if (n_nodes <= 0) return P;
    if (base < 0) P.status |= VA_DEV_NEGATIVE_POS;
    int dmin = kMaxNodes;
#pragma unroll
    for (int i = 0; i < kMaxNodes; ++i) {
        if (i >= n_nodes) break;
        const unsigned m = (unsigned)anc[i];
        if (!((m >> i) & 1u) || (m >> n_nodes) != 0u) P.status |= VA_DEV_TREE_MASK;
        dmin = min(dmin, tree_depth((int)m));
    }
    const long long hi = (long long)base + n_nodes;
    if (window == 0 && hi > (long long)slots) P.status |= VA_DEV_BEYOND_CACHE;
    if (window > 0 && hi - ((long long)base + dmin - window + 1) > (long long)slots) P.status |= VA_DEV_RING_SPAN;
    if (P.status) return P;
    P.hi = hi;
    P.lo = window > 0 ? min((long long)base, max(0LL, (long long)base + dmin - window + 1)) : 0LL;
    deal_tiles(P, n_splits, split);
    return P;
}

// Host-side tensor-map encoders (attn_tc.cu, attn_q8.cu) and the per-thread cache of their results.
namespace tc {
typedef bool (*MapEncodeFn)(CUtensorMap* map, const void* base, int rows, int box_rows);
bool encode_rows_map(CUtensorMap* map, const void* base, int rows, int box_rows);
bool cached_map(CUtensorMap* map, MapEncodeFn encode, const void* base, int rows, int box_rows);
}  // namespace tc

// Opt a kernel into `bytes` of dynamic shared memory on the current device, once per device
// (so that a later launch under stream capture issues no attribute call).
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Launch configuration with programmatic stream serialisation: the kernel may start while the previous
// kernel of the stream finishes; it waits for it (griddepcontrol.wait) before touching memory.
inline void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream) {
    cfg->gridDim = grid;
    cfg->blockDim = block;
    cfg->dynamicSmemBytes = smem;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

// Launchers (return the cudaError_t of the launch).
cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, int n_live, uint16_t* k_cache,
                          uint16_t* v_cache, int slots, const int32_t* pos, int32_t* dev_status,
                          cudaStream_t stream);
cudaError_t launch_attn(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const float* part_o, const float* part_lse, int n_splits, const float* sink,
                           int n_rows, int n_live, uint16_t* out, float* out_lse, cudaStream_t stream);

}  // namespace va
