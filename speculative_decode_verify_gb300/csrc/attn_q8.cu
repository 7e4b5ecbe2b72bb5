// Split-KV verify attention over the quantised K/V cache: keys FP8 (E4M3) after a Hadamard rotation,
// values INT8, one fp32 scale per cached row ("Qwen3.8-27B on one RTX 4090", section "A cheaper cache
// and state").  The split plan, masks, partials and combine are those of the bf16 kernel (IQuestRT
// report, "Read only the KV tiles needed by the current positions", "Expose more parallelism in
// attention").
//
// Design for one GB300 SM per split (same roles as the bf16 kernel: warp 0 K loads, warp 1 MMAs,
// warp 2 V loads, warps 3..10 softmax):
//   * A 128-position tile is 16 KB of K codes plus 16 KB of V codes (half the bf16 bytes), so the rings
//     hold K 5 / V 3 tiles.  Each tile's 128 row scales arrive with it by a bulk copy on the same barrier.
//   * QK runs on the codes as stored: S^T[128 keys x 48] = K8 . Qr^T with tcgen05 kind::f8f6f4 (E4M3 x
//     E4M3).  q is rotated on the tensor core first: the +-1 Hadamard matrix (exact in bf16) is written
//     once into the idle fp16 V buffer and one bf16 MMA forms (H q)^T in TMEM; the softmax warps then
//     scale each row by a power of two s_r into [128, 256) and split it into three E4M3 terms
//     (q = s_r (e1 + e2 + e3) up to 2^-12 relative), so QK is three MMAs per 32-wide step.
//     The score of key j is then scale / 128 * s_r * k_scale_j * S^T.
//   * PV runs in fp16 (kind::f16): the softmax warps widen the tile's INT8 values to fp16 in shared
//     memory (exact), and write P' = p * v_scale_j as fp16 (one term: 2^-12 relative) over the tile's
//     K codes once QK has read them.  The running sums use p itself.
//   * The V code stage is released as soon as it is widened; the fp16 V buffer is double-buffered and
//     reused once the PV two tiles back has completed.
//   * Draft trees ("Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees", over the
//     cache of "A cheaper cache and state"): as in the bf16 kernel, each node's ancestor mask replaces the
//     causal tail in the node region, and up to 16 nodes run as two groups of 8 rows (grid.y).
#include <cuda.h>
#include <cuda_fp16.h>

#include <climits>
#include <cstring>
#include <mutex>

#include "codec_dev.cuh"
#include "kv_codec.h"
#include "tc_ptx.cuh"
#include "va_internal.cuh"

namespace va {
namespace tc {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();                                                  // attn_tc.cu
bool encode_rows_map(CUtensorMap* map, const void* base, int rows, int box_rows);   // attn_tc.cu: bf16 rows
}  // namespace tc

namespace q8 {

#ifndef VA_POLL_EVERY
#define VA_POLL_EVERY 64
#endif
// VA_POLL_EVERY: the MMA issuer's poll loop reads the timer and the abort flag (its give-up checks) once
// every VA_POLL_EVERY rounds that find nothing ready, which shortens a round (64 against 1: -0.01 us per
// 192K quantised verify call).

// Tiles of a split pulled into L2 before the launch dependency resolves (0: none), as in the bf16 kernel.
// Measured on GB300 at 192K: +0.4 us per launch and +2.7 us per verify_attn_q8_step call with 2 tiles
// (+1.5 us at 1K), so off: this kernel's start is not where its time goes.
#ifndef VA_PREWARM
#define VA_PREWARM 0
#endif

// QK sums the three q terms in the tensor core (three N = 48 MMAs per k-step into one accumulator), so the
// softmax warps read one 48-column score block; 0: one N = 144 MMA per k-step (each K slice read once) and
// the three blocks added by the softmax warps.
#ifndef VA_Q8_ACC3
#define VA_Q8_ACC3 0
#endif

constexpr int kNK = 5;                     // K code ring depth (tiles of 128 positions); P' reuses K's stage
constexpr int kNV = 3;                     // V code ring depth
constexpr uint32_t kStage = 16384;         // 128 positions x 128 codes
constexpr uint32_t kHalfBox = 8192;        // one TMA box: 64 positions x 128 codes
constexpr uint32_t kV16Half = 16384;       // fp16 V: 128 positions x 64 d
constexpr uint32_t kV16 = 2 * kV16Half;
constexpr uint32_t kQTerm = 6144;          // one E4M3 term of q: 48 rows x 128 codes
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kNK * kStage;
constexpr uint32_t kOffV16 = kOffV + kNV * kStage;
constexpr uint32_t kOffQ = kOffV16 + 2 * kV16;
constexpr uint32_t kOffMisc = kOffQ + 3 * kQTerm;
constexpr uint32_t kOffH = kOffV16;              // +-1 Hadamard matrix, bf16 K-major (two 16 KB d halves)
constexpr uint32_t kOffQStage = kOffV16 + kV16;  // q, bf16 K-major (two 6 KB d halves)
constexpr uint32_t kQHalf16 = 6144;
// Softmax / widening warps: 8 (two column halves of the 48 matrix rows, 24 columns a thread) or 16 (four
// column quarters, 12 columns a thread, 96 registers).  Measured on GB300 at 192K: 16 warps +0.8 us per
// launch, bit-identical: each step of a tile takes as long with half the work a warp (the exponentials
// are bound by the MUFU pipe, 6,144 a tile and SM, and the rest by fixed latencies), so 8.
#ifndef VA_Q8_SOFT_WARPS
#define VA_Q8_SOFT_WARPS 8
#endif
constexpr int kSoftWarps = VA_Q8_SOFT_WARPS;
static_assert(kSoftWarps == 8 || kSoftWarps == 16, "softmax warps: 8 or 16");
constexpr int kSoftWarp0 = 3;
constexpr int kThreads = 32 * (kSoftWarp0 + kSoftWarps);
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kColParts = kSoftWarps / 4;        // column parts: each lane quadrant has one warp per part
constexpr int kCols = kMaxM / kColParts;         // matrix rows (accumulator columns) per softmax thread
constexpr int kPartRows = kMaxRows / kColParts;  // verify rows per column part
constexpr int kVChunks = 8 / kColParts;          // 16-code chunks of a V row widened per thread
// S^T of a tile is three 48-column blocks, one per E4M3 term of q (QK runs as one N = 144 MMA per k-step,
// so that each K slice is read once), in VA_Q8_S_BUFS buffers; then O^T (48 columns).
constexpr uint32_t kTmemCols = 512;
// Order of a tile's steps in the softmax warps.  0: widen V, then the scores; 1: the scores' TMEM loads
// first, then V's codes, and the widening in the same block of code as the exponentials, so that the
// INT8 -> fp16 work (ALU, shared stores) fills the time the exponentials spend in the MUFU pipe.
// Measured on GB300 at 192K (per launch, back to back, bit-identical): 1 alone -0.23 us; with three score
// buffers (VA_Q8_S_BUFS) -0.94 us (19.67 -> 18.74 us); three buffers alone +0.09 us.
#ifndef VA_Q8_FUSE
#define VA_Q8_FUSE 1
#endif
// The per-tile vote on raising the reference maximum: 0 a block barrier of the softmax warps; 1 an mbarrier
// (split phase): each warp arrives with its vote, writes P' as if no warp wanted a rescale, then waits and
// rewrites P' in the rare tile that needs one.  Measured on GB300 at 192K: +0.03 us per launch, so 0.
#ifndef VA_Q8_VOTE_MB
#define VA_Q8_VOTE_MB 0
#endif
// VA_Q8_S_BUFS score buffers: QK may run that many tiles minus one ahead of PV (see VA_Q8_FUSE).
#ifndef VA_Q8_S_BUFS
#define VA_Q8_S_BUFS 3
#endif
constexpr int kSBufs = VA_Q8_S_BUFS;
static_assert(kSBufs == 2 || kSBufs == 3, "score buffers: 2 or 3");
constexpr uint32_t kSStride = kSBufs == 2 ? 160 : 144;   // TMEM columns between score buffers
constexpr uint32_t kColS0 = 0, kColO = kSBufs * kSStride;
constexpr uint32_t kTermCols = 48;
constexpr float kThresh = 256.0f;
constexpr float kRefInit = -1.0e30f;
constexpr uint64_t kWaitNs = 2000000000ull;

struct Misc {
    uint64_t k_full[kNK], k_empty[kNK], v_full[kNV], v_empty[kNV];
    uint64_t q_tma, h_ready, q_rot, q_full, s_full[kSBufs], s_free[kSBufs], vote_bar[2], p_full[2], pv_done[2], o_ready, drain;
    uint64_t app_done;                // verify_attn_q8_step: this split's live rows are coded into the cache
    uint32_t tmem_base;
    int abort;
    int vote[2][kSoftWarps];
    float red[4][kMaxM];
    float ref[kMaxM];
    float alpha[kMaxM];
    float inv_l[kMaxM];
    float qsig[kMaxM];                // power-of-two scale of each rotated q row
    float qinv[kMaxM];
    long long row_lo[kMaxRows], row_hi[kMaxRows];
    long long tree_base;              // tree calls: slot of node 0; chain calls: no node region (LLONG_MAX)
    unsigned row_anc[kMaxRows];       // ancestor-or-self mask of each row of this CTA's group
    int anc[kMaxNodes];               // tree calls: every node's mask
    int base;
    __align__(16) float kscale[kNK][128];
    __align__(16) float vscale[kNV][128];
};
constexpr uint32_t kSmemBytes = kOffMisc + (uint32_t)sizeof(Misc) + 1024;
static_assert(kOffV16 % 1024 == 0 && kOffQ % 1024 == 0 && kOffMisc % 16 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");

// ------------------------------------------------------------------------------- small helpers
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
                 : "memory");
}

// Two floats to E4M3 codes (round to nearest even, saturating): lo in bits 0..7, hi in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Values of two E4M3 codes (lo in bits 0..7) by the hardware conversion to f16, which is exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t c) {
    float2 r;
    asm("{\n .reg .b32 h;\n .reg .f16 lo, hi;\n cvt.rn.f16x2.e4m3x2 h, %2;\n mov.b32 {lo, hi}, h;\n"
        " cvt.f32.f16 %0, lo;\n cvt.f32.f16 %1, hi;\n}" : "=f"(r.x), "=f"(r.y) : "h"((uint16_t)c));
    return r;
}

// Four INT8 codes (one 32-bit word) to four exact fp16 values: 1152 + x is exact in fp16 for x in
// [-128, 127], so the bytes are biased, placed under the exponent of 1024 and the bias is subtracted.
__device__ __forceinline__ void int8x4_to_half(uint32_t w, uint32_t& h01, uint32_t& h23) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    h01 = *reinterpret_cast<uint32_t*>(&ha);
    h23 = *reinterpret_cast<uint32_t*>(&hb);
}

// Packed fp32 pairs (one instruction for two IEEE round-to-nearest operations, each rounded as the scalar
// operation would be).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 r;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n add.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}" : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 r;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mul.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}" : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

// This thread's kCols accumulator columns of its TMEM lane from taddr on, loaded (then waited for) or stored.
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[kCols]) {
    if constexpr (kCols == 24) ptx::tmem_ld24_wait(taddr, v);
    else ptx::tmem_ld12_wait(taddr, v);
}
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[kCols]) {
    if constexpr (kCols == 24) {
        ptx::tmem_st16(taddr, v);
        ptx::tmem_st8(taddr + 16, v + 16);
    } else {
        ptx::tmem_st8(taddr, v);
        ptx::tmem_st4(taddr + 8, v + 8);
    }
}

__device__ __forceinline__ int scatter_col_base(int lane) {
    return kCols == 24 ? ((lane >> 4) & 1) * 12 + ((lane >> 3) & 1) * 6 + ((lane >> 2) & 1) * 3
                       : ((lane >> 4) & 1) * 6 + ((lane >> 3) & 1) * 3;
}
// the lanes that hold distinct column totals after warp_reduce_scatter
__device__ __forceinline__ bool scatter_writer(int lane) { return (lane & (kCols == 24 ? 3 : 7)) == 0; }

// Reduce the kCols per-thread columns over the warp; afterwards the lane holds the warp totals of columns
// [scatter_col_base(lane), +3) in v[0..2].
template <bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[kCols], int lane) {
#define VA_STAGE(W, BIT)                                                   \
    _Pragma("unroll") for (int i = 0; i < (W); ++i) {                      \
        const bool up = (lane & (BIT)) != 0;                               \
        const float send = up ? v[i] : v[i + (W)];                         \
        const float keep = up ? v[i + (W)] : v[i];                         \
        const float got = __shfl_xor_sync(0xffffffffu, send, (BIT));       \
        v[i] = kMax ? fmaxf(keep, got) : keep + got;                       \
    }
    VA_STAGE(kCols / 2, 16)
    VA_STAGE(kCols / 4, 8)
    if (kCols == 24) {
        VA_STAGE(3, 4)
    }
#undef VA_STAGE
#pragma unroll
    for (int b = kCols == 24 ? 2 : 4; b >= 1; b >>= 1)
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const float got = __shfl_xor_sync(0xffffffffu, v[i], b);
            v[i] = kMax ? fmaxf(v[i], got) : v[i] + got;
        }
}

// kAppend: the verify_attn_q8_step instantiation, which codes the live rows itself (a.k_new / a.v_new);
// the instantiation without it carries none of that code.  kTree: the instantiation for tree calls (a.tree
// set), as in the bf16 kernel (VA_TREE_TEMPLATE).
template <bool kAppend, bool kTree>
__global__ void __launch_bounds__(kThreads, 1)
attn_q8_kernel(const AttnArgs a, const float* __restrict__ kscale_g, const float* __restrict__ vscale_g,
               const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const __grid_constant__ CUtensorMap tmk2, const __grid_constant__ CUtensorMap tmv2) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw_s = ptx::smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    Misc& ms = *reinterpret_cast<Misc*>(base + kOffMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, group = blockIdx.y;
    const bool is_tree = VA_TREE_TEMPLATE ? kTree : a.tree != nullptr;
    // rows of this CTA: group g holds rows 8 g .. 8 g + 7 (one group for chains)
    const int n_live_g = is_tree ? min(max(a.n_live - kMaxRows * group, 0), kMaxRows) : a.n_live;
    const int M_all = a.n_rows * kH;
    const int M = min(kMaxM, M_all - kMaxM * group);
    const int ML = n_live_g * kH;
    auto bar = [](const uint64_t& b) { return ptx::smem_u32(&b); };

    // ---------------------------------------------------------------- set-up without global memory
    if (tid == 0) {
        ptx::mbar_init(bar(ms.q_tma), 1);
        ptx::mbar_init(bar(ms.h_ready), kSoftWarps);
        ptx::mbar_init(bar(ms.q_rot), 1);
        ptx::mbar_init(bar(ms.q_full), kSoftWarps);
        for (int i = 0; i < kNK; ++i) {
            ptx::mbar_init(bar(ms.k_full[i]), 1);
            ptx::mbar_init(bar(ms.k_empty[i]), 1);
        }
        for (int i = 0; i < kNV; ++i) {
            ptx::mbar_init(bar(ms.v_full[i]), 1);
            ptx::mbar_init(bar(ms.v_empty[i]), kSoftWarps);
        }
        for (int i = 0; i < kSBufs; ++i) {
            ptx::mbar_init(bar(ms.s_full[i]), 1);
            ptx::mbar_init(bar(ms.s_free[i]), kSoftWarps);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(ms.vote_bar[i]), kSoftWarps);
            ptx::mbar_init(bar(ms.p_full[i]), kSoftWarps);
            ptx::mbar_init(bar(ms.pv_done[i]), 1);
        }
        ptx::mbar_init(bar(ms.o_ready), 1);
        ptx::mbar_init(bar(ms.drain), 1);
        ptx::mbar_init(bar(ms.app_done), kSoftWarps);
        ms.abort = 0;
        ptx::mbar_init_fence();
    }
    if (tid == 32) {
        ptx::tma_prefetch_desc(&tmq);
        ptx::tma_prefetch_desc(&tmk);
        ptx::tma_prefetch_desc(&tmv);
        ptx::tma_prefetch_desc(&tmk2);
        ptx::tma_prefetch_desc(&tmv2);
    }
    if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&ms.tmem_base), kTmemCols);
    // the +-1 Hadamard matrix H[i][j] = (-1)^popcount(i & j) as the bf16 A operand of the rotation, written
    // by the softmax warps before the dependency wait (it needs no global memory): thread st writes row
    // st & 127, d half (st >> 7) & 1, kHChunks of its eight 16-byte chunks of 8 entries (128-byte swizzle)
    if (warp >= kSoftWarp0) {
        constexpr int kHChunks = 8 * 256 / kSoftThreads;
        const int st = (warp - kSoftWarp0) * 32 + lane, row = st & 127, h = (st >> 7) & 1;
        const int c0 = (st >> 8) * kHChunks;
        const uint32_t roff = kOffH + (uint32_t)h * 16384u + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u;
#pragma unroll
        for (int c = c0; c < c0 + kHChunks; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int d0 = 64 * h + 8 * c + 2 * e;
                const uint32_t lo = (__popc((unsigned)(row & d0)) & 1) ? 0xBF80u : 0x3F80u;
                const uint32_t hi = (__popc((unsigned)(row & (d0 + 1))) & 1) ? 0xBF80u : 0x3F80u;
                w[e] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(base + roff + (((uint32_t)c ^ (uint32_t)(row & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
        ptx::fence_proxy_async_smem();
    }
    // the only block barrier before the roles start: barriers, TMEM and H are in place.  After the launch
    // dependency every warp reads the positions itself and derives the plan, so the producers request
    // tiles, the MMA thread rotates q and the softmax warps code it without waiting for one another
    // (measured on GB300 against a positions -> barrier -> plan -> row set-up -> barrier start: 192K launch
    // 18.46 -> 17.92 us back to back, 1K call 10.90 -> 10.07 us)
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp >= kSoftWarp0 && lane == 0) ptx::mbar_arrive(bar(ms.h_ready));   // H is written

    ptx::griddep_launch_dependents();
#if VA_PREWARM
    // a thread off the start's critical path pulls this split's first tiles (codes and row scales) into L2,
    // and their address translations into the TLBs, while the kernel before may still run: from positions (or
    // a tree descriptor) read now, a hint only (an L2 prefetch of the wrong lines costs bandwidth, never a
    // result)
    if (tid == 2 * 32 + 31 && n_live_g > 0) {   // lane 31 of the V producer warp: idle until the tail
        Plan Q;
        if (!is_tree) {
            int sp[kMaxRows];
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) sp[r] = (r < a.n_live) ? ptx::ld_relaxed_int(a.pos + r) : 0;
            Q = make_plan(sp, a.n_live, a.window, a.slots, a.n_splits, split);
        } else {
            int anc[kMaxNodes];
#pragma unroll
            for (int i = 0; i < kMaxNodes; ++i) anc[i] = (i < a.n_live) ? ptx::ld_relaxed_int(a.tree + 1 + i) : 0;
            Q = make_tree_plan(ptx::ld_relaxed_int(a.tree), anc, a.n_live, a.window, a.slots, a.n_splits, split);
        }
        for (int j = 0; !Q.status && j < VA_PREWARM && Q.t0 + 2LL * j < Q.t1; ++j) {
            const long long t = Q.t0 + 2LL * j;
            const int halves = (t + 1 < Q.t1) ? 2 : 1;
            const int s0 = (int)((t * kTile) % a.slots), s1 = (int)(((t + 1) * kTile) % a.slots);
            if (halves == 2 && s1 == s0 + kTile) {
                ptx::tma_prefetch_l2_2d(&tmk2, 0, s0);
                ptx::tma_prefetch_l2_2d(&tmv2, 0, s0);
            } else {
                for (int hh = 0; hh < halves; ++hh) {
                    ptx::tma_prefetch_l2_2d(&tmk, 0, hh ? s1 : s0);
                    ptx::tma_prefetch_l2_2d(&tmv, 0, hh ? s1 : s0);
                }
            }
            for (int hh = 0; hh < halves; ++hh) {
                ptx::bulk_prefetch_l2(kscale_g + (hh ? s1 : s0), 256u);
                ptx::bulk_prefetch_l2(vscale_g + (hh ? s1 : s0), 256u);
            }
        }
    }
#endif
    ptx::griddep_wait();   // every global access of this kernel comes after this (the prefetches above only
                           // pick lines for L2)

    // q first (two 48-row boxes, 128-byte swizzle, the B operand of the rotation) into the second fp16 V
    // buffer, which is idle until the second tile is widened.  The K and V tiles are requested by their
    // producer warps as soon as they have the plan.
    if (tid == 0) {
        const uint64_t keep = ptx::policy_evict_last();
        ptx::mbar_arrive_expect_tx(bar(ms.q_tma), kMaxM * kD * 2);
        ptx::tma_load_2d_hint(base_s + kOffQStage, &tmq, 0, kMaxM * group, bar(ms.q_tma), keep);
        ptx::tma_load_2d_hint(base_s + kOffQStage + kQHalf16, &tmq, 64, kMaxM * group, bar(ms.q_tma), keep);
    }
    // the positions (or the tree): every warp reads them (one 32-byte request) and derives the plan
    int row_pos[kMaxRows];
    int tree_word = 0;   // tree calls: lane 0 the base, lane i + 1 node i's mask
    Plan P;
    if (!is_tree) {
        const int pv = lane < a.n_live ? ptx::ld_int_policy(a.pos + lane, ptx::policy_evict_last()) : 0;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) row_pos[r] = __shfl_sync(0xffffffffu, pv, r);
        P = make_plan(row_pos, a.n_live, a.window, a.slots, a.n_splits, split);
    } else {
        tree_word = lane <= a.n_live ? ptx::ld_int_policy(a.tree + lane, ptx::policy_evict_last()) : 0;
        int anc[kMaxNodes];
#pragma unroll
        for (int i = 0; i < kMaxNodes; ++i) anc[i] = i < a.n_live ? __shfl_sync(0xffffffffu, tree_word, i + 1) : 0;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) row_pos[r] = 0;
        P = make_tree_plan(__shfl_sync(0xffffffffu, tree_word, 0), anc, a.n_live, a.window, a.slots, a.n_splits, split);
    }
    if (P.status && split == 0 && group == 0 && tid == 0 && a.dev_status) atomicOr(a.dev_status, P.status);
    const int n64 = (P.status || n_live_g == 0) ? 0 : (int)(P.t1 - P.t0);
    const int ntiles = (n64 + 1) >> 1;
    float* part_o = a.part_o + ((long long)split * M_all + kMaxM * group) * kD;
    float* part_lse = a.part_lse + (long long)split * M_all + kMaxM * group;
    const long long own_lo = max(P.lo, P.t0 * kTile);
    const long long own_hi = min(P.hi, P.t1 * kTile);

    auto tile_slots = [&](int j, int& slot0, int& slot1, int& halves) {
        const long long t = P.t0 + 2LL * j;
        halves = (t + 1 < P.t1) ? 2 : 1;
        slot0 = (int)((t * kTile) % a.slots);
        slot1 = (int)(((t + 1) * kTile) % a.slots);
    };
    // codes of tile j (one 128-row box, or one 64-row box per half) and its row scales, on one barrier
    auto load_tile = [&](const CUtensorMap* m64, const CUtensorMap* m128, const float* scales, uint32_t stage,
                         uint32_t scale_dst, uint64_t& full, int j) {
        int s0, s1, halves;
        tile_slots(j, s0, s1, halves);
        const uint64_t pol = ptx::policy_evict_first();
        ptx::mbar_arrive_expect_tx(bar(full), (uint32_t)halves * (kHalfBox + 256u));
        if (halves == 2 && s1 == s0 + kTile) {
            ptx::tma_load_2d_hint(stage, m128, 0, s0, bar(full), pol);
        } else {
            for (int hh = 0; hh < halves; ++hh)
                ptx::tma_load_2d_hint(stage + hh * kHalfBox, m64, 0, hh ? s1 : s0, bar(full), pol);
        }
        for (int hh = 0; hh < halves; ++hh)
            bulk_load(scale_dst + hh * 256u, scales + (hh ? s1 : s0), 256u, bar(full), pol);
    };
    // verify_attn_q8_step: the live rows are coded into the cache by this launch (a.k_new set); a tile that
    // holds a live row's position is requested only after this split's softmax warps have written them
    // (app_done).  Positions never decrease, so the live rows are the positions [pos[0], hi).
    const bool fused_append = kAppend && a.k_new != nullptr;
    auto tile_has_new = [&](int j) {
        const long long t = P.t0 + 2LL * j;
        return fused_append && (long long)row_pos[0] < (t + ((t + 1 < P.t1) ? 2 : 1)) * kTile;
    };
    auto load_k = [&](int j) {
        load_tile(&tmk, &tmk2, kscale_g, base_s + kOffK + (uint32_t)(j % kNK) * kStage,
                  ptx::smem_u32(&ms.kscale[j % kNK][0]), ms.k_full[j % kNK], j);
    };
    auto load_v = [&](int j) {
        load_tile(&tmv, &tmv2, vscale_g, base_s + kOffV + (uint32_t)(j % kNV) * kStage,
                  ptx::smem_u32(&ms.vscale[j % kNV][0]), ms.v_full[j % kNV], j);
    };

    // row set-up by thread u (u < kMaxM): row u of this group (u < kMaxRows): the positions it sees inside this
    // split, [lo, hi), and its mask of the node region [tree_base, hi); the reference maximum of matrix row u
    auto row_setup = [&](int u) {
        if (u < kMaxRows) {
            long long lo = 0, hi = 0;
            unsigned m = 0xFFFFFFFFu;
            if (!is_tree) {
#pragma unroll
                for (int r = 0; r < kMaxRows; ++r) {
                    if (r == u && r < a.n_live) {
                        const long long p = row_pos[r];
                        lo = max(a.window > 0 ? max(0LL, p - a.window + 1) : 0LL, own_lo);
                        hi = min(p + 1, own_hi);
                    }
                }
            } else if (u < n_live_g) {
                m = (unsigned)ms.anc[kMaxRows * group + u];
                const long long logical = (long long)ms.base + tree_depth((int)m);   // the node's own position
                lo = max(a.window > 0 ? max(0LL, logical - a.window + 1) : 0LL, own_lo);
                hi = min(P.hi, own_hi);
            }
            if (hi < lo) hi = lo;
            ms.row_lo[u] = lo;
            ms.row_hi[u] = hi;
            ms.row_anc[u] = m;
            if (u == 0) ms.tree_base = is_tree ? (long long)ms.base : LLONG_MAX;
        }
        if (u < kMaxM) ms.ref[u] = u < ML ? kRefInit : INFINITY;
    };

    const uint32_t tmem = ms.tmem_base;
    volatile int* abort_flag = &ms.abort;
    auto fail = [&]() {
        *abort_flag = 1;
        if (a.dev_status) atomicOr(a.dev_status, VA_DEV_TIMEOUT);
    };

    if (ntiles == 0) {
        for (int i = tid; i < M * kD; i += kThreads) part_o[i] = 0.0f;
        for (int i = tid; i < M; i += kThreads) part_lse[i] = -INFINITY;
    } else if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ K (warp 0) / V (warp 2) code producers
        const bool is_k = warp == 0;
        const int depth = is_k ? kNK : kNV;
        if (lane == 0) {
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                uint64_t& empty = is_k ? ms.k_empty[j % kNK] : ms.v_empty[j % kNV];
                if ((tile_has_new(j) && !ptx::mbar_wait(bar(ms.app_done), 0, abort_flag, kWaitNs)) ||
                    !ptx::mbar_wait(bar(empty), ((j / depth) & 1) ^ 1, abort_flag, kWaitNs)) {
                    fail();
                    break;
                }
                if (is_k) load_k(j); else load_v(j);
                issued = j + 1;
            }
            for (int j = max(0, issued - depth); j < issued; ++j)   // every issued copy lands before exit
                ptx::mbar_wait(bar(is_k ? ms.k_full[j % kNK] : ms.v_full[j % kNV]), (j / depth) & 1, nullptr, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // QK: A = K codes, B = q terms, both E4M3 K-major; PV: A = V^T fp16, B = P'^T fp16, MN-major
            constexpr uint32_t idesc_qk =
                (1u << 4) | (0u << 7) | (0u << 10) | (((VA_Q8_ACC3 ? 48u : 144u) >> 3) << 17) | ((128u >> 4) << 24);
            constexpr uint32_t idesc_pv =
                (1u << 4) | (0u << 7) | (0u << 10) | (1u << 15) | (1u << 16) | ((48u >> 3) << 17) | ((128u >> 4) << 24);
            // rotation: (H q)^T [128 x 48] = H . q^T into the first S buffer (A = H, B = q: bf16, K-major)
            bool ok = ptx::mbar_wait(bar(ms.q_tma), 0, abort_flag, kWaitNs) &&
                      ptx::mbar_wait(bar(ms.h_ready), 0, abort_flag, kWaitNs);
            if (ok) {
                constexpr uint32_t idesc_rot = ptx::idesc_bf16_f32(128, 48, 0, 0);
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t h = (uint32_t)kk >> 2, off = (uint32_t)(kk & 3) * 32u;
                    ptx::mma_bf16(tmem + kColS0, ptx::smem_desc(base_s + kOffH + h * 16384u + off, 0, 1024),
                                  ptx::smem_desc(base_s + kOffQStage + h * kQHalf16 + off, 0, 1024), idesc_rot, kk > 0);
                }
                ptx::mma_commit(bar(ms.q_rot));
            }
            ok = ok && ptx::mbar_wait(bar(ms.q_full), 0, abort_flag, kWaitNs);
            int qk = 0, pv = 0;
            uint64_t idle_since = 0;
            unsigned idle_polls = 0;
            while (ok && pv < ntiles) {
                bool progressed = false;
                if (qk < ntiles && qk <= pv + kSBufs - 1 &&
                    ptx::mbar_test_wait(bar(ms.k_full[qk % kNK]), (qk / kNK) & 1) &&
                    ptx::mbar_test_wait(bar(ms.s_free[qk % kSBufs]), ((qk / kSBufs) & 1) ^ 1)) {
                    const int ks = qk % kNK, sb = qk % kSBufs;
                    ptx::tc_fence_after();
                    const uint32_t d = tmem + kColS0 + (uint32_t)sb * kSStride;
#if VA_Q8_ACC3
                    // the three q terms (48 K-major rows, 6 KB each) accumulated into one block
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int t = 0; t < 3; ++t)
                            asm volatile(
                                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                                " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
                                "l"(ptx::smem_desc(base_s + kOffK + ks * kStage + kk * 32, 0, 1024)),
                                "l"(ptx::smem_desc(base_s + kOffQ + t * kQTerm + kk * 32, 0, 1024)), "r"(idesc_qk),
                                "r"(kk > 0 || t > 0 ? 1u : 0u)
                                : "memory");
#else
                    // B = the three q terms as 144 consecutive K-major rows (each term 48 rows, 6 KB)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        asm volatile(
                            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                            " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
                            "l"(ptx::smem_desc(base_s + kOffK + ks * kStage + kk * 32, 0, 1024)),
                            "l"(ptx::smem_desc(base_s + kOffQ + kk * 32, 0, 1024)), "r"(idesc_qk),
                            "r"(kk > 0 ? 1u : 0u)
                            : "memory");
#endif
                    ptx::mma_commit(bar(ms.s_full[sb]));
                    ++qk;
                    progressed = true;
                }
                if (pv < qk && ptx::mbar_test_wait(bar(ms.p_full[pv & 1]), (pv >> 1) & 1)) {
                    const int i = pv, ps = i % kNK;
                    ptx::tc_fence_after();
                    const long long t = P.t0 + 2LL * i;
                    const int nk = (t + 1 < P.t1) ? 8 : 4;
                    const uint32_t v16 = base_s + kOffV16 + (uint32_t)(i & 1) * kV16;
                    for (int kk = 0; kk < nk; ++kk)
                        ptx::mma_bf16(tmem + kColO, ptx::smem_desc(v16 + kk * 2048, kV16Half, 1024),
                                      ptx::smem_desc(base_s + kOffK + ps * kStage + kk * 2048, 8192, 1024), idesc_pv,
                                      (i > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(bar(ms.pv_done[i & 1]));
                    ptx::mma_commit(bar(ms.k_empty[ps]));
                    if (i == ntiles - 1) ptx::mma_commit(bar(ms.o_ready));
                    ++pv;
                    progressed = true;
                }
                if (progressed) {
                    idle_since = 0;
                    idle_polls = 0;
                } else if (VA_POLL_EVERY <= 1 || ++idle_polls % VA_POLL_EVERY == 0) {
                    const uint64_t now = ptx::globaltimer_ns();
                    if (idle_since == 0) idle_since = now;
                    if (*abort_flag || now - idle_since > kWaitNs) ok = false;
                }
            }
            if (!ok) fail();
            ptx::mma_commit(bar(ms.drain));
            ptx::mbar_wait(bar(ms.drain), 0, nullptr, kWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax / widening warps
        const int sw = warp - kSoftWarp0;
        const int q = warp & 3;
        const int ch = sw >> 2;
        const int n0 = ch * kCols;
        const int L = q * 32 + lane;
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        bool ok = true;

        if (kAppend && fused_append) {
            // verify_attn_q8_step: softmax warp r codes live row r (key and value, the separate append's
            // encoder) if its position lies in this split's tiles; a row whose successor has the same
            // position is skipped, so the rows land as if written in row order.  The TMA loads of these
            // rows come after the proxy fence and the barrier.
            int pr = 0, pn = -1;
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r == sw) pr = row_pos[r];
                if (r == sw + 1 && r < a.n_live) pn = row_pos[r];
            }
            if (sw < a.n_live && pr >= P.t0 * kTile && pr < P.t1 * kTile && pn != pr) {
                const int slot = pr % a.slots;
                const uint2 kraw = __ldcg(reinterpret_cast<const uint2*>(a.k_new) + sw * 32 + lane);
                const uint2 vraw = __ldcg(reinterpret_cast<const uint2*>(a.v_new) + sw * 32 + lane);
                codec::code_key_row(kraw, lane, reinterpret_cast<uint8_t*>(const_cast<uint16_t*>(a.k)) + (size_t)slot * kD,
                                    const_cast<float*>(kscale_g) + slot);
                codec::code_value_row(vraw, lane, reinterpret_cast<int8_t*>(const_cast<uint16_t*>(a.v)) + (size_t)slot * kD,
                                      const_cast<float*>(vscale_g) + slot);
                ptx::fence_proxy_async_global();
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.app_done));
        }
        if (is_tree && warp == kSoftWarp0 && lane <= a.n_live) {   // the tree, for the row set-up
            if (lane == 0) ms.base = tree_word;
            else ms.anc[lane - 1] = tree_word;
        }
        __syncwarp();
        row_setup((warp - kSoftWarp0) * 32 + lane);   // published by the first barrier below
        // (H q)^T: thread L holds rotated element d' = L of rows n0 .. n0 + kCols - 1.  Per row, a power of two
        // s_r brings the largest element into [128, 256); the scaled row splits into three E4M3 terms.
        if (!ptx::mbar_wait(bar(ms.q_rot), 0, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        {
            float hq[kCols];
            tmem_ld_cols(tl + kColS0 + n0, hq);
            float m[kCols];
#pragma unroll
            for (int i = 0; i < kCols; ++i) m[i] = fabsf(hq[i]);
            warp_reduce_scatter<true>(m, lane);
            const int cb = n0 + scatter_col_base(lane);
            if (scatter_writer(lane)) {
                ms.red[q][cb] = m[0];
                ms.red[q][cb + 1] = m[1];
                ms.red[q][cb + 2] = m[2];
            }
            ptx::named_bar_sync(1, kSoftThreads);
            if (ch == 0 && L < kMaxM) {
                const float mx = fmaxf(fmaxf(ms.red[0][L], ms.red[1][L]), fmaxf(ms.red[2][L], ms.red[3][L]));
                // s_r = 2^(E - 8) for mx = f 2^E, f in [0.5, 1), from the exponent field (rows below 2^-119
                // are scaled as if they were 2^-119)
                const int ef = max(8, (int)((__float_as_uint(mx) >> 23) & 0xFFu));
                ms.qsig[L] = mx > 0.0f ? __uint_as_float((uint32_t)(ef - 7) << 23) : 1.0f;
                ms.qinv[L] = mx > 0.0f ? __uint_as_float((uint32_t)(261 - ef) << 23) : 1.0f;
            }
            ptx::named_bar_sync(1, kSoftThreads);
            // byte L of rows n, n + 1 in each term (K-major, 128-byte swizzle); two values per conversion
#pragma unroll
            for (int i = 0; i < kCols; i += 2) {
                const int n = n0 + i;
                float r0 = hq[i] * ms.qinv[n], r1 = hq[i + 1] * ms.qinv[n + 1];
                const uint32_t off0 = (uint32_t)(n >> 3) * 1024u + (uint32_t)(n & 7) * 128u +
                                      ((((uint32_t)L >> 4) ^ (uint32_t)(n & 7)) << 4) + ((uint32_t)L & 15u);
                const uint32_t off1 = (uint32_t)((n + 1) >> 3) * 1024u + (uint32_t)((n + 1) & 7) * 128u +
                                      ((((uint32_t)L >> 4) ^ (uint32_t)((n + 1) & 7)) << 4) + ((uint32_t)L & 15u);
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    const uint32_t c = e4m3x2(r0, r1);
                    base[kOffQ + t * kQTerm + off0] = (unsigned char)(c & 0xFFu);
                    base[kOffQ + t * kQTerm + off1] = (unsigned char)(c >> 8);
                    const float2 dq = e4m3x2_to_float2(c);
                    r0 -= dq.x;   // exact: the residual of a rounding to 4 significant bits
                    r1 -= dq.y;
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(ms.q_full));

        const float c0 = a.scale * 1.4426950408889634f * (1.0f / 128.0f);   // rotated-space scores in log2 units
        float cq[kCols], ref[kCols], l[kCols];
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
            cq[i] = c0 * ms.qsig[n0 + i];
            ref[i] = ms.ref[n0 + i];
            l[i] = 0.0f;
        }
        long long all_lo = own_lo, all_hi = own_hi;
        for (int r = 0; r < n_live_g; ++r) {
            all_lo = max(all_lo, ms.row_lo[r]);
            all_hi = min(all_hi, ms.row_hi[r]);
        }
        if (is_tree) all_hi = min(all_hi, ms.tree_base);   // the node region of a tree is never interior
        for (int j = 0; j < ntiles; ++j) {
            const long long t = P.t0 + 2LL * j;
            const int nkeys = (t + 1 < P.t1) ? 128 : 64;
            const long long kbase = t * kTile;
            const long long kp = kbase + L;
            const int sb = j % kSBufs, ks = j % kNK, vs = j % kNV;
            const bool own = L < nkeys && kp >= own_lo && kp < own_hi;
            // V: its scales, then its codes (key L, the d range of column part ch), widened to fp16 into the
            // buffer of this tile's parity once the PV two tiles back has read it; the code stage is free as
            // soon as the codes are in registers.  Keys outside the split's range keep the finite values their
            // stale codes widen to (every byte is an INT8 code) and get P' = 0 through a zero V scale (their p
            // is zero too).
            float sv;
            uint4 raw[kVChunks];
            auto read_v = [&]() {
                if (!ptx::mbar_wait(bar(ms.v_full[vs]), (j / kNV) & 1, abort_flag, kWaitNs)) ok = false;
                sv = own ? ms.vscale[vs][L] : 0.0f;
                const uint32_t roff = kOffV + (uint32_t)vs * kStage + (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u;
#pragma unroll
                for (int c = 0; c < kVChunks; ++c)
                    raw[c] = *reinterpret_cast<const uint4*>(
                        base + roff + (((uint32_t)(kVChunks * ch + c) ^ (uint32_t)(L & 7)) << 4));
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(ms.v_empty[vs]));
                if (j >= 2 && !ptx::mbar_wait(bar(ms.pv_done[j & 1]), ((j - 2) >> 1) & 1, abort_flag, kWaitNs)) ok = false;
            };
            auto widen = [&]() {
                // d = kVChunks * 16 * ch + 16 c + ...: d half (64 values, one 128-byte row per key) and the
                // 16-byte fp16 chunk inside it
                const int dh = (kVChunks * ch) >> 2, k0 = 2 * ((kVChunks * ch) & 3);
                const uint32_t woff = kOffV16 + (uint32_t)(j & 1) * kV16 + (uint32_t)dh * kV16Half +
                                      (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u;
#pragma unroll
                for (int c = 0; c < kVChunks; ++c) {
                    uint4 h0, h1;   // 16 codes -> two 16-byte chunks of 8 fp16 values
                    int8x4_to_half(raw[c].x, h0.x, h0.y);
                    int8x4_to_half(raw[c].y, h0.z, h0.w);
                    int8x4_to_half(raw[c].z, h1.x, h1.y);
                    int8x4_to_half(raw[c].w, h1.z, h1.w);
                    *reinterpret_cast<uint4*>(base + woff + (((uint32_t)(k0 + 2 * c) ^ (uint32_t)(L & 7)) << 4)) = h0;
                    *reinterpret_cast<uint4*>(base + woff + (((uint32_t)(k0 + 2 * c + 1) ^ (uint32_t)(L & 7)) << 4)) = h1;
                }
            };
            if (!VA_Q8_FUSE) {
                read_v();
                widen();
            }
            // which of the rows of this column part see key L (no score needed)
            const bool interior = kbase >= all_lo && kbase + nkeys <= all_hi;
            bool vis[kCols];
            {
                bool rv[kPartRows];
                if (interior) {
#pragma unroll
                    for (int k = 0; k < kPartRows; ++k) rv[k] = L < nkeys;
                } else {
                    const long long dk = kp - ms.tree_base;   // node index of key kp in a tree's node region
#pragma unroll
                    for (int k = 0; k < kPartRows; ++k) {
                        const int r = kPartRows * ch + k;
                        const bool in_mask = !is_tree || dk < 0 || (dk < 32 && ((ms.row_anc[r] >> (int)dk) & 1u));
                        rv[k] = (r < n_live_g) && kp >= ms.row_lo[r] && kp < ms.row_hi[r] && in_mask;
                    }
                }
#pragma unroll
                for (int i = 0; i < kCols; ++i) vis[i] = rv[i / kH];
            }
            if (!ptx::mbar_wait(bar(ms.s_full[sb]), (j / kSBufs) & 1, abort_flag, kWaitNs)) ok = false;
            ptx::tc_fence_after();
            float x[kCols];
            {   // the three terms' scores, added
                const uint32_t sc = tl + kColS0 + (uint32_t)sb * kSStride + n0;
                if (VA_Q8_ACC3) {
                    tmem_ld_cols(sc, x);
                } else if constexpr (kCols == 12) {   // all three terms in flight together: (x + y) + z
                    float y[kCols], z[kCols];
                    ptx::tmem_ld12x3_wait(sc, kTermCols, x, y, z);
#pragma unroll
                    for (int i = 0; i < kCols; i += 2) {
                        const float2 s2 = add2(add2(make_float2(x[i], x[i + 1]), make_float2(y[i], y[i + 1])),
                                               make_float2(z[i], z[i + 1]));
                        x[i] = s2.x;
                        x[i + 1] = s2.y;
                    }
                } else {
                    float y[kCols];
                    tmem_ld_cols(sc, x);
#pragma unroll
                    for (int t = 1; t < 3; ++t) {
                        tmem_ld_cols(sc + t * kTermCols, y);
#pragma unroll
                        for (int i = 0; i < kCols; i += 2) {
                            const float2 s2 = add2(make_float2(x[i], x[i + 1]), make_float2(y[i], y[i + 1]));
                            x[i] = s2.x;
                            x[i + 1] = s2.y;
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.s_free[sb]));
            const float sk = ms.kscale[ks][L];
#pragma unroll
            for (int i = 0; i < kCols; i += 2) {   // score = x * cq[i] in log2 units
                const float2 s2 = mul2(make_float2(x[i], x[i + 1]), make_float2(sk, sk));
                x[i] = s2.x;
                x[i + 1] = s2.y;
            }
            if (j == 0) {
                if (L == 0) {
#pragma unroll
                    for (int i = 0; i < kCols; ++i)
                        if (n0 + i < ML) ms.ref[n0 + i] = vis[i] ? x[i] * cq[i] : kRefInit;
                }
                ptx::named_bar_sync(1, kSoftThreads);
#pragma unroll
                for (int i = 0; i < kCols; ++i) ref[i] = ms.ref[n0 + i];
            }
            if (VA_Q8_FUSE) read_v();
            float p[kCols];
            float pmax = 0.0f;
#pragma unroll
            for (int i = 0; i < kCols; i += 2) {
                const float2 e2 = fma2(make_float2(x[i], x[i + 1]), make_float2(cq[i], cq[i + 1]),
                                       make_float2(-ref[i], -ref[i + 1]));
                p[i] = vis[i] ? ptx::ex2(e2.x) : 0.0f;
                p[i + 1] = vis[i + 1] ? ptx::ex2(e2.y) : 0.0f;
                pmax = fmaxf(pmax, fmaxf(p[i], p[i + 1]));
            }
            if (VA_Q8_FUSE) widen();
            // P' = p * v_scale as fp16, over this tile's K codes (QK(j) has read them)
            auto store_p = [&]() {
                uint32_t pw[kCols / 2];
#pragma unroll
                for (int i = 0; i < kCols / 2; ++i) {
                    const float2 s2 = mul2(make_float2(p[2 * i], p[2 * i + 1]), make_float2(sv, sv));
                    pw[i] = pack_half2(s2.x, s2.y);
                }
                const uint32_t roff = kOffK + (uint32_t)ks * kStage + (uint32_t)(L >> 3) * 1024u + (uint32_t)(L & 7) * 128u;
                if constexpr (kCols == 24) {   // 48 bytes from byte 48 ch: three 16-byte chunks
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const uint32_t off = roff + ((uint32_t)((3 * ch + k) ^ (L & 7)) << 4);
                        *reinterpret_cast<uint4*>(base + off) = make_uint4(pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3]);
                    }
                } else {   // 24 bytes from byte 24 ch: three 8-byte pieces
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const uint32_t b = 24u * (uint32_t)ch + 8u * (uint32_t)k;
                        const uint32_t off = roff + ((((b >> 4) ^ (uint32_t)(L & 7))) << 4) + (b & 15u);
                        *reinterpret_cast<uint2*>(base + off) = make_uint2(pw[2 * k], pw[2 * k + 1]);
                    }
                }
            };
            const unsigned want = __any_sync(0xffffffffu, !(pmax <= kThresh));
            if (lane == 0) {
                ms.vote[j & 1][sw] = want ? 1 : 0;
                if (VA_Q8_VOTE_MB) ptx::mbar_arrive(bar(ms.vote_bar[j & 1]));
            }
            if (VA_Q8_VOTE_MB) {
                store_p();
                if (!ptx::mbar_wait(bar(ms.vote_bar[j & 1]), (j >> 1) & 1, abort_flag, kWaitNs)) ok = false;
            } else {
                ptx::named_bar_sync(1, kSoftThreads);
            }
            int any = 0;
#pragma unroll
            for (int w = 0; w < kSoftWarps; ++w) any |= ms.vote[j & 1][w];
            if (any) {
                if (j > 0 && !ptx::mbar_wait(bar(ms.pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort_flag, kWaitNs))
                    ok = false;
                float v[kCols];
#pragma unroll
                for (int i = 0; i < kCols; ++i) v[i] = vis[i] ? x[i] * cq[i] : -INFINITY;
                warp_reduce_scatter<true>(v, lane);
                const int cb = n0 + scatter_col_base(lane);
                if (scatter_writer(lane)) {
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
#pragma unroll
                for (int i = 0; i < kCols; ++i) {
                    ref[i] = ms.ref[n0 + i];
                    l[i] *= ms.alpha[n0 + i];
                    p[i] = vis[i] ? ptx::ex2(fmaf(x[i], cq[i], -ref[i])) : 0.0f;
                }
                if (j > 0) {
                    ptx::tc_fence_after();
                    float o[kCols];
                    tmem_ld_cols(tl + kColO + n0, o);
#pragma unroll
                    for (int i = 0; i < kCols; ++i) o[i] *= ms.alpha[n0 + i];
                    tmem_st_cols(tl + kColO + n0, o);
                    ptx::tmem_wait_st();
                }
                if (VA_Q8_VOTE_MB) store_p();
            }
#pragma unroll
            for (int i = 0; i < kCols; i += 2) {
                const float2 s2 = add2(make_float2(l[i], l[i + 1]), make_float2(p[i], p[i + 1]));
                l[i] = s2.x;
                l[i + 1] = s2.y;
            }

            if (!VA_Q8_VOTE_MB) store_p();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(ms.p_full[j & 1]));
        }
        // ------------------------------------------------------------ epilogue
        warp_reduce_scatter<false>(l, lane);
        {
            const int cb = n0 + scatter_col_base(lane);
            if (scatter_writer(lane)) {
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
        float o[kCols];
        tmem_ld_cols(tl + kColO + n0, o);
#pragma unroll
        for (int i = 0; i < kCols; ++i) {
            const int n = n0 + i;
            if (n < M) part_o[n * kD + L] = o[i] * ms.inv_l[n];
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
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// [rows][128] uint8 codes, boxes of box_rows rows x 128 bytes with the 128-byte swizzle
bool encode_codes_map(CUtensorMap* map, const void* base, int rows, int box_rows) {
    tc::EncodeTiledFn fn = tc::encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace q8

cudaError_t launch_attn_q8(const AttnArgs& a, const float* k_scale, const float* v_scale, cudaStream_t stream) {
    if (a.n_groups < 1 || a.n_groups * kMaxRows < a.n_rows || (a.n_groups > 1 && !a.tree)) return cudaErrorInvalidValue;
    CUtensorMap tmq, tmk, tmv, tmk2, tmv2;
    const tc::MapEncodeFn rows = tc::encode_rows_map, codes = q8::encode_codes_map;
    if (!tc::cached_map(&tmq, rows, a.q, a.n_rows * kH, kMaxM) || !tc::cached_map(&tmk, codes, a.k, a.slots, 64) ||
        !tc::cached_map(&tmv, codes, a.v, a.slots, 64) || !tc::cached_map(&tmk2, codes, a.k, a.slots, 128) ||
        !tc::cached_map(&tmv2, codes, a.v, a.slots, 128))
        return cudaErrorInvalidValue;
    const bool append = a.k_new != nullptr;
    const bool tree = VA_TREE_TEMPLATE && a.tree != nullptr;
    const void* fn = append ? (const void*)q8::attn_q8_kernel<true, false>
                            : tree ? (const void*)q8::attn_q8_kernel<false, true> : (const void*)q8::attn_q8_kernel<false, false>;
    cudaError_t e = ensure_smem_attr(fn, (int)q8::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3(a.n_splits, a.n_groups), dim3(q8::kThreads), q8::kSmemBytes, stream);
    e = append ? cudaLaunchKernelEx(&cfg, q8::attn_q8_kernel<true, false>, a, k_scale, v_scale, tmq, tmk, tmv, tmk2, tmv2)
        : tree ? cudaLaunchKernelEx(&cfg, q8::attn_q8_kernel<false, true>, a, k_scale, v_scale, tmq, tmk, tmv, tmk2, tmv2)
               : cudaLaunchKernelEx(&cfg, q8::attn_q8_kernel<false, false>, a, k_scale, v_scale, tmq, tmk, tmv, tmk2, tmv2);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
