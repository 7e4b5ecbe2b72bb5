/*
 * verify_attn.h - C ABI of the GB300 (sm_103a) speculative-decoding verify-attention library.
 *
 * One rank's share of a decode step's verification attention: one KV head serves six query
 * heads (head_dim 128); up to eight verify rows (one committed token plus drafts, the rest
 * padding) are folded with the six heads into 48 matrix rows that share every K/V tile; the
 * history is partitioned along the sequence (split-KV) and the split partials are merged by a
 * separate log-sum-exp combine.
 *   Source: IQuestRT technical report, sections "Read only the KV tiles needed by the current
 *   positions" (48-row folding, sequence partition, valid extent, causal boundary, zero-value
 *   sink, separate combine, sliding-window ring of the window plus one 64-slot tile written
 *   before it is read) and "Expose more parallelism in attention" (split-KV partials merged with
 *   their log-sum-exp values, sink correction inside the combine).
 *
 * Conventions shared by every call
 *   - bf16 data is passed as raw bit patterns (va_bf16).  All tensors are dense, row-major and
 *     contiguous; every pointer named "device" must be a CUDA device (or managed) address.  The
 *     q, K/V, new-row, partial and output buffers must be 16-byte aligned (VA_INVALID_ARG
 *     otherwise); pos, sink, out_lse and dev_status need only their element alignment.
 *   - Positions are 0-based absolute token positions, int32, in DEVICE memory so that a call can
 *     be captured in a CUDA graph.  Verify row r sits at pos[r]; rows r < n_live are live; the
 *     remaining rows up to n_rows are padding: their outputs are exactly 0 and their LSEs -inf.
 *     Live positions must be non-decreasing (consecutive for a chain of drafts).
 *   - A row at position p sees keys j <= p (full attention) or p - window < j <= p (sliding
 *     window).  The read extent is [lo, hi) with hi = pos[n_live-1] + 1 and lo = 0 (full) or
 *     max(0, pos[0] - window + 1) (sliding window): capacity beyond it is never read.
 *   - Matrix row m = r * 6 + h (row r, query head h), i.e. q's own [n_rows][6][128] order.
 *   - Sequence splits: 64-position tiles aligned to absolute position.  With t_lo = lo / 64,
 *     t_hi = ceil(hi / 64) - 1 and T = t_hi - t_lo + 1, split s owns tiles
 *     [t_lo + floor(s*T/S), t_lo + floor((s+1)*T/S)).  Splits that own no tile (S > T) write
 *     o = 0 and lse = -inf.
 *   - Ownership: the caller owns all memory; no call allocates, frees or synchronizes.  Every
 *     call is asynchronous on `stream` (NULL = the legacy default stream); calls on one stream
 *     run in order, which is what puts a ring append before the reads that need it.
 *   - Errors: each call returns a va_status and launches nothing unless it returns VA_OK.
 *     VA_CUDA_ERROR means a CUDA launch error was reported (cudaGetLastError).  Errors that
 *     depend on device-resident positions are reported through the optional device word
 *     `dev_status` (bits VA_DEV_*, OR-ed in; the caller clears it); the affected call then
 *     writes empty partials.  No kernel traps, asserts or spins.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define VA_API __attribute__((visibility("default")))
#else
#define VA_API
#endif

typedef uint16_t va_bf16;               /* raw bfloat16 bits */
typedef struct CUstream_st *va_stream;  /* the same type as cudaStream_t */
typedef int va_status;

#define VA_OK 0
#define VA_INVALID_ARG 1      /* null pointer, size out of range, non-finite scale ... */
#define VA_UNSUPPORTED 2      /* a shape this library is not built for (ring_slots % 64 != 0) */
#define VA_RING_TOO_SMALL 3   /* ring_slots < window + n_live - 1: appends would evict history */
#define VA_CUDA_ERROR 4       /* a CUDA error was reported when launching */

#define VA_HEAD_DIM 128       /* head dimension d */
#define VA_Q_HEADS 6          /* query heads per KV head */
#define VA_MAX_ROWS 8         /* verify rows per call (one committed token + up to 7 drafts) */
#define VA_MAX_TREE_NODES 16  /* nodes of a draft tree per verify_attn_tree call */
#define VA_TILE 64            /* positions per K/V tile and split granule */
#define VA_MAX_SPLITS 4096    /* largest accepted split count */

/* device status bits (dev_status) */
#define VA_DEV_NEGATIVE_POS 1     /* a live position is < 0 */
#define VA_DEV_NOT_MONOTONE 2     /* live positions decrease */
#define VA_DEV_BEYOND_CACHE 4     /* full attention: pos[n_live-1] >= capacity */
#define VA_DEV_RING_SPAN 8        /* sliding window: pos[n_live-1] - pos[0] > ring_slots - window */
#define VA_DEV_TIMEOUT 16         /* a kernel gave up on a bounded wait; its outputs are not valid */
#define VA_DEV_TREE_MASK 32       /* a tree mask lacks its own node's bit or names a node >= n_nodes */

/*
 * kv_ring_append - write the live rows' new K and V into the cache before they are read.
 * Source: IQuestRT report, "Read only the KV tiles needed by the current positions" (the
 * sliding-window ring; verification writes its KV rows before reading them) and "Let correctness
 * checks change the design" (ring of window + one 64-slot tile).
 *   k_new, v_new  device [n_live][128] bf16: the new rows, row r for position pos[r]
 *   n_live        0..16 (0: nothing is written; up to 16 for the nodes of a draft tree)
 *   k_cache, v_cache  device [slots][128] bf16, updated in place
 *   slots         rows of the cache: the ring size for a sliding-window layer, the capacity for a
 *                 full-attention layer; row r goes to slot pos[r] mod slots
 *   pos           device int32 [>= n_live]
 *   dev_status    optional device int32 (NULL = none): VA_DEV_NEGATIVE_POS for a negative
 *                 position, whose row is then not written
 * Returns VA_OK, VA_INVALID_ARG (null pointers with n_live > 0, n_live outside 0..8,
 * slots < 1) or VA_CUDA_ERROR.
 */
VA_API va_status kv_ring_append(const va_bf16 *k_new, const va_bf16 *v_new, int n_live,
                         va_bf16 *k_cache, va_bf16 *v_cache, int slots,
                         const int32_t *pos, int32_t *dev_status, va_stream stream);

/*
 * verify_attn_full - split-KV verify attention of a full-attention layer.
 * Source: IQuestRT report, "Read only the KV tiles needed by the current positions" (48 matrix
 * rows, sequence partition, read extent from the current positions, causal mask at the
 * boundary) and "Expose more parallelism in attention" (partials carry their LSE).
 *   q             device [n_rows][6][128] bf16
 *   n_rows        1..8; n_live 0..n_rows
 *   k_cache, v_cache  device [capacity][128] bf16; row j holds absolute position j.  Rows at and
 *                 beyond the extent are never read (they may hold anything, NaN included).
 *   pos           device int32 [n_rows]
 *   scale         softmax scale applied to q.k (finite; 1/sqrt(128) for this model)
 *   n_splits      1..VA_MAX_SPLITS, or 0 = va_auto_splits(capacity, 0)
 *   part_o        device float [n_splits][n_rows][6][128]: per split sum_j exp(s_j - lse_s) v_j
 *                 (0 where the split sees nothing)
 *   part_lse      device float [n_splits][n_rows][6]: per split ln sum_j exp(s_j) (natural log,
 *                 post-scale scores; -inf where the split sees nothing).  No sink here.
 *   splits_used   optional HOST int (NULL = none): receives the split count launched
 *   dev_status    optional device int32: VA_DEV_NEGATIVE_POS / NOT_MONOTONE / BEYOND_CACHE
 * Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_full(const va_bf16 *q, int n_rows, int n_live,
                           const va_bf16 *k_cache, const va_bf16 *v_cache, int capacity,
                           const int32_t *pos, float scale, int n_splits,
                           float *part_o, float *part_lse, int *splits_used,
                           int32_t *dev_status, va_stream stream);

/*
 * verify_attn_swa - split-KV verify attention of a sliding-window layer read from its ring.
 * Source: IQuestRT report, "Read only the KV tiles needed by the current positions" (separate
 * sliding-window path; ring of the window plus one 64-slot tile; every live row sees its
 * complete window).  Call kv_ring_append for the same rows first, on the same stream.
 *   As verify_attn_full, except:
 *   k_ring, v_ring  device [ring_slots][128] bf16; position p lives in slot p mod ring_slots
 *   ring_slots    a multiple of 64 (else VA_UNSUPPORTED), at least window + n_live - 1 (else
 *                 VA_RING_TOO_SMALL); 4,160 for a 4,096 window
 *   window        W >= 1: a row at p sees positions max(0, p - W + 1) .. p
 *   n_splits      0 = va_auto_splits(window + n_live - 1, window)
 *   dev_status    also VA_DEV_RING_SPAN if pos[n_live-1] - pos[0] > ring_slots - window
 */
VA_API va_status verify_attn_swa(const va_bf16 *q, int n_rows, int n_live,
                          const va_bf16 *k_ring, const va_bf16 *v_ring, int ring_slots, int window,
                          const int32_t *pos, float scale, int n_splits,
                          float *part_o, float *part_lse, int *splits_used,
                          int32_t *dev_status, va_stream stream);

/*
 * verify_attn_tree - split-KV verify attention of a draft TREE under its tree attention mask.
 * Source: "Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees" (the drafts
 * are grown best-first into a 16-node tree that the target verifies in one pass with a tree
 * attention mask).  The kernel is the verify_attn_full / verify_attn_swa split kernel with each
 * node's ancestor mask in place of the causal tail; up to 16 nodes run as two groups of 8 rows.
 *   q             device [n_rows][6][128] bf16, row i = node i
 *   n_rows        1..16; n_nodes 0..n_rows (rows past n_nodes are padding: 0 / -inf)
 *   k_cache, v_cache, slots   window == 0: the full-attention cache [capacity][128] (row j holds
 *                 position j); window > 0: the sliding-window ring (position p in slot p mod slots;
 *                 slots a multiple of 64 (else VA_UNSUPPORTED) and >= window + n_nodes - 1 (else
 *                 VA_RING_TOO_SMALL)).  Node i's K/V sit at position base + i: append them first
 *                 (kv_ring_append with pos[i] = base + i, same stream).
 *   window        0 (full attention) or W >= n_nodes (smaller windows: VA_UNSUPPORTED)
 *   tree          device int32 [1 + n_nodes]: tree[0] = base, the position of node 0 (the committed
 *                 prefix is positions 0 .. base - 1); tree[1 + i] = ancestor-or-self mask of node i:
 *                 bit k set iff node k is node i or one of its ancestors
 *   Node i at depth d_i = popcount(mask_i) - 1 has logical position base + d_i and sees the prefix
 *   positions max(0, base + d_i - W + 1) .. base - 1 (all of them for full attention) and the
 *   positions base + k of the nodes k in its mask.  Read extent: [lo, base + n_nodes) with lo = 0
 *   (full) or max(0, base + min_i d_i - W + 1); splits are dealt over it as for the chain calls.
 *   scale         as verify_attn_full
 *   n_splits      1..VA_MAX_SPLITS, or 0 = auto (the ceil(n_rows / 8) node groups share the SMs)
 *   part_o, part_lse  device float [n_splits][n_rows][6][128] / [n_splits][n_rows][6], as for
 *                 verify_attn_full; merge them with attn_split_combine (n_rows, n_live = n_nodes)
 *   splits_used   optional HOST int: the split count launched
 *   dev_status    optional device int32: VA_DEV_NEGATIVE_POS (base < 0), VA_DEV_BEYOND_CACHE
 *                 (full: base + n_nodes > capacity), VA_DEV_RING_SPAN (window: the extent is longer
 *                 than the ring), VA_DEV_TREE_MASK (a mask without its own bit, or naming a node
 *                 >= n_nodes); the call then writes empty partials
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_RING_TOO_SMALL or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_tree(const va_bf16 *q, int n_rows, int n_nodes,
                           const va_bf16 *k_cache, const va_bf16 *v_cache, int slots, int window,
                           const int32_t *tree, float scale, int n_splits,
                           float *part_o, float *part_lse, int *splits_used,
                           int32_t *dev_status, va_stream stream);

/*
 * attn_split_combine - merge split partials by log-sum-exp and fold in the learned sink.
 * Source: IQuestRT report, "Read only the KV tiles needed by the current positions" (a separate
 * combine kernel issues the partial loads together and keeps four independent FP32
 * accumulation chains) and "Expose more parallelism in attention" (the combine applies the
 * sink correction and keeps the BF16 rounding boundaries).
 *   part_o, part_lse  device, as written by verify_attn_full / verify_attn_swa
 *   n_splits      0..VA_MAX_SPLITS
 *   sink          device float [6] (NULL = no sink): logit of a zero-value key, post-scale
 *   n_rows, n_live as for the attention call (n_rows up to 16 after verify_attn_tree)
 *   out           device [n_rows][6][128] bf16: sum_s exp(lse_s - L) o_s rounded once to bf16
 *                 (nearest, ties to even), L = logsumexp({lse_s} U {sink_h}); padding rows 0
 *   out_lse       optional device float [n_rows][6]: L (-inf for padding rows)
 * Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
VA_API va_status attn_split_combine(const float *part_o, const float *part_lse, int n_splits,
                             const float *sink, int n_rows, int n_live,
                             va_bf16 *out, float *out_lse, va_stream stream);

/* Bytes of one workspace holding part_o followed by part_lse for n_splits splits and 8 rows
 * (part_lse then starts at n_splits * 8 * 6 * 128 floats).  0 if n_splits is out of range. */
VA_API size_t va_workspace_bytes(int n_splits);

/* Split count for a call whose extent is about extent_hint positions (window > 0: sliding
 * window layer), chosen for the current device's SM count.  Host only; never launches. */
VA_API int va_auto_splits(int extent_hint, int window);

/* The same policy for an explicit SM count (no device query; usable without a GPU). */
VA_API int va_auto_splits_for(int extent_hint, int window, int sm_count);

/* Name of a va_status value. */
VA_API const char *va_status_string(va_status status);

/*
 * verify_attn_step - one whole verify call: the append of the live rows, the split attention of a
 * full-attention or sliding-window layer and the combine with the sink, in two launches instead of the
 * three of kv_ring_append + verify_attn_full / verify_attn_swa + attn_split_combine (the append runs
 * inside the attention launch).  It computes exactly what those three calls compute.
 * Source: IQuestRT report, "Read only the KV tiles needed by the current positions" (append before read,
 * split-KV partials, separate combine) and "Expose more parallelism in attention" (LSE merge, sink
 * correction, bf16 rounding once).
 * The split that owns a live row's position writes that row to its slot before it loads the row's tile;
 * no other split reads it (in a ring, a stale row of the same slot lies below every window).
 *   q, n_rows, n_live, pos, scale   as verify_attn_full
 *   k_new, v_new  device [n_live][128] bf16 (may be NULL when n_live == 0), as kv_ring_append
 *   k_cache, v_cache, slots, window  window == 0: the full-attention cache, slots = capacity (row j holds
 *                 position j); window >= 1: the ring of a sliding-window layer, as verify_attn_swa
 *                 (slots a multiple of 64 (else VA_UNSUPPORTED), >= window + n_live - 1 (else
 *                 VA_RING_TOO_SMALL)).  Updated in place.
 *   sink          device float [6] or NULL, as attn_split_combine
 *   n_splits      1..VA_MAX_SPLITS, or 0 = auto (as verify_attn_full / verify_attn_swa)
 *   workspace     device float, 16-byte aligned, va_workspace_bytes(n_splits) bytes: part_o then
 *                 part_lse (at n_splits * 8 * 6 * 128 floats), laid out as verify_attn_full's partials
 *                 for n_rows rows; they stay there after the call
 *   out, out_lse  as attn_split_combine (n_rows, n_live)
 *   splits_used   optional HOST int: the split count launched
 *   dev_status    optional device int32: the bits of verify_attn_full / verify_attn_swa
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_RING_TOO_SMALL or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_step(const va_bf16 *q, const va_bf16 *k_new, const va_bf16 *v_new,
                                  int n_rows, int n_live, va_bf16 *k_cache, va_bf16 *v_cache, int slots,
                                  int window, const int32_t *pos, const float *sink, float scale,
                                  int n_splits, float *workspace, va_bf16 *out, float *out_lse,
                                  int *splits_used, int32_t *dev_status, va_stream stream);

/*
 * verify_attn_full_noalloc - verify_attn_full followed by attn_split_combine, with the split partials
 * kept in a fixed device buffer owned by this library, so that the caller allocates nothing.
 * The pages have no counterpart to this entry point.  It is for callers that cannot allocate device
 * memory when they call this library - a decode loop embedded in another runtime that hands it only
 * tensors and a stream (and no allocator), or a latency-critical loop that must not call cudaMalloc
 * because cudaMalloc can synchronise the device - and therefore cannot provide the part_o / part_lse
 * workspace that verify_attn_full needs.
 *   Scratch: a file-scope device array of VA_NOALLOC_MAX_SPLITS x 8 x 6 x 129 floats (3.96 MB) for the
 *   partials, held in the memory of every GPU that loads this library's device code until the process
 *   exits.  The first call on a device looks up that array's device address (cudaGetSymbolAddress, with
 *   that device current); make that first call before any stream capture.  Every call reuses the same
 *   array and overwrites it completely, so calls that may overlap on the GPU (unordered streams, several
 *   host threads) race with each other: the caller must order them.
 *   Arguments as verify_attn_full (q, n_rows, n_live, k_cache, v_cache, capacity, pos, scale, n_splits,
 *   splits_used, dev_status) and attn_split_combine (sink, out, out_lse).  n_splits 0 means
 *   va_auto_splits(capacity, 0) capped at VA_NOALLOC_MAX_SPLITS; an explicit count above
 *   VA_NOALLOC_MAX_SPLITS returns VA_INVALID_ARG.
 *   Allocates and frees nothing.  Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
#define VA_NOALLOC_MAX_SPLITS 160
VA_API va_status verify_attn_full_noalloc(const va_bf16 *q, int n_rows, int n_live,
                                          const va_bf16 *k_cache, const va_bf16 *v_cache, int capacity,
                                          const int32_t *pos, float scale, int n_splits,
                                          const float *sink, va_bf16 *out, float *out_lse,
                                          int *splits_used, int32_t *dev_status, va_stream stream);

/*
 * va_selftest_bounded_wait - failure detection without a fault.  Every wait in the library's kernels
 * (on a TMA arrival, an MMA completion, another warp) gives up after a time limit, or at once when a
 * warp of the same CTA has raised the CTA's abort flag, and reports VA_DEV_TIMEOUT.  This call runs that
 * wait routine on a shared-memory barrier that nothing completes (one CTA of 64 threads).
 *   limit_ns        1 .. VA_SELFTEST_MAX_WAIT_NS: the wait's limit
 *   abort_after_ns  0 (no abort) or <= limit_ns: a second warp raises the abort flag after this long
 *   dev_status      optional device int32: VA_DEV_TIMEOUT is OR-ed in when the wait gives up
 *   elapsed_ns      optional device uint64: how long the wait lasted (globaltimer)
 * Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.  The context stays usable afterwards.
 */
#define VA_SELFTEST_MAX_WAIT_NS 1000000000ull
VA_API va_status va_selftest_bounded_wait(unsigned long long limit_ns, unsigned long long abort_after_ns,
                                          int32_t *dev_status, unsigned long long *elapsed_ns, va_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
