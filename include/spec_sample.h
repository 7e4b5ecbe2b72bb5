/*
 * spec_sample.h - C ABI of the steps that follow verification attention in a speculative round:
 * top-k / top-p sampling of the target's logits, rejection-sampling acceptance of a chain of drafts,
 * and acceptance plus cache settlement of a draft tree.  Same library, conventions and status codes
 * as verify_attn.h (every call asynchronous on `stream`, nothing allocated or synchronised, all
 * per-step values - tokens, counts, lengths - stay in device memory so that a step can be captured
 * in a CUDA graph).
 *
 * Sources:
 *   IQuestRT technical report, section "Include sampling and acceptance in the execution path":
 *     temperature 1, top-k 20, top-p 0.95 over a 160,000-token vocabulary; the draft keeps its
 *     actual proposal distribution q; a draft d is accepted with probability min(1, p(d)/q(d)); at
 *     the first rejection a replacement is drawn from normalise(max(0, p - q)); if every draft is
 *     accepted the target's extra row supplies a bonus token; acceptance, next-round input
 *     preparation and KV rollback belong to the decode step.
 *   the same report, section "Parallelize the Top-K vocabulary scan": logits in tiles of 8,192,
 *     candidates collected per tile in parallel, an ordered merge, tile maxima that let the merge
 *     skip tiles that cannot contribute.
 *   the same report, sections "IQuestRT execution" and "Keep the request loop on the GPU": tokens,
 *     acceptance counts and cache lengths stay on the device; the step settles the caches.
 *   "Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees".
 *
 * Definitions (where the pages leave a step open, the plainest reading):
 *   - candidate order: logit descending, equal logits by lower token id; NaN logits rank lowest;
 *   - the filtered distribution of a row: the top_k candidates, weights w_j = exp((l_j - l_0) / T),
 *     then the shortest prefix whose weight sum reaches top_p of the total (run / total >= top_p; the
 *     crossing candidate included), renormalised;
 *   - a draw with uniform u in [0, 1) from weights w_0..w_{n-1}: the first j whose running sum exceeds
 *     u * sum(w) (the last positive weight if rounding leaves none);
 *   - weights, running sums and these comparisons are float32 operations in candidate order (IEEE
 *     division, expf);
 *   - the acceptance test u < min(1, p/q) is evaluated exactly, as u * q < p (the sign of one fused
 *     multiply-add);
 *   - uniforms are inputs (device float arrays), so that the caller decides how they are generated
 *     (the pages derive them from the request seed and the token position).
 */
#ifndef SPEC_SAMPLE_H
#define SPEC_SAMPLE_H

#include "verify_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define VA_SAMPLE_MAX_K 32        /* largest top_k */
#define VA_SAMPLE_TILE 8192       /* logits per tile of the top-k scan */
#define VA_SAMPLE_MAX_VOCAB 262144 /* 32 tiles: the merge ranks at most 32 x 32 candidates */
#define VA_SAMPLE_MAX_ROWS 64       /* rows of one sampling call */
#define VA_SAMPLE_COUNTER_BYTES 256 /* the workspace's first bytes: one arrival counter per row */
#define VA_DEV_BAD_PATH 64        /* acceptance inputs that do not describe a valid draft / tree */

/*
 * va_sample_workspace_bytes - device workspace that va_sample_topk_topp needs for n_rows rows of
 * `vocab` logits.  Layout: the first VA_SAMPLE_COUNTER_BYTES hold one 32-bit arrival counter per row
 * (at the same place for every shape), then per row and 8,192-logit tile the top_k sorted candidates
 * (8 bytes each).  0 for arguments out of range.  Zero-fill a workspace once before its first use
 * (cudaMemsetAsync); every call leaves the counters at zero again, so one workspace sized for the
 * largest shape serves calls of any smaller (n_rows, vocab, top_k).  Calls that may run at the same
 * time need separate workspaces.
 */
VA_API size_t va_sample_workspace_bytes(int n_rows, int vocab, int top_k);

/*
 * va_sample_topk_topp - top-k / temperature / top-p sampling of n_rows rows of logits.
 *   logits        device float [n_rows][vocab] (16-byte aligned; vocab a multiple of 4)
 *   n_rows        1..VA_SAMPLE_MAX_ROWS (64)
 *   vocab         top_k .. VA_SAMPLE_MAX_VOCAB, a multiple of 4 (160,000 for this model)
 *   top_k         1..VA_SAMPLE_MAX_K (20 for this model)
 *   top_p         (0, 1] (0.95 for this model)
 *   temperature   > 0 (1 for this model)
 *   u             device float [n_rows]: the uniform of each row's draw, in [0, 1)
 *   ids           device int32 [n_rows][top_k]: the kept candidates in candidate order (-1 past count)
 *   probs         device float [n_rows][top_k]: their renormalised probabilities (0 past count)
 *   counts        device int32 [n_rows]: kept candidates per row (1..top_k)
 *   tokens        device int32 [n_rows]: the drawn token of each row
 *   workspace     device memory of va_sample_workspace_bytes(n_rows, vocab, top_k) bytes, 16-byte aligned
 * One launch: a CTA per (row, tile) collects the tile's candidates; the last CTA of a row to finish
 * merges them and draws.  Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
VA_API va_status va_sample_topk_topp(const float *logits, int n_rows, int vocab, int top_k, float top_p,
                                     float temperature, const float *u, int32_t *ids, float *probs,
                                     int32_t *counts, int32_t *tokens, void *workspace,
                                     size_t workspace_bytes, va_stream stream);

/*
 * va_accept_chain - rejection-sampling acceptance of a chain of drafts and the length update.
 * Verify row r (r = 0 .. n_drafts) took token drafts[r] as input (row 0: the committed token; rows
 * 1..n_drafts: the drafts) and produced the target's filtered distribution p_r (ids/probs/counts as
 * written by va_sample_topk_topp) and its own draw target_tokens[r].  Draft i was proposed from the
 * draft's filtered distribution q_i (q_ids/q_probs/q_counts row i; row 0 unused).
 * For i = 1, 2, ..: draft i is accepted iff u_accept[i] * q_i(d_i) < p_{i-1}(d_i); at the first
 * rejection the replacement is drawn with u_replace[0] from max(0, p_{i-1} - q_i) over p_{i-1}'s
 * candidates (from p_{i-1} itself if that is zero everywhere); if all n_drafts are accepted the bonus
 * token is target_tokens[n_drafts].
 *   k_stride      row stride (entries) of the ids / probs arrays (the top_k they were written with)
 *   n_accepted    device int32: the number of accepted drafts a (0 .. n_drafts)
 *   out_tokens    device int32 [n_drafts + 1]: the a accepted drafts, then the replacement or bonus
 *                 (entries past a + 1 are set to -1)
 *   pos           device int32: position of row 0 (the committed token)
 *   next_pos      optional device int32: pos + a + 1, the position of the next round's first row (for a
 *                 full-attention cache this is the whole rollback: rows past it are simply overwritten)
 * n_drafts 0..63.  Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
VA_API va_status va_accept_chain(const int32_t *p_ids, const float *p_probs, const int32_t *p_counts,
                                 const int32_t *q_ids, const float *q_probs, const int32_t *q_counts,
                                 int k_stride, const int32_t *drafts, const int32_t *target_tokens,
                                 int n_drafts, const float *u_accept, const float *u_replace,
                                 const int32_t *pos, int32_t *n_accepted, int32_t *out_tokens,
                                 int32_t *next_pos, va_stream stream);

/*
 * va_tree_accept_settle - acceptance of a draft tree and settlement of one layer's K/V cache.
 * The tree is the descriptor of verify_attn_tree (tree[0] = base, tree[1 + i] = ancestor-or-self mask
 * of node i; node i's parent is the highest-index ancestor other than itself).  Starting at the root,
 * the target's draw target_tokens[v] at node v selects the lowest-index child of v whose token
 * node_tokens[c] equals it; the walk stops at a node without such a child.  The accepted path
 * (root first) is then settled: the K/V rows of the node at depth d move from position base + node to
 * position base + d (slots taken modulo `slots`, so full caches and rings both work; all rows are read
 * before any is written).
 *   k_cache, v_cache  device [slots][128] bf16, updated in place (NULL: acceptance only)
 *   n_nodes       1..VA_MAX_TREE_NODES
 *   node_tokens   device int32 [n_nodes]: each node's token (node 0: the committed token)
 *   target_tokens device int32 [n_nodes]: the target's draw at each node (va_sample_topk_topp tokens)
 *   path          device int32 [n_nodes]: the accepted path, root first (-1 past its length)
 *   emitted       device int32 [n_nodes]: the emitted tokens - the accepted children's tokens, then the
 *                 target's token at the last node (-1 past the path length)
 *   n_accepted    device int32: path length - 1 (accepted draft nodes)
 *   next_pos      optional device int32: base + path length
 *   dev_status    optional device int32: VA_DEV_BAD_PATH if a mask is malformed (then nothing moves),
 *                 VA_DEV_NEGATIVE_POS if base < 0
 * Returns VA_OK, VA_INVALID_ARG or VA_CUDA_ERROR.
 */
VA_API va_status va_tree_accept_settle(va_bf16 *k_cache, va_bf16 *v_cache, int slots, const int32_t *tree,
                                       int n_nodes, const int32_t *node_tokens, const int32_t *target_tokens,
                                       int32_t *path, int32_t *emitted, int32_t *n_accepted, int32_t *next_pos,
                                       int32_t *dev_status, va_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_SAMPLE_H */
