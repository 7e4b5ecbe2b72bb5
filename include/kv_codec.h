/*
 * kv_codec.h - C ABI of the quantised K/V cache: keys FP8 (E4M3) after a Hadamard rotation, values INT8,
 * one fp32 scale per cached row, and verify attention read straight from it.
 * Source: "Qwen3.8-27B on one RTX 4090", section "A cheaper cache and state" (values INT8; keys FP8 after
 * a Hadamard rotation; verify attention gets faster too).  Conventions, status codes and the split
 * partials are those of verify_attn.h; attn_split_combine merges the partials unchanged.
 *
 * The codec (the plainest reading where the page is silent):
 *   keys     k' = H k with H the 128 x 128 Sylvester Hadamard matrix of +-1 entries (the butterfly
 *            (a, b) -> (a + b, a - b) in stages of width 1, 2, .., 64, float32); s_k = max|k'| / 448;
 *            code = E4M3(k' / s_k), round to nearest even, saturating (a zero result is coded +0)
 *   values   s_v = max|v| / 127; code = round-half-even(v / s_v), an int8 in [-127, 127]
 *   all-zero rows have scale 0 and codes 0; scale and quotient are float32 operations
 *   decoded  k^ = H (s_k code) / 128, v^ = s_v code: attention over the decoded cache.  Scores are formed
 *            in the rotated space, q . k^ = (H q) . (s_k code) / 128.
 * Cache layout: codes [slots][128] bytes (row = slot, position p in slot p mod slots), scales [slots]
 * fp32; slots a multiple of 64; 16-byte aligned buffers.  One position costs 264 bytes instead of 512.
 */
#ifndef KV_CODEC_H
#define KV_CODEC_H

#include "verify_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define VA_Q8_MAX_APPEND 16777216   /* rows one kv_ring_append_q8 call may encode */

/*
 * kv_ring_append_q8 - encode the live rows' new K and V and write them (codes and scales) to slot
 * pos[r] mod slots, before they are read.
 *   k_new, v_new  device [n_live][128] bf16
 *   n_live        0..VA_Q8_MAX_APPEND: the verify rows of a step, or a whole prefill history at once
 *   k_codes, v_codes  device uint8 / int8 [slots][128]; k_scale, v_scale device float [slots]
 *   slots         a multiple of 64 (else VA_UNSUPPORTED)
 *   pos           device int32 [>= n_live]; dev_status: VA_DEV_NEGATIVE_POS (the row is not written).
 *                 A row whose slot the next row also writes is skipped, so adjacent rows that share a slot
 *                 land as if written in row order (rows that share a slot must be adjacent).
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED or VA_CUDA_ERROR.
 */
VA_API va_status kv_ring_append_q8(const va_bf16 *k_new, const va_bf16 *v_new, int n_live, uint8_t *k_codes,
                                   int8_t *v_codes, float *k_scale, float *v_scale, int slots, const int32_t *pos,
                                   int32_t *dev_status, va_stream stream);

/*
 * verify_attn_q8 - split-KV verify attention over the quantised cache: full attention (window 0, the
 * cache indexed by position) or a sliding window (window W, a ring; slots >= W + n_live - 1).
 * Arguments as verify_attn_full / verify_attn_swa with the codes and scales in place of the bf16
 * cache; n_rows 1..8; n_splits 0 = va_auto_splits(slots or W + n_live - 1, window).
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED (slots % 64 != 0), VA_RING_TOO_SMALL or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_q8(const va_bf16 *q, int n_rows, int n_live, const uint8_t *k_codes,
                                const int8_t *v_codes, const float *k_scale, const float *v_scale, int slots,
                                int window, const int32_t *pos, float scale, int n_splits, float *part_o,
                                float *part_lse, int *splits_used, int32_t *dev_status, va_stream stream);

/*
 * verify_attn_q8_step - a whole verify call over the quantised cache in one call: verify_attn_q8 in which
 * the split that owns the live rows' positions first codes them into the cache (the same bytes as
 * kv_ring_append_q8 writes) and loads their tile after them, then attn_split_combine, on the stream in that
 * order (two launches, the second waiting for the first by programmatic dependent launch; capturable in a
 * CUDA graph).  Source as verify_attn_q8 and kv_ring_append_q8.  Positions the plan rejects (negative,
 * decreasing, beyond the cache or the ring) set their dev_status bits and code no row.
 *   q, n_rows, n_live, k_codes, v_codes, k_scale, v_scale, slots, window, pos, scale, n_splits
 *                 as verify_attn_q8 (the codes and scales are updated in place)
 *   k_new, v_new  device [n_live][128] bf16, 16-byte aligned: the live rows' new K and V
 *   sink          device float [6] or NULL, as attn_split_combine
 *   workspace     device float, 16-byte aligned, va_workspace_bytes(n_splits) bytes, laid out as for
 *                 verify_attn_step
 *   out, out_lse  as attn_split_combine (n_rows, n_live)
 *   splits_used   optional HOST int; dev_status optional device int32 (the bits of the two calls)
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_RING_TOO_SMALL or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_q8_step(const va_bf16 *q, const va_bf16 *k_new, const va_bf16 *v_new, int n_rows,
                                     int n_live, uint8_t *k_codes, int8_t *v_codes, float *k_scale, float *v_scale,
                                     int slots, int window, const int32_t *pos, const float *sink, float scale,
                                     int n_splits, float *workspace, va_bf16 *out, float *out_lse, int *splits_used,
                                     int32_t *dev_status, va_stream stream);

/*
 * verify_attn_q8_tree - verify attention of a draft TREE over the quantised cache.
 * Source: "Qwen3.8-27B on one RTX 4090": the 16-node verify trees of "More tokens per round: verify
 * trees" read the cache of "A cheaper cache and state".  The kernel is verify_attn_q8's with each node's
 * ancestor mask in place of the causal tail (the masks, extent and split plan of verify_attn_tree); up
 * to 16 nodes run as two groups of 8 rows.
 *   q, n_rows, n_nodes, window, tree, scale  as verify_attn_tree (n_rows 1..16; window 0 or >= n_nodes)
 *   k_codes, v_codes, k_scale, v_scale, slots  the quantised cache as for verify_attn_q8 (slots a
 *                 multiple of 64, else VA_UNSUPPORTED; window > 0: slots >= window + n_nodes - 1, else
 *                 VA_RING_TOO_SMALL).  Node i's codes sit at position base + i: append them first
 *                 (kv_ring_append_q8 with pos[i] = base + i, same stream).
 *   n_splits      1..VA_MAX_SPLITS, or 0 = auto (the ceil(n_rows / 8) node groups share the SMs)
 *   part_o, part_lse, splits_used, dev_status  as verify_attn_tree; merge with attn_split_combine
 * Returns VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_RING_TOO_SMALL or VA_CUDA_ERROR.
 */
VA_API va_status verify_attn_q8_tree(const va_bf16 *q, int n_rows, int n_nodes, const uint8_t *k_codes,
                                     const int8_t *v_codes, const float *k_scale, const float *v_scale, int slots,
                                     int window, const int32_t *tree, float scale, int n_splits, float *part_o,
                                     float *part_lse, int *splits_used, int32_t *dev_status, va_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* KV_CODEC_H */
