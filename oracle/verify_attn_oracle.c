/*
 * FP64 CPU oracle for speculative-decoding verify attention.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline / reference arm may load this library.  It
 * shares no source, header, table or helper with the CUDA library.
 *
 * What it computes (IQuestRT technical report, section "Read only the KV tiles
 * needed by the current positions"; vLLM notes in the same report, section
 * "Expose more parallelism in attention"):
 *
 *   one KV head shared by 6 query heads, head_dim 128; verify row r at absolute
 *   (0-based) position pos[r]; the live rows r < n_live are computed, padding
 *   rows produce a zero output and an LSE of -inf.
 *
 *   visible set of row r:   full attention   { j : 0 <= j <= pos[r] }
 *                           sliding window W { j : max(0, pos[r]-W+1) <= j <= pos[r] }
 *   score                   s_j = scale * sum_d q[r,h,d] * K[j,d]
 *   learned sink            a logit sink_h in the same (post-scale) domain whose
 *                           value vector is zero: it enters the denominator only
 *   result                  M   = max(max_j s_j, sink_h)
 *                           Z   = exp(sink_h - M) + sum_j exp(s_j - M)
 *                           out = sum_j exp(s_j - M) V[j] / Z
 *                           LSE = M + ln Z
 *
 *   split partials (sequence partition, merged by log-sum-exp): for a position
 *   range [a, b) the partial over the visible keys inside it is
 *                           lse_s = ln sum_j exp(s_j)          (-inf if empty)
 *                           o_s   = sum_j exp(s_j - lse_s) V[j] (0 if empty)
 *   The ranges themselves are an input here; the oracle's Python side derives
 *   them from the 64-position tile plan.
 *
 *   combine (separate merge step): L = logsumexp({lse_s} U {sink_h}),
 *                           out = sum_s exp(lse_s - L) o_s.
 *
 * Inputs are the bf16 bit patterns of q and of the LINEAR history K/V indexed
 * by absolute position (never a ring), widened exactly to double.  Everything
 * is computed in double with plain loops; threads only split the independent
 * (row, head) pairs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 128
#define OR_H 6

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *kh, *vh;
    int64_t ctx;
    const int32_t *pos;
    int n_rows, n_live;
    const double *sink; /* may be NULL: no sink */
    double scale;
    int64_t window;     /* 0: full attention */
    const int32_t *tree; /* NULL, or tree verify: tree[0] = base slot, tree[1 + r] = ancestor mask of node r */
    const double *kd, *vd; /* NULL, or the history given as doubles (a decoded quantised cache) */
    int n_splits;
    const int64_t *split_a, *split_b; /* [n_splits] position ranges, may be NULL if n_splits == 0 */
    double *out, *lse, *part_o, *part_lse;
    int next_pair;      /* work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

/* Element d of the key / value at absolute position j: bf16 history widened exactly, or the given doubles. */
static double key_at(const job_t *J, int64_t j, int d)
{
    return J->kd ? J->kd[j * OR_D + d] : widen_bf16(J->kh[j * OR_D + d]);
}

static double value_at(const job_t *J, int64_t j, int d)
{
    return J->vd ? J->vd[j * OR_D + d] : widen_bf16(J->vh[j * OR_D + d]);
}

/* Depth of a tree node: the number of its strict ancestors (bits of its mask other than its own). */
static int tree_depth(int32_t mask)
{
    int n = 0;
    for (int b = 0; b < 31; ++b) n += (mask >> b) & 1;
    return n - 1;
}

/* First prefix position a row may see: 0 for full attention, else the start of its window.  A tree
 * node's window ends at its own logical position base + depth (the slot index of the node plays no part). */
static int64_t row_first(const job_t *J, int r)
{
    if (J->window <= 0) return 0;
    const int64_t p = J->tree ? (int64_t)J->tree[0] + tree_depth(J->tree[1 + r]) : (int64_t)J->pos[r];
    return p - J->window + 1 > 0 ? p - J->window + 1 : 0;
}

/* Is key j visible to row r?  Plain definitions:
 *   chain:  row_first(r) <= j <= pos[r];
 *   tree:   row_first(r) <= j < base (the committed prefix), or j = base + i where bit i of node r's
 *           ancestor-or-self mask is set and, with a window W, node i lies inside node r's window
 *           (depth_i >= depth_r - W + 1: ancestors are ordered by their logical positions). */
static int visible(const job_t *J, int r, int64_t j)
{
    if (J->tree) {
        const int64_t base = J->tree[0];
        if (j < 0) return 0;
        if (j < base) return j >= row_first(J, r);
        const int64_t i = j - base;
        if (i >= J->n_live || !((J->tree[1 + r] >> i) & 1)) return 0;
        return J->window <= 0 || tree_depth(J->tree[1 + i]) >= tree_depth(J->tree[1 + r]) - J->window + 1;
    }
    return j >= row_first(J, r) && j <= J->pos[r];
}

/* Attention of one live (row, head) pair over its whole visible set.  The keys considered are the
 * contiguous range [first, p]; keys in it that are not visible get no weight. */
static void one_pair(job_t *J, int r, int h, double *scores)
{
    int64_t first = row_first(J, r);
    if (J->tree && first > J->tree[0]) first = J->tree[0];   /* node slots are decided by visible() alone */
    const int64_t p = J->pos[r];   /* tree: base + n_nodes - 1, the last slot any node may see */
    const int64_t n = p - first + 1;
    double qd[OR_D];
    for (int d = 0; d < OR_D; ++d)
        qd[d] = widen_bf16(J->q[((int64_t)r * OR_H + h) * OR_D + d]);

    for (int64_t i = 0; i < n; ++i) {
        if (!visible(J, r, first + i)) {
            scores[i] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int d = 0; d < OR_D; ++d)
            acc += qd[d] * key_at(J, first + i, d);
        scores[i] = J->scale * acc;
    }

    const double sink = J->sink ? J->sink[h] : -INFINITY;
    double M = sink;
    for (int64_t i = 0; i < n; ++i)
        if (scores[i] > M) M = scores[i];

    double *o = J->out + ((int64_t)r * OR_H + h) * OR_D;
    double Z = 0.0;
    double acc[OR_D];
    for (int d = 0; d < OR_D; ++d) acc[d] = 0.0;
    if (M == -INFINITY) {
        /* nothing visible and no sink: defined as a zero output, LSE -inf */
        for (int d = 0; d < OR_D; ++d) o[d] = 0.0;
        J->lse[r * OR_H + h] = -INFINITY;
    } else {
        Z = exp(sink - M);
        for (int64_t i = 0; i < n; ++i) {
            if (scores[i] == -INFINITY) continue;
            const double w = exp(scores[i] - M);
            Z += w;
            for (int d = 0; d < OR_D; ++d)
                acc[d] += w * value_at(J, first + i, d);
        }
        for (int d = 0; d < OR_D; ++d) o[d] = acc[d] / Z;
        J->lse[r * OR_H + h] = M + log(Z);
    }

    /* split partials: same scores, restricted to each split's position range */
    for (int s = 0; s < J->n_splits; ++s) {
        const int64_t a = J->split_a[s] > first ? J->split_a[s] : first;
        const int64_t b = J->split_b[s] < p + 1 ? J->split_b[s] : p + 1;
        double *po = J->part_o + (((int64_t)s * J->n_rows + r) * OR_H + h) * OR_D;
        double *pl = J->part_lse + ((int64_t)s * J->n_rows + r) * OR_H + h;
        if (b <= a) {
            for (int d = 0; d < OR_D; ++d) po[d] = 0.0;
            *pl = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = a; j < b; ++j)
            if (scores[j - first] > m) m = scores[j - first];
        if (m == -INFINITY) {   /* nothing of this split is visible to the row */
            for (int d = 0; d < OR_D; ++d) po[d] = 0.0;
            *pl = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int d = 0; d < OR_D; ++d) acc[d] = 0.0;
        for (int64_t j = a; j < b; ++j) {
            if (scores[j - first] == -INFINITY) continue;
            const double w = exp(scores[j - first] - m);
            z += w;
            for (int d = 0; d < OR_D; ++d)
                acc[d] += w * value_at(J, j, d);
        }
        /* o_s = sum exp(s_j - lse_s) v_j with lse_s = m + ln z */
        for (int d = 0; d < OR_D; ++d) po[d] = acc[d] / z;
        *pl = m + log(z);
    }
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int64_t longest = 0;
    for (int r = 0; r < J->n_live; ++r)
        if ((int64_t)J->pos[r] + 1 > longest) longest = (int64_t)J->pos[r] + 1;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(longest > 0 ? longest : 1));
    if (!scores) return (void *)1;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int pair = J->next_pair++;
        pthread_mutex_unlock(&J->mu);
        if (pair >= J->n_live * OR_H) break;
        one_pair(J, pair / OR_H, pair % OR_H, scores);
    }
    free(scores);
    return NULL;
}

/*
 * Verify attention over the linear history.
 *   q        [n_rows][6][128] bf16 bits
 *   kh, vh   [ctx][128] bf16 bits, row j holds absolute position j
 *   pos      [n_rows] 0-based positions; live rows must satisfy 0 <= pos[r] < ctx
 *   sink     [6] logits or NULL (no sink)
 *   window   0 for full attention, else the sliding-window length W
 *   split_a/split_b [n_splits] position ranges of the partials (n_splits may be 0)
 *   out      [n_rows][6][128], lse [n_rows][6]
 *   part_o   [n_splits][n_rows][6][128], part_lse [n_splits][n_rows][6]
 * Returns 0, or -1 on invalid arguments, -2 on allocation failure.
 */
static int run(const uint16_t *q, const uint16_t *kh, const uint16_t *vh, const double *kd, const double *vd,
               int64_t ctx, const int32_t *pos, int n_rows, int n_live, const double *sink, double scale,
               int64_t window, const int32_t *tree, int n_splits, const int64_t *split_a, const int64_t *split_b,
               double *out, double *lse, double *part_o, double *part_lse, int n_threads);

int oracle_verify_attn(const uint16_t *q, const uint16_t *kh, const uint16_t *vh, int64_t ctx,
                       const int32_t *pos, int n_rows, int n_live, const double *sink,
                       double scale, int64_t window, int n_splits, const int64_t *split_a,
                       const int64_t *split_b, double *out, double *lse, double *part_o,
                       double *part_lse, int n_threads)
{
    return run(q, kh, vh, NULL, NULL, ctx, pos, n_rows, n_live, sink, scale, window, NULL, n_splits, split_a,
               split_b, out, lse, part_o, part_lse, n_threads);
}

/*
 * The same attention over a history given as doubles (kd, vd [ctx][128]): the keys and values a
 * quantised cache decodes to (see oracle/kv_codec.py).  Other arguments as oracle_verify_attn.
 */
int oracle_verify_attn_f64kv(const uint16_t *q, const double *kd, const double *vd, int64_t ctx,
                             const int32_t *pos, int n_rows, int n_live, const double *sink, double scale,
                             int64_t window, int n_splits, const int64_t *split_a, const int64_t *split_b,
                             double *out, double *lse, double *part_o, double *part_lse, int n_threads)
{
    if (!kd || !vd) return -1;
    return run(q, NULL, NULL, kd, vd, ctx, pos, n_rows, n_live, sink, scale, window, NULL, n_splits, split_a,
               split_b, out, lse, part_o, part_lse, n_threads);
}

/*
 * Tree verification ("Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees"): the
 * draft is a tree of n_nodes nodes verified in one pass under a tree attention mask.  Node i's key and
 * value sit in slot base + i; node i sees the committed prefix (positions < base; with a window, from
 * base + depth_i - W + 1 on) and the nodes whose bit is set in its ancestor-or-self mask.
 *   tree  [1 + n_rows] int32: tree[0] = base, tree[1 + i] = ancestor-or-self mask of node i (i < n_nodes)
 * Other arguments as oracle_verify_attn; rows past n_nodes are padding.
 */
static int tree_run(const uint16_t *q, const uint16_t *kh, const uint16_t *vh, const double *kd,
                    const double *vd, int64_t ctx, const int32_t *tree, int n_rows, int n_nodes, const double *sink,
                    double scale, int64_t window, int n_splits, const int64_t *split_a, const int64_t *split_b,
                    double *out, double *lse, double *part_o, double *part_lse, int n_threads)
{
    if (!tree || n_rows < 1 || n_rows > 64 || n_nodes < 0 || n_nodes > n_rows || n_nodes > 31 || tree[0] < 0)
        return -1;
    for (int i = 0; i < n_nodes; ++i)   /* every node sees itself; masks name existing nodes only */
        if (!((tree[1 + i] >> i) & 1) || (tree[1 + i] >> n_nodes) != 0 || tree[1 + i] < 0) return -1;
    int32_t last[64];
    for (int r = 0; r < n_rows; ++r) last[r] = tree[0] + (n_nodes > 0 ? n_nodes - 1 : 0);
    return run(q, kh, vh, kd, vd, ctx, last, n_rows, n_nodes, sink, scale, window, tree, n_splits, split_a,
               split_b, out, lse, part_o, part_lse, n_threads);
}

int oracle_verify_attn_tree(const uint16_t *q, const uint16_t *kh, const uint16_t *vh, int64_t ctx,
                            const int32_t *tree, int n_rows, int n_nodes, const double *sink, double scale,
                            int64_t window, int n_splits, const int64_t *split_a, const int64_t *split_b,
                            double *out, double *lse, double *part_o, double *part_lse, int n_threads)
{
    if (!kh || !vh) return -1;
    return tree_run(q, kh, vh, NULL, NULL, ctx, tree, n_rows, n_nodes, sink, scale, window, n_splits, split_a,
                    split_b, out, lse, part_o, part_lse, n_threads);
}

/*
 * The tree verification above over a history given as doubles (kd, vd [ctx][128]), as
 * oracle_verify_attn_f64kv is to oracle_verify_attn: the quantised cache's decoded keys and values
 * ("Qwen3.8-27B on one RTX 4090": the verify trees of "More tokens per round: verify trees" read the
 * cache of "A cheaper cache and state").
 */
int oracle_verify_attn_tree_f64kv(const uint16_t *q, const double *kd, const double *vd, int64_t ctx,
                                  const int32_t *tree, int n_rows, int n_nodes, const double *sink, double scale,
                                  int64_t window, int n_splits, const int64_t *split_a, const int64_t *split_b,
                                  double *out, double *lse, double *part_o, double *part_lse, int n_threads)
{
    if (!kd || !vd) return -1;
    return tree_run(q, NULL, NULL, kd, vd, ctx, tree, n_rows, n_nodes, sink, scale, window, n_splits, split_a,
                    split_b, out, lse, part_o, part_lse, n_threads);
}

static int run(const uint16_t *q, const uint16_t *kh, const uint16_t *vh, const double *kd, const double *vd,
               int64_t ctx, const int32_t *pos, int n_rows, int n_live, const double *sink, double scale,
               int64_t window, const int32_t *tree, int n_splits, const int64_t *split_a, const int64_t *split_b,
               double *out, double *lse, double *part_o, double *part_lse, int n_threads)
{
    if (!q || (!kh && !kd) || (!vh && !vd) || !pos || !out || !lse) return -1;
    if (n_rows < 1 || n_live < 0 || n_live > n_rows || window < 0 || n_splits < 0) return -1;
    if (n_splits > 0 && (!split_a || !split_b || !part_o || !part_lse)) return -1;
    for (int r = 0; r < n_live; ++r)
        if (pos[r] < 0 || (int64_t)pos[r] >= ctx) return -1;

    /* padding rows: zero output, LSE -inf, empty partials */
    for (int r = n_live; r < n_rows; ++r)
        for (int h = 0; h < OR_H; ++h) {
            for (int d = 0; d < OR_D; ++d) out[((int64_t)r * OR_H + h) * OR_D + d] = 0.0;
            lse[r * OR_H + h] = -INFINITY;
            for (int s = 0; s < n_splits; ++s) {
                for (int d = 0; d < OR_D; ++d)
                    part_o[(((int64_t)s * n_rows + r) * OR_H + h) * OR_D + d] = 0.0;
                part_lse[((int64_t)s * n_rows + r) * OR_H + h] = -INFINITY;
            }
        }

    job_t J;
    J.q = q; J.kh = kh; J.vh = vh; J.kd = kd; J.vd = vd; J.ctx = ctx; J.pos = pos;
    J.n_rows = n_rows; J.n_live = n_live; J.sink = sink; J.scale = scale; J.window = window; J.tree = tree;
    J.n_splits = n_splits; J.split_a = split_a; J.split_b = split_b;
    J.out = out; J.lse = lse; J.part_o = part_o; J.part_lse = part_lse;
    J.next_pair = 0;
    pthread_mutex_init(&J.mu, NULL);

    int nt = n_threads < 1 ? 1 : n_threads;
    if (nt > n_live * OR_H) nt = n_live * OR_H > 0 ? n_live * OR_H : 1;
    pthread_t th[64];
    if (nt > 64) nt = 64;
    int rc = 0;
    if (nt == 1) {
        if (worker(&J)) rc = -2;
    } else {
        int started = 0;
        for (int t = 0; t < nt; ++t)
            if (pthread_create(&th[t], NULL, worker, &J) == 0) ++started;
        if (started == 0 && worker(&J)) rc = -2;
        for (int t = 0; t < started; ++t) {
            void *res = NULL;
            pthread_join(th[t], &res);
            if (res) rc = -2;
        }
    }
    pthread_mutex_destroy(&J.mu);
    return rc;
}

/*
 * Log-sum-exp merge of split partials with the sink folded in (the separate
 * combine step).
 *   part_o   [n_splits][n_rows][6][128], part_lse [n_splits][n_rows][6]
 *   sink     [6] or NULL
 *   out      [n_rows][6][128], out_lse [n_rows][6]
 * Live rows only; padding rows get 0 / -inf.  If every term is -inf the
 * output is 0 and the LSE -inf.
 */
int oracle_combine(const double *part_o, const double *part_lse, int n_splits, const double *sink,
                   int n_rows, int n_live, double *out, double *out_lse)
{
    if (!part_o || !part_lse || !out || !out_lse || n_splits < 0 || n_rows < 1 || n_live < 0 ||
        n_live > n_rows)
        return -1;
    for (int r = 0; r < n_rows; ++r)
        for (int h = 0; h < OR_H; ++h) {
            double *o = out + ((int64_t)r * OR_H + h) * OR_D;
            for (int d = 0; d < OR_D; ++d) o[d] = 0.0;
            out_lse[r * OR_H + h] = -INFINITY;
            if (r >= n_live) continue;
            const double sk = sink ? sink[h] : -INFINITY;
            double L = sk;
            for (int s = 0; s < n_splits; ++s) {
                const double l = part_lse[((int64_t)s * n_rows + r) * OR_H + h];
                if (l > L) L = l;
            }
            if (L == -INFINITY) continue;
            double z = exp(sk - L);
            for (int s = 0; s < n_splits; ++s)
                z += exp(part_lse[((int64_t)s * n_rows + r) * OR_H + h] - L);
            L += log(z);
            for (int s = 0; s < n_splits; ++s) {
                const double w = exp(part_lse[((int64_t)s * n_rows + r) * OR_H + h] - L);
                const double *po = part_o + (((int64_t)s * n_rows + r) * OR_H + h) * OR_D;
                if (w == 0.0) continue;
                for (int d = 0; d < OR_D; ++d) o[d] += w * po[d];
            }
            out_lse[r * OR_H + h] = L;
        }
    return 0;
}
