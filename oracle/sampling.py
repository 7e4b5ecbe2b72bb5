"""CPU oracle of the steps after verification: sampling, acceptance and cache settlement.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rules as the rest of ``oracle/``): only the tests, the
smoke check and the benchmark's CPU baseline may use it; it shares no code with the CUDA library.

Sources:
  * IQuestRT technical report, section "Include sampling and acceptance in the execution path":
    temperature 1, top-k 20, top-p 0.95 over a 160,000-token vocabulary; the draft keeps its actual
    proposal distribution q; a draft d is accepted with probability min(1, p(d) / q(d)); at the first
    rejection a replacement is drawn from normalise(max(0, p - q)); when every draft is accepted the
    target's extra row supplies a bonus token (at most 7 drafts + 1 bonus = 8 tokens); acceptance,
    next-round input preparation and KV rollback belong to the decode step.
  * the same report, section "Parallelize the Top-K vocabulary scan": 8,192-logit tiles, candidates
    collected per tile, an ordered merge, tile maxima that let the merge skip tiles.
  * the same report, sections "IQuestRT execution" and "Keep the request loop on the GPU": tokens,
    acceptance counts and cache lengths stay on the device; the step settles the caches.
  * "Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees": a draft tree is
    verified in one pass.

Readings where the pages leave a step open:
  * top-k order: by logit descending, equal logits by lower token id;
  * temperature T scales logits before the softmax over the k candidates; top-p keeps the shortest
    prefix of that order whose probability sum reaches top_p (the crossing token included);
  * a draw from a finite distribution with weights w_0.. in candidate order and a uniform u in [0, 1)
    returns the first j whose running sum w_0 + .. + w_j exceeds u * sum(w);
  * these decisions turn floating point into integers, so they are taken in the kernels' precision,
    float32: weights exp((l_j - l_0) / T), running sums in candidate order, the top-p comparison
    run / total >= top_p and the draw threshold u * total are float32 operations here too;
  * the acceptance test "u < min(1, p/q)" is evaluated exactly as u * q < p;
  * the replacement after a rejection is drawn from max(0, p - q) over p's candidates, in p's order;
  * tree acceptance: the target's sampled token at a node selects the child carrying that token (the
    lowest-index child if several do); the walk stops at a node with no such child and emits the
    target's token there (lossless, since every emitted token is a draw from the target);
  * settlement moves the accepted path's K/V from slot base + node to slot base + depth (positions
    taken modulo the cache's slot count) and advances the committed length to base + path length.
"""
from __future__ import annotations

import numpy as np

__all__ = ["TOP_K", "TOP_P", "VOCAB", "TILE_LOGITS", "topk_order", "filtered_distribution", "draw",
           "sample_row", "accept_chain", "tree_accept", "settle", "emitted_distribution"]

TOP_K = 20
TOP_P = 0.95
VOCAB = 160000
TILE_LOGITS = 8192


def topk_order(logits, k: int):
    """Token ids of the k largest logits, largest first, equal logits by lower id (plain sort)."""
    x = np.asarray(logits).astype(np.float64)
    order = np.lexsort((np.arange(x.shape[0]), -x))   # primary: logit descending; then id ascending
    return [int(j) for j in order[:k]]


def filtered_distribution(logits, k: int = TOP_K, top_p: float = TOP_P, temperature: float = 1.0):
    """The sampling distribution after top-k, temperature and top-p, in candidate order.

    Returns (ids, weights, probs): ids of the kept candidates, their unnormalised float32 weights
    exp((l - l_max) / T) and the probabilities weights / sum(weights) (float64 of the float32 values)."""
    f32 = np.float32
    x = np.asarray(logits, dtype=f32)
    ids = topk_order(x, k)
    l0 = x[ids[0]]
    with np.errstate(invalid="ignore", over="ignore"):
        w = np.array([np.exp((x[j] - l0) / f32(temperature)) for j in ids], dtype=f32)
    total = f32(0.0)
    for wi in w:
        total = f32(total + wi)
    keep, run = 0, f32(0.0)
    for wi in w:                      # shortest prefix whose probability reaches top_p
        run = f32(run + wi)
        keep += 1
        if f32(run / total) >= f32(top_p):
            break
    w = w[:keep]
    z = f32(0.0)
    for wi in w:
        z = f32(z + wi)
    return ids[:keep], w, w.astype(np.float64) / float(z)


def draw(weights, u: float) -> int:
    """Index drawn from the finite distribution `weights` (any positive scale) with uniform u in [0, 1):
    the first j whose float32 running sum exceeds u * sum(weights) (float32 operations)."""
    f32 = np.float32
    total = f32(0.0)
    for w in weights:
        total = f32(total + f32(w))
    t = f32(f32(u) * total)
    run = f32(0.0)
    last = -1
    for j, w in enumerate(weights):
        if f32(w) <= 0.0:
            continue
        run = f32(run + f32(w))
        last = j
        if run > t:
            return j
    return last                       # u * total rounded up to the total: the last positive entry


def sample_row(logits, u: float, k: int = TOP_K, top_p: float = TOP_P, temperature: float = 1.0):
    """Top-k / top-p sampling of one row: dict(ids, probs, count, token)."""
    ids, w, probs = filtered_distribution(logits, k, top_p, temperature)
    return dict(ids=ids, probs=probs, weights=w, count=len(ids), token=ids[draw(w, u)])


def accept_chain(p_dists, q_dists, drafts, n_drafts: int, u_accept, u_replace: float, bonus_token: int):
    """Rejection-sampling acceptance of a chain of drafts.

    p_dists[r] = (ids, probs) of the target's distribution at verify row r (r = 0 .. n_drafts), which
    predicts the token after row r's input; drafts[i] (i = 1 .. n_drafts) is the input token of row i,
    proposed from q_dists[i] = (ids, probs).  u_accept[i] tests draft i.  bonus_token is the target's
    own draw at row n_drafts (used when every draft is accepted).
    Returns (n_accepted, tokens): the accepted drafts followed by the replacement or bonus token."""
    out = []
    for i in range(1, n_drafts + 1):
        d = int(drafts[i])
        p_ids, p_pr = p_dists[i - 1]
        q_ids, q_pr = q_dists[i]
        p_d = float(p_pr[p_ids.index(d)]) if d in p_ids else 0.0
        q_d = float(q_pr[q_ids.index(d)]) if d in q_ids else 0.0
        # u < min(1, p/q)  <=>  u * q < p   (q > 0 for a token the draft proposed)
        if float(u_accept[i]) * q_d < p_d:
            out.append(d)
            continue
        f32 = np.float32
        resid = []
        for j, t in enumerate(p_ids):
            qt = f32(q_pr[q_ids.index(t)]) if t in q_ids else f32(0.0)
            resid.append(max(f32(0.0), f32(f32(p_pr[j]) - qt)))
        if not any(r > 0 for r in resid):   # p <= q on all of p's support: draw from p itself
            resid = [f32(x) for x in p_pr]
        out.append(int(p_ids[draw(resid, u_replace)]))
        return i - 1, out
    out.append(int(bonus_token))
    return n_drafts, out


def tree_accept(parents, node_tokens, target_tokens):
    """Walk a draft tree from the root: at node v the target's token target_tokens[v] selects the
    lowest-index child carrying it.  Returns (path, emitted): the accepted node path (root first) and the
    emitted tokens (the accepted children's tokens, then the target's token at the last node)."""
    n = len(parents)
    path = [0]
    emitted = []
    v = 0
    while True:
        t = int(target_tokens[v])
        nxt = -1
        for c in range(n):
            if parents[c] == v and int(node_tokens[c]) == t:
                nxt = c
                break
        if nxt < 0:
            emitted.append(t)
            return path, emitted
        path.append(nxt)
        emitted.append(t)
        v = nxt


def settle(k_cache, v_cache, base: int, path):
    """Move the accepted path's K/V rows from slot (base + node) to slot (base + depth), modulo the
    cache's slot count, on copies; returns (k, v, next_base)."""
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    slots = k.shape[0]
    rows_k = [np.array(k_cache[(base + node) % slots]) for node in path]
    rows_v = [np.array(v_cache[(base + node) % slots]) for node in path]
    for depth in range(len(path)):
        k[(base + depth) % slots] = rows_k[depth]
        v[(base + depth) % slots] = rows_v[depth]
    return k, v, base + len(path)


def emitted_distribution(p_ids, p_probs, q_ids, q_probs, n_grid: int = 4096):
    """Distribution of the first emitted token when one draft d ~ q is tested against p and the
    replacement is drawn from max(0, p - q): exact in d and in the acceptance coin (its probability
    min(1, p/q)), a midpoint grid of n_grid values for the replacement's uniform.  For testing only."""
    dist = {}
    for d, qd in zip(q_ids, q_probs):
        pd = float(p_probs[p_ids.index(d)]) if d in p_ids else 0.0
        a = min(1.0, pd / float(qd))
        dist[d] = dist.get(d, 0.0) + float(qd) * a
        if a < 1.0:
            resid = []
            for j, t in enumerate(p_ids):
                qt = float(q_probs[q_ids.index(t)]) if t in q_ids else 0.0
                resid.append(max(0.0, float(p_probs[j]) - qt))
            counts = np.zeros(len(p_ids))
            for g in range(n_grid):
                counts[draw(resid, (g + 0.5) / n_grid)] += 1
            for j, t in enumerate(p_ids):
                dist[t] = dist.get(t, 0.0) + float(qd) * (1.0 - a) * counts[j] / n_grid
    return dist
