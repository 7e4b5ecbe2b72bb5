"""Pins of the sampling / acceptance / settlement oracle (no GPU).

IQuestRT report, section "Include sampling and acceptance in the execution path" (top-k 20, top-p 0.95,
temperature 1, rejection sampling with min(1, p/q), replacement from max(0, p - q), bonus token) and
"Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees".  Each check reaches the
oracle's result by another route: brute force, torch.topk, closed forms, exact counting over a grid of
uniforms, and the losslessness of speculative sampling (the emitted token is distributed as p).
"""
import numpy as np
import pytest
import torch

from oracle import sampling as S


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------- top-k
def test_topk_order_brute_force_with_ties():
    for seed in range(20):
        x = _rng(seed).integers(-5, 6, size=300).astype(np.float32)   # many ties
        brute = sorted(range(300), key=lambda j: (-float(x[j]), j))[:20]
        assert S.topk_order(x, 20) == brute


def test_topk_values_match_torch_topk():
    x = _rng(1).standard_normal(S.VOCAB).astype(np.float32) * 3
    ids = S.topk_order(x, S.TOP_K)
    v, _ = torch.topk(torch.from_numpy(x), S.TOP_K)
    assert np.array_equal(x[ids], v.numpy())


# ----------------------------------------------------------------------------- top-p, temperature
def test_top_p_closed_form():
    p = np.array([0.5, 0.3, 0.12, 0.05, 0.03])
    logits = np.full(100, -50.0, dtype=np.float32)
    logits[[7, 3, 50, 9, 60]] = np.log(p).astype(np.float32)
    ids, w, probs = S.filtered_distribution(logits, 20, 0.95, 1.0)
    assert ids == [7, 3, 50, 9]                       # 0.5, 0.8, 0.92 < 0.95 <= 0.97
    pf = np.exp(logits[[7, 3, 50, 9]].astype(np.float64))
    np.testing.assert_allclose(probs, pf / pf.sum(), rtol=1e-6)   # float32 weights
    ids1, _, _ = S.filtered_distribution(logits, 20, 0.5, 1.0)
    assert ids1 == [7]                                # the crossing token alone reaches 0.5
    idsk, _, _ = S.filtered_distribution(logits, 2, 1.0, 1.0)
    assert idsk == [7, 3]                             # top-k bounds the set


def test_temperature_closed_form():
    logits = np.array([2.0, 1.0, 0.0, -1.0], dtype=np.float32)
    for T in (0.5, 1.0, 1.25, 2.0):
        _, _, probs = S.filtered_distribution(logits, 4, 1.0, T)
        e = np.exp(np.array([2.0, 1.0, 0.0, -1.0]) / T)
        np.testing.assert_allclose(probs, e / e.sum(), rtol=1e-6)


# ----------------------------------------------------------------------------- draws
def test_draw_is_the_inverse_cdf_counting_over_a_grid():
    for seed in range(5):
        w = _rng(seed).random(7) + 0.01
        w[3] = 0.0
        N = 7000
        counts = np.zeros(7)
        for g in range(N):
            counts[S.draw(w, (g + 0.5) / N)] += 1
        np.testing.assert_allclose(counts / N, w / w.sum(), atol=1.5 / N)
        assert counts[3] == 0


def test_draw_edges():
    assert S.draw([1.0, 1.0], 0.0) == 0
    assert S.draw([1.0, 1.0], np.nextafter(1.0, 0.0)) == 1
    assert S.draw([0.0, 2.0, 0.0], 0.3) == 1


# ----------------------------------------------------------------------------- rejection sampling
def _sparse(rng, vocab_ids, k):
    ids = list(rng.choice(vocab_ids, size=k, replace=False))
    pr = rng.random(k) + 0.05
    order = np.argsort(-pr, kind="stable")
    return [int(ids[i]) for i in order], pr[order] / pr.sum()


@pytest.mark.parametrize("seed", range(6))
def test_speculative_sampling_is_lossless(seed):
    # the first emitted token of one draft step is distributed as p, whatever q is
    rng = _rng(seed)
    p_ids, p_pr = _sparse(rng, np.arange(30), 8)
    q_ids, q_pr = _sparse(rng, np.arange(30), 9)
    dist = S.emitted_distribution(p_ids, p_pr, q_ids, q_pr, n_grid=8192)
    for t, pt in zip(p_ids, p_pr):
        assert abs(dist.get(t, 0.0) - pt) < 2e-3, (t, dist.get(t), pt)
    assert sum(v for t, v in dist.items() if t not in p_ids) < 1e-12


def test_accept_chain_cases():
    p = [([5, 6], np.array([0.6, 0.4]))] * 4
    q = [None] + [([5, 6], np.array([0.6, 0.4]))] * 3
    # q == p: every draft accepted, the bonus follows
    n, toks = S.accept_chain(p, q, [0, 5, 6, 5], 3, [0, 0.99, 0.99, 0.99], 0.5, bonus_token=77)
    assert n == 3 and toks == [5, 6, 5, 77]
    # a draft the target never proposes is rejected; the replacement comes from p - q
    q2 = [None, ([9, 5], np.array([0.9, 0.1])), ([5], np.array([1.0])), ([5], np.array([1.0]))]
    n, toks = S.accept_chain(p, q2, [0, 9, 5, 5], 3, [0, 0.0, 0.0, 0.0], 0.0, bonus_token=77)
    assert n == 0 and toks[0] == 5                   # max(0, p - q) = (0.5, 0.4): u = 0 -> id 5
    n, toks = S.accept_chain(p, q2, [0, 9, 5, 5], 3, [0, 0.0, 0.0, 0.0], 0.99, bonus_token=77)
    assert n == 0 and toks == [6]
    # min(1, p/q) against u, tested exactly as u * q < p
    q3 = [None, ([5], np.array([1.0]))] + [([5], np.array([1.0]))] * 2
    n, _ = S.accept_chain(p, q3, [0, 5, 5, 5], 3, [0, 0.5999999, 0.6, 0.1], 0.0, bonus_token=77)
    assert n == 1                                    # 0.6 * 1 < 0.6 is false: rejected at draft 2


# ----------------------------------------------------------------------------- trees
def test_tree_accept_on_a_chain_is_the_matching_prefix():
    parents = [-1, 0, 1, 2, 3]
    node_tokens = [100, 11, 12, 13, 14]
    path, em = S.tree_accept(parents, node_tokens, [11, 12, 99, 14, 15])
    assert path == [0, 1, 2] and em == [11, 12, 99]
    path, em = S.tree_accept(parents, node_tokens, [11, 12, 13, 14, 15])
    assert path == [0, 1, 2, 3, 4] and em == [11, 12, 13, 14, 15]


def test_tree_accept_chooses_the_matching_child():
    parents = [-1, 0, 0, 0, 2, 2, 5]
    node_tokens = [1, 10, 20, 30, 40, 50, 60]
    path, em = S.tree_accept(parents, node_tokens, [20, 0, 50, 0, 0, 60, 7])
    assert path == [0, 2, 5, 6] and em == [20, 50, 60, 7]
    path, em = S.tree_accept(parents, node_tokens, [31, 0, 0, 0, 0, 0, 0])
    assert path == [0] and em == [31]
    # duplicate sibling tokens: the lowest index wins
    path, _ = S.tree_accept([-1, 0, 0], [1, 5, 5], [5, 9, 9])
    assert path == [0, 1]


# ----------------------------------------------------------------------------- settlement
def _rand_tree(rng, n):
    return [-1] + [int(rng.integers(0, i)) for i in range(1, n)]


def _path_to(parents, v):
    path = []
    while v >= 0:
        path.append(v)
        v = parents[v]
    return path[::-1]


def test_settle_moves_the_path_and_matches_an_in_order_copy():
    rng = _rng(7)
    for trial in range(30):
        n = 16
        parents = _rand_tree(rng, n)
        path = _path_to(parents, int(rng.integers(0, n)))
        slots = int(rng.choice([64, 100, 4160]))
        base = int(rng.integers(0, 3 * slots))
        k = rng.integers(0, 1 << 16, size=(slots, 8)).astype(np.uint16)
        v = rng.integers(0, 1 << 16, size=(slots, 8)).astype(np.uint16)
        k2, v2, nb = S.settle(k, v, base, path)
        assert nb == base + len(path)
        # sequential in-order copy (safe because a path node's index is never below its depth)
        kk, vv = k.copy(), v.copy()
        for d, node in enumerate(path):
            assert node >= d
            kk[(base + d) % slots] = kk[(base + node) % slots]
            vv[(base + d) % slots] = vv[(base + node) % slots]
        assert np.array_equal(k2, kk) and np.array_equal(v2, vv)
        # every other slot is untouched
        moved = {(base + d) % slots for d in range(len(path))}
        for s in range(slots):
            if s not in moved:
                assert np.array_equal(k2[s], k[s])


def test_settle_of_a_chain_changes_nothing():
    k = np.arange(64 * 4, dtype=np.uint16).reshape(64, 4)
    k2, v2, nb = S.settle(k, k, 10, [0, 1, 2, 3])
    assert np.array_equal(k2, k) and nb == 14
