"""Pins of the FP64 tree-verify oracle (no GPU).

"Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees": the drafts form a tree
that the target verifies in one pass under a tree attention mask.  Node i's K/V sit at slot base + i;
node i sees the committed prefix and its ancestors.  The oracle takes ancestor-or-self bitmasks; the
pins below reach the same results through other routes:

  * a parent-array walk plus torch's float64 SDPA with the sink as an extra zero key (library route);
  * chain-shaped trees reduce exactly to the causal verify of consecutive rows (full and windowed);
  * closed forms (uniform scores give the mean of the visible values) on star and chain trees;
  * invariants: a node ignores the K/V of every node that is not its ancestor; split partials merge
    to the direct result;
  * planted mistakes (a slot-index window instead of the depth one, a causal mask in slot order, the
    sink dropped) fail the parity bars.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from speculative_decode_verify_gb300 import synth

D, H = 128, 6


def _f64(t):
    return oracle.bf16_bits_to_f64(synth.bits(t).numpy())


def _run(w, n_splits=0, ranges=None, masks=None, window=None, n_nodes=None):
    return oracle.verify_attn_tree(
        synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(), synth.bits(w.v_hist).numpy(), w.base,
        (w.masks if masks is None else masks).numpy(), w.n_nodes if n_nodes is None else n_nodes,
        w.sink.numpy(), w.scale, window=w.window if window is None else window, n_splits=n_splits,
        split_ranges=ranges, n_threads=4)


def _walk_visible(w, i, window):
    """Slots node i sees, from the parent array: the prefix window of its logical position base + depth,
    then itself and its ancestors found by walking the parents (those inside the window)."""
    chain = []
    n = i
    while n >= 0:
        chain.append(n)
        n = w.parents[n]
    depth = len(chain) - 1
    logical = w.base + depth
    first = max(0, logical - window + 1) if window > 0 else 0
    vis = [j for j in range(first, w.base)]
    for k in chain:   # the ancestor at depth dk has logical position base + dk
        dk = len([None for _ in _ancestors(w, k)])
        if window <= 0 or w.base + dk >= first:
            vis.append(w.base + k)
    return sorted(vis)


def _ancestors(w, k):
    n = w.parents[k]
    while n >= 0:
        yield n
        n = w.parents[n]


def _sdpa_tree(w, window, with_sink=True):
    q = torch.from_numpy(_f64(w.q))
    K = torch.from_numpy(_f64(w.k_hist))
    V = torch.from_numpy(_f64(w.v_hist))
    ctx = K.shape[0]
    Kx = torch.cat([K, torch.zeros(1, D, dtype=torch.float64)])
    Vx = torch.cat([V, torch.zeros(1, D, dtype=torch.float64)])
    out = np.zeros((w.n_rows, H, D))
    lse = np.full((w.n_rows, H), -np.inf)
    for i in range(w.n_nodes):
        mask = torch.full((ctx + 1,), float("-inf"), dtype=torch.float64)
        mask[_walk_visible(w, i, window)] = 0.0
        for h in range(H):
            m = mask.clone()
            m[ctx] = float(w.sink[h]) if with_sink else float("-inf")
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, i:i + 1, h, :], Kx[None, None], Vx[None, None], attn_mask=m[None, None, None],
                scale=w.scale)
            out[i, h] = o[0, 0, 0].numpy()
            lse[i, h] = float(torch.logsumexp((Kx @ q[i, h]) * w.scale + m, dim=0))
    return out, lse


def _tree(seed, base, n_nodes, shape="best_first", window=0, n_rows=16):
    return synth.make_tree("pin", seed, base=base, n_nodes=n_nodes, shape=shape, window=window, n_rows=n_rows)


# ----------------------------------------------------------------------------- library route
@pytest.mark.parametrize("seed,base,n_nodes,shape,window", [
    (31, 0, 1, "best_first", 0), (32, 5, 16, "best_first", 0), (33, 150, 16, "best_first", 0),
    (34, 70, 11, "star", 0), (35, 90, 16, "best_first", 20), (36, 40, 16, "chain", 6),
    (37, 64, 9, "best_first", 3), (38, 200, 16, "best_first", 130)])
def test_tree_oracle_matches_parent_walk_sdpa(seed, base, n_nodes, shape, window):
    w = _tree(seed, base, n_nodes, shape, window)
    res = _run(w)
    ref_out, ref_lse = _sdpa_tree(w, window)
    n = w.n_nodes
    np.testing.assert_allclose(res["out"][:n], ref_out[:n], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["lse"][:n], ref_lse[:n], rtol=1e-12, atol=1e-12)
    assert np.all(res["out"][n:] == 0.0) and np.all(np.isneginf(res["lse"][n:]))


def test_tree_visible_positions_model_matches_parent_walk():
    for seed, window in ((41, 0), (42, 5), (43, 4096)):
        w = _tree(seed, 300, 16, window=window)
        for i in range(w.n_nodes):
            assert oracle.tree_visible_positions(w.base, w.masks.numpy(), w.n_nodes, i, window) == \
                _walk_visible(w, i, window)


# ----------------------------------------------------------------------------- reduction to the chain
@pytest.mark.parametrize("window,n_nodes", [(0, 8), (0, 16), (4096, 16), (37, 7), (1, 5)])
def test_chain_tree_equals_causal_verify_of_consecutive_rows(window, n_nodes):
    base = 5000 if window == 4096 else 700
    w = _tree(51, base, n_nodes, "chain", window, n_rows=n_nodes)
    tree = _run(w, n_splits=5)
    chain = oracle.verify_attn(synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(),
                               synth.bits(w.v_hist).numpy(), w.node_pos.numpy(), n_nodes, w.sink.numpy(),
                               w.scale, window=window, n_splits=5, split_ranges=tree["ranges"], n_threads=4)
    assert np.array_equal(tree["out"], chain["out"]) and np.array_equal(tree["lse"], chain["lse"])
    assert np.array_equal(tree["part_o"], chain["part_o"])
    assert np.array_equal(tree["part_lse"], chain["part_lse"])


def test_tree_extent_of_a_chain_equals_the_chain_extent():
    for window in (0, 100, 4096):
        w = _tree(52, 3000, 16, "chain", window)
        assert oracle.tree_extent(w.base, w.masks.numpy(), 16, window) == \
            oracle.read_extent(w.node_pos.numpy(), 16, window)


# ----------------------------------------------------------------------------- closed forms
def test_star_tree_with_uniform_scores_is_the_mean_of_prefix_root_and_self():
    w = _tree(53, 90, 12, "star")
    w.q = torch.zeros_like(w.q)
    res = _run(w)
    V = _f64(w.v_hist)
    prefix = V[:w.base].sum(0)
    for i in range(w.n_nodes):
        keys = [w.base] if i == 0 else [w.base, w.base + i]
        n = w.base + len(keys)
        for h in range(H):
            zs = np.exp(float(w.sink[h]))   # scores are all 0: weights 1, sink weight e^sink
            expect = (prefix + V[keys].sum(0)) / (n + zs)
            np.testing.assert_allclose(res["out"][i, h], expect, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(res["lse"][i, h], np.log(n + zs), rtol=1e-13)


def test_root_alone_sees_prefix_and_itself():
    w = _tree(54, 33, 1)
    w.q = torch.zeros_like(w.q)
    w.sink = torch.full((H,), float("-inf"))
    res = _run(w)
    expect = _f64(w.v_hist)[:34].mean(0)
    for h in range(H):
        np.testing.assert_allclose(res["out"][0, h], expect, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------- invariants
def test_node_ignores_non_ancestor_nodes():
    w = _tree(55, 120, 16)
    base_res = _run(w)
    masks = w.masks.numpy()
    for k in range(1, w.n_nodes):
        w2 = _tree(55, 120, 16)
        w2.k_hist[w.base + k] = synth.normal_bf16((D,), synth.generator(900 + k), 3.0)
        w2.v_hist[w.base + k] = synth.normal_bf16((D,), synth.generator(950 + k), 3.0)
        res = _run(w2)
        for i in range(w.n_nodes):
            same = np.array_equal(res["out"][i], base_res["out"][i])
            assert same == (not ((int(masks[i]) >> k) & 1)), (k, i)


@pytest.mark.parametrize("window", [0, 30])
def test_tree_split_partials_merge_to_the_direct_result(window):
    w = _tree(56, 700, 16, window=window)
    res = _run(w, n_splits=7)
    out, lse = oracle.combine(res["part_o"], res["part_lse"], w.sink.numpy(), w.n_nodes)
    np.testing.assert_allclose(out[:16], res["out"][:16], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(lse[:16], res["lse"][:16], rtol=1e-12, atol=1e-12)
    lo, hi = oracle.tree_extent(w.base, w.masks.numpy(), 16, window)
    assert res["ranges"] == oracle.split_position_ranges(lo, hi, 7)


def test_oracle_rejects_malformed_masks():
    w = _tree(57, 50, 6, n_rows=8)
    bad_self = w.masks.clone()
    bad_self[3] &= ~(1 << 3)
    bad_range = w.masks.clone()
    bad_range[2] |= 1 << 6
    for m in (bad_self, bad_range):
        with pytest.raises(ValueError):
            _run(w, masks=m)


def test_synthetic_trees_are_well_formed():
    for seed in range(20):
        parents = synth.best_first_tree(synth.generator(seed), 16)
        assert parents[0] == -1 and all(0 <= p < i for i, p in enumerate(parents) if i > 0)
        masks = synth.ancestor_masks(parents).numpy()
        assert np.array_equal(masks, oracle.tree_masks_from_parents(parents))


# ----------------------------------------------------------------------------- planted mistakes
def _bf16(x):
    return oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(x))


def _fails(w, got, ref):
    m = parity.out_metrics(_bf16(got), _bf16(ref), w.n_nodes)
    return not parity.out_ok(m)


def test_negative_control_window_by_slot_index_fails_the_bar():
    # planted in the oracle's inputs: a window that ends at the node's slot (base + i) instead of its
    # logical position (base + depth) drops prefix keys every deep-slot node should see
    w = _tree(58, 400, 16, window=24)
    right = _run(w)
    wrong_out = right["out"].copy()
    for i in range(w.n_nodes):
        tw = _tree(58, 400, 16, window=24)
        # same node, but seen as a chain row at slot base + i
        chain = oracle.verify_attn(synth.bits(tw.q).numpy()[i:i + 1], synth.bits(tw.k_hist).numpy(),
                                   synth.bits(tw.v_hist).numpy(), np.array([w.base + i]), 1, w.sink.numpy(),
                                   w.scale, window=24)
        wrong_out[i] = chain["out"][0]
    assert _fails(w, wrong_out, right["out"])


def test_negative_control_causal_mask_in_slot_order_fails_the_bar():
    w = _tree(59, 64, 16)
    right = _run(w)
    causal = np.array([(1 << (i + 1)) - 1 for i in range(16)], dtype=np.int32)
    wrong = _run(w, masks=torch.from_numpy(causal))
    assert _fails(w, wrong["out"], right["out"])


def test_negative_control_dropped_sink_fails_the_bar():
    w = _tree(60, 30, 16)
    right = _run(w)
    w.sink = w.sink + 4.0
    wrong = _run(w)
    assert _fails(w, wrong["out"], right["out"])
