"""Pins of the FP64 oracle of tree verification over the quantised cache (no GPU).

"Qwen3.8-27B on one RTX 4090": the 16-node verify trees of section "More tokens per round: verify trees"
read the cache of section "A cheaper cache and state" (FP8 keys after a Hadamard rotation, INT8 values).
``oracle.kv_codec.verify_attn_tree_decoded`` is the tree oracle over the decoded keys and values; it is
pinned through other routes:

  * a parent-array walk plus torch's float64 SDPA over the decoded cache, the sink as an extra zero key
    (library route; full attention and a window);
  * over a history whose "decoded" values are the bf16 history widened, it equals the bf16 tree oracle
    bit for bit (the same arithmetic reached through the other entry);
  * a chain-shaped tree equals the chain oracle over the same decoded cache;
  * split partials merge to the direct result;
  * planted mistakes (K and V swapped, the masks ignored, a window on the slot index, a split plan over
    the nodes' logical positions) fail one of the pins.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_codec as C
from speculative_decode_verify_gb300 import synth

D, H = 128, 6


def _bits(t):
    return synth.bits(t).numpy()


def _decoded(w):
    kc, ks = C.encode_k(_bits(w.k_hist))
    vc, vs = C.encode_v(_bits(w.v_hist))
    return C.decode_k(kc, ks), C.decode_v(vc, vs)


def _run(w, kd, vd, n_splits=0, masks=None, window=None):
    return C.verify_attn_tree_decoded(_bits(w.q), kd, vd, w.base, (w.masks if masks is None else masks).numpy(),
                                      w.n_nodes, w.sink.numpy(), w.scale,
                                      window=w.window if window is None else window, n_splits=n_splits, n_threads=4)


def _walk_visible(w, i, window):
    """Positions node i sees, from the parent array: the prefix from its logical position's window start
    (base + depth - window + 1), then itself and its ancestors."""
    chain = []
    n = i
    while n >= 0:
        chain.append(n)
        n = w.parents[n]
    logical = w.base + len(chain) - 1
    first = max(0, logical - window + 1) if window > 0 else 0
    return sorted(list(range(first, w.base)) + [w.base + k for k in chain])


def _sdpa(w, kd, vd, window):
    q = torch.from_numpy(oracle.bf16_bits_to_f64(_bits(w.q)))
    ctx = kd.shape[0]
    K = torch.cat([torch.from_numpy(kd), torch.zeros(1, D, dtype=torch.float64)])
    V = torch.cat([torch.from_numpy(vd), torch.zeros(1, D, dtype=torch.float64)])
    out = np.zeros((w.n_rows, H, D))
    lse = np.full((w.n_rows, H), -np.inf)
    for i in range(w.n_nodes):
        base_mask = torch.full((ctx + 1,), float("-inf"), dtype=torch.float64)
        base_mask[_walk_visible(w, i, window)] = 0.0
        for h in range(H):
            m = base_mask.clone()
            m[ctx] = float(w.sink[h])
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, i:i + 1, h], K[None, None], V[None, None], attn_mask=m[None, None, None], scale=w.scale)
            out[i, h] = o[0, 0, 0].numpy()
            lse[i, h] = float(torch.logsumexp((K @ q[i, h]) * w.scale + m, dim=0))
    return out, lse


def _check_sdpa(w, res, kd, vd):
    ref_out, ref_lse = _sdpa(w, kd, vd, w.window)
    n = w.n_nodes
    np.testing.assert_allclose(res["out"][:n], ref_out[:n], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["lse"][:n], ref_lse[:n], rtol=1e-12, atol=1e-12)
    assert np.all(res["out"][n:] == 0.0) and np.all(np.isneginf(res["lse"][n:]))


@pytest.mark.parametrize("seed,base,n_nodes,shape,window", [
    (81, 0, 1, "best_first", 0), (82, 150, 16, "best_first", 0), (83, 70, 11, "star", 0),
    (84, 90, 16, "best_first", 20), (85, 200, 16, "best_first", 130), (86, 40, 9, "chain", 12)])
def test_decoded_tree_oracle_matches_parent_walk_sdpa(seed, base, n_nodes, shape, window):
    w = synth.make_tree("q8tpin", seed, base=base, n_nodes=n_nodes, shape=shape, window=window)
    kd, vd = _decoded(w)
    _check_sdpa(w, _run(w, kd, vd), kd, vd)


@pytest.mark.parametrize("window", [0, 25])
def test_widened_bf16_history_gives_the_bf16_tree_oracle_bit_for_bit(window):
    w = synth.make_tree("q8tbits", 87, base=230, n_nodes=16, window=window)
    kd, vd = oracle.bf16_bits_to_f64(_bits(w.k_hist)), oracle.bf16_bits_to_f64(_bits(w.v_hist))
    got = _run(w, kd, vd, n_splits=5)
    ref = oracle.verify_attn_tree(_bits(w.q), _bits(w.k_hist), _bits(w.v_hist), w.base, w.masks.numpy(), w.n_nodes,
                                  w.sink.numpy(), w.scale, window=window, n_splits=5, n_threads=4)
    for key in ("out", "lse", "part_o", "part_lse"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["ranges"] == ref["ranges"]


@pytest.mark.parametrize("window", [0, 30])
def test_chain_tree_equals_the_chain_oracle_over_the_same_decoded_cache(window):
    w = synth.make_tree("q8tchain", 88, base=300, n_nodes=8, shape="chain", window=window, n_rows=8)
    kd, vd = _decoded(w)
    got = _run(w, kd, vd)
    ref = C.verify_attn_decoded(_bits(w.q), kd, vd, w.node_pos.numpy(), 8, w.sink.numpy(), w.scale, window)
    np.testing.assert_allclose(got["out"], ref["out"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(got["lse"], ref["lse"], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("window", [0, 40])
def test_decoded_tree_split_partials_merge_to_the_direct_result(window):
    w = synth.make_tree("q8tsplit", 89, base=500, n_nodes=16, window=window)
    kd, vd = _decoded(w)
    res = _run(w, kd, vd, n_splits=6)
    lo, hi = oracle.tree_extent(w.base, w.masks.numpy(), w.n_nodes, window)
    assert res["ranges"] == oracle.split_position_ranges(lo, hi, 6)
    out, lse = oracle.combine(res["part_o"], res["part_lse"], w.sink.numpy(), w.n_nodes)
    np.testing.assert_allclose(out[:w.n_nodes], res["out"][:w.n_nodes], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(lse[:w.n_nodes], res["lse"][:w.n_nodes], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- planted mistakes
def _fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_fail_the_pins():
    w = synth.make_tree("q8tplant", 90, base=120, n_nodes=16, window=0)
    kd, vd = _decoded(w)
    # K and V swapped on the way in
    assert _fails(lambda: _check_sdpa(w, _run(w, vd, kd), kd, vd))
    # the masks ignored: every node sees every node
    full = torch.full_like(w.masks, (1 << w.n_nodes) - 1)
    full[w.n_nodes:] = 0
    assert _fails(lambda: _check_sdpa(w, _run(w, kd, vd, masks=full), kd, vd))
    # a window on the slot index instead of the node's logical position
    ww = synth.make_tree("q8tplant", 91, base=120, n_nodes=16, window=20)
    kdw, vdw = _decoded(ww)
    slot_window = C.verify_attn_decoded(_bits(ww.q), kdw, vdw, ww.node_pos.numpy(), 16, ww.sink.numpy(), ww.scale, 20)
    assert _fails(lambda: _check_sdpa(ww, slot_window, kdw, vdw))
    # the split plan over the nodes' logical positions (base + depth) instead of their slots: the partials
    # miss the deeper slots and no longer merge to the direct result
    depth = max(bin(int(m)).count("1") - 1 for m in ww.masks[:16])
    lo, _ = oracle.tree_extent(ww.base, ww.masks.numpy(), 16, 20)
    wrong = oracle.split_position_ranges(lo, ww.base + depth + 1, 4)
    res = C.verify_attn_tree_decoded(_bits(ww.q), kdw, vdw, ww.base, ww.masks.numpy(), 16, ww.sink.numpy(), ww.scale,
                                     window=20, split_ranges=wrong)
    out, _ = oracle.combine(res["part_o"], res["part_lse"], ww.sink.numpy(), 16)

    def merge_pin():
        np.testing.assert_allclose(out[:16], res["out"][:16], rtol=1e-10, atol=1e-13)
    assert depth + 1 < 16 and _fails(merge_pin)
