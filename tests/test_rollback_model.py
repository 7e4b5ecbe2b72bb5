"""Two rounds of verification with partial acceptance, modelled on the CPU with the oracle alone.

IQuestRT report, "Include sampling and acceptance in the execution path" and "Keep the request loop on the
GPU": after round 1 accepts k of its 7 drafts, round 2 appends its rows from next_pos = P0 + k + 1 on (over
the rejected drafts' slots) and verifies; "Let correctness checks change the design": the sliding-window
ring must hold W + n - 1 positions (4,160 = 4,096 + 64 slots here), since the append comes before the reads.

The model runs the oracle's append (slot = position mod slots), the oracle's chain acceptance or tree
acceptance and settlement, then reads back, through the slots, what every round-2 row would see.  Two
checks hold for the correct model and must fail for a planted mistake:
  * cache bytes: for every position a round-2 row can see, its slot holds the accepted history's K/V;
  * outputs: FP64 attention over what the slots hold equals attention over the accepted linear history.
The GPU test (tests/test_gpu_rollback.py) makes the same comparisons through the CUDA library.
"""
import numpy as np
import pytest

import oracle
from oracle import sampling as S
from rollback_cases import N_DRAFTS, N_ROWS, Scenario, dists, forced_chain_acceptance, ring_view
from speculative_decode_verify_gb300 import synth

W, RING = synth.WINDOW, synth.RING_SLOTS


def _bits(t):
    return synth.bits(t).numpy()


def chain_model(sc: Scenario, slots: int, k_accept: int, next_pos_shift: int = 0):
    k, v = (x.numpy() for x in sc.initial_cache(slots))
    pos1 = sc.p0 + np.arange(N_ROWS)
    k, v = oracle.ring_append(k, v, _bits(sc.r1_k[:N_ROWS]), _bits(sc.r1_v[:N_ROWS]), pos1, N_ROWS)
    a = forced_chain_acceptance(k_accept)
    n_acc, _ = S.accept_chain(dists(a["p_ids"], a["p_probs"], a["p_counts"]),
                              dists(a["q_ids"], a["q_probs"], a["q_counts"]), a["drafts"].tolist(), N_DRAFTS,
                              a["u_accept"].tolist(), float(a["u_replace"][0]), int(a["target"][N_DRAFTS]))
    next_pos = sc.p0 + n_acc + 1 + next_pos_shift
    pos2 = next_pos + np.arange(N_ROWS)
    k, v = oracle.ring_append(k, v, _bits(sc.r2_k), _bits(sc.r2_v), pos2, N_ROWS)
    return k, v, n_acc, next_pos


def tree_model(sc: Scenario, slots: int, seed: int, next_pos_shift: int = 0):
    parents, tokens, target = synth.tree_round(seed)
    k, v = (x.numpy() for x in sc.initial_cache(slots))
    k, v = oracle.ring_append(k, v, _bits(sc.r1_k), _bits(sc.r1_v), sc.p0 + np.arange(16), 16)
    path, _ = S.tree_accept(parents, tokens.tolist(), target.tolist())
    k, v, next_pos = S.settle(k, v, sc.p0, path)
    next_pos += next_pos_shift
    k, v = oracle.ring_append(k, v, _bits(sc.r2_k), _bits(sc.r2_v), next_pos + np.arange(N_ROWS), N_ROWS)
    return k, v, path, next_pos


def round2_checks(sc: Scenario, k, v, accepted_rows, next_pos_true: int, next_pos_used: int):
    """(bytes_ok, out_equal) of round 2 against the accepted linear history."""
    hk, hv = (x.numpy() for x in sc.history_round2(accepted_rows, next_pos_true))
    pos_true = next_pos_true + np.arange(N_ROWS)
    lo, hi = oracle.read_extent(pos_true, N_ROWS, sc.window)
    vk, vv = ring_view(k, v, max(hi, next_pos_used + N_ROWS))
    bytes_ok = bool(np.array_equal(vk[lo:hi], hk[lo:hi]) and np.array_equal(vv[lo:hi], hv[lo:hi]))
    q = _bits(sc.q2)
    ref = oracle.verify_attn(q, hk, hv, pos_true, N_ROWS, sc.sink.numpy(), sc.scale, sc.window)
    got = oracle.verify_attn(q, vk, vv, next_pos_used + np.arange(N_ROWS), N_ROWS, sc.sink.numpy(), sc.scale,
                             sc.window)
    return bytes_ok, bool(np.array_equal(got["out"], ref["out"]))


@pytest.mark.parametrize("k_accept", range(N_DRAFTS + 1))
@pytest.mark.parametrize("layer", ["full", "ring", "ring_wrap"])
def test_chain_rounds_model_matches_the_accepted_history(layer, k_accept):
    if layer == "full":
        sc, slots = Scenario(10 + k_accept, 3000), 3100
    elif layer == "ring":
        sc, slots = Scenario(20 + k_accept, 40000, window=W), RING
    else:                       # round 1 straddles the end of the ring: slots 4156..4159, then 0..
        sc, slots = Scenario(30 + k_accept, 10 * RING - 4, window=W), RING
    k, v, n_acc, nxt = chain_model(sc, slots, k_accept)
    assert n_acc == k_accept and nxt == sc.p0 + k_accept + 1
    assert round2_checks(sc, k, v, list(range(k_accept + 1)), nxt, nxt) == (True, True)


@pytest.mark.parametrize("k_accept", [0, 3, 7])
def test_planted_next_pos_off_by_one_fails(k_accept):
    sc = Scenario(40 + k_accept, 40000, window=W)
    for shift in (1, -1):
        k, v, n_acc, nxt = chain_model(sc, RING, k_accept, next_pos_shift=shift)
        true_next = sc.p0 + n_acc + 1
        assert round2_checks(sc, k, v, list(range(k_accept + 1)), true_next, nxt) == (False, False)


@pytest.mark.parametrize("k_accept", [0, 4, 7])
def test_planted_ring_one_slot_short_fails(k_accept):
    # W + n - 1 = 4,103 slots is the least that keeps round 2's first window whole; with 4,102 the last
    # appended row lands on the slot of row 0's oldest visible position
    sc = Scenario(50 + k_accept, 40000, window=W)
    for slots in (W + N_ROWS - 1, RING):
        k, v, n_acc, nxt = chain_model(sc, slots, k_accept)
        assert round2_checks(sc, k, v, list(range(k_accept + 1)), nxt, nxt) == (True, True)
    k, v, n_acc, nxt = chain_model(sc, W + N_ROWS - 2, k_accept)
    assert round2_checks(sc, k, v, list(range(k_accept + 1)), nxt, nxt) == (False, False)


@pytest.mark.parametrize("layer", ["full", "ring"])
@pytest.mark.parametrize("seed", [200, 203, 207])
def test_tree_settle_then_chain_model(layer, seed):
    sc = Scenario(seed, 3000) if layer == "full" else Scenario(seed, 41590, window=W)
    slots = 3100 if layer == "full" else RING
    k, v, path, nxt = tree_model(sc, slots, seed)
    assert nxt == sc.p0 + len(path)
    assert round2_checks(sc, k, v, path, nxt, nxt) == (True, True)
    if len(path) > 1:           # settlement skipped: the path nodes stay at base + node
        k0, v0 = (x.numpy() for x in sc.initial_cache(slots))
        k0, v0 = oracle.ring_append(k0, v0, _bits(sc.r1_k), _bits(sc.r1_v), sc.p0 + np.arange(16), 16)
        if any(node != d for d, node in enumerate(path)):
            k0, v0 = oracle.ring_append(k0, v0, _bits(sc.r2_k), _bits(sc.r2_v), nxt + np.arange(N_ROWS), N_ROWS)
            assert round2_checks(sc, k0, v0, path, nxt, nxt) == (False, False)
    k, v, path, nxt = tree_model(sc, slots, seed, next_pos_shift=1)
    assert round2_checks(sc, k, v, path, sc.p0 + len(path), nxt) == (False, False)
