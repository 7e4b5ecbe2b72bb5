"""GPU parity of tree verification (verify_attn_tree) against the FP64 tree oracle.

"Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees": a 16-node draft tree
is verified in one pass under its tree attention mask.  The nodes' K/V are appended at slots
base .. base + n_nodes - 1 with kv_ring_append, then verify_attn_tree + attn_split_combine run through
the C ABI.  Same bars as the chain parity tests (tests/parity.py).  Cache slots the kernels must not
use hold NaN (full cache) or finite sentinels (ring).
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from gpu_cases import DEV
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu


def _caches(w: synth.TreeWorkload):
    """Device caches holding the committed prefix [0, base); node slots are left for the append."""
    kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
    if w.window == 0:
        k = torch.full((w.slots, 128), synth.BF16_NAN, dtype=torch.int16)
        v = torch.full((w.slots, 128), synth.BF16_NAN, dtype=torch.int16)
        k[:w.base] = kb[:w.base]
        v[:w.base] = vb[:w.base]
    else:
        k = torch.full((w.slots, 128), synth.BF16_K_SENTINEL, dtype=torch.int16)
        v = torch.full((w.slots, 128), synth.BF16_V_SENTINEL, dtype=torch.int16)
        first = max(0, w.base - w.slots)
        p = torch.arange(first, w.base)
        k[p % w.slots] = kb[first:w.base]
        v[p % w.slots] = vb[first:w.base]
    return k.to(DEV), v.to(DEV)


def run_tree(w: synth.TreeWorkload, n_splits: int = 0, tree=None, append: bool = True):
    k, v = _caches(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if append and w.n_nodes > 0:
        idx = torch.arange(w.base, w.base + w.n_nodes)
        va.kv_ring_append(synth.bits(w.k_hist)[idx].contiguous().to(DEV),
                          synth.bits(w.v_hist)[idx].contiguous().to(DEV), w.n_nodes, k, v,
                          w.node_pos.to(DEV), dev_status=status)
    tree_dev = (w.tree if tree is None else tree).to(DEV)
    q = synth.bits(w.q).to(DEV)
    S = n_splits
    # the auto policy never picks more splits than the device has SMs
    cap = S if S else torch.cuda.get_device_properties(0).multi_processor_count
    part_o = torch.full((cap, w.n_rows, 6, 128), float("nan"), dtype=torch.float32, device=DEV)
    part_lse = torch.full((cap, w.n_rows, 6), float("nan"), dtype=torch.float32, device=DEV)
    used = va.verify_attn_tree(q, w.n_nodes, k, v, tree_dev, w.scale, part_o, part_lse, window=w.window,
                               n_splits=S, dev_status=status)
    assert used >= 1 and (S == 0 or used == S)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), dtype=torch.float32, device=DEV)
    va.attn_split_combine(part_o[:used], part_lse[:used], used, w.sink.to(DEV), w.n_nodes, out, out_lse)
    torch.cuda.synchronize()
    return dict(out=oracle.bf16_bits_to_f64(out.cpu().numpy()), out_bits=out.cpu().numpy().view(np.uint16),
                out_lse=out_lse.cpu().numpy().astype(np.float64),
                part_o=part_o[:used].cpu().numpy().astype(np.float64),
                part_lse=part_lse[:used].cpu().numpy().astype(np.float64), n_splits=used,
                status=int(status.item()))


def expected_tree(w: synth.TreeWorkload, n_splits: int):
    res = oracle.verify_attn_tree(synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(),
                                  synth.bits(w.v_hist).numpy(), w.base, w.masks.numpy(), w.n_nodes,
                                  w.sink.numpy(), w.scale, window=w.window, n_splits=n_splits, n_threads=8)
    res["out_bf16"] = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(res["out"]))
    return res


def _assert_parity(got, ref, w):
    assert got["status"] == 0, f"device status {got['status']:#x}"
    n = w.n_nodes
    m = parity.out_metrics(got["out"], ref["out_bf16"], n, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:n], ref["lse"][:n]) <= parity.LSE_ABS
    assert np.all(got["out_bits"][n:] == 0) and np.all(np.isneginf(got["out_lse"][n:]))
    assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS
    assert np.abs(got["part_o"] - ref["part_o"]).max() <= parity.OUT_MAX_ABS
    return m


@pytest.mark.parametrize("S", [1, 3, 4, 7, 17, 40])
def test_tree16_small_context_split_counts(S):
    w = synth.make_tree("t1k", 61, base=1000, n_nodes=16)
    got = run_tree(w, n_splits=S)
    _assert_parity(got, expected_tree(w, S), w)


@pytest.mark.parametrize("n_nodes,n_rows", [(1, 16), (5, 16), (8, 8), (8, 16), (9, 16), (12, 16), (16, 16),
                                            (3, 4), (0, 16)])
def test_tree_node_counts_and_padding(n_nodes, n_rows):
    w = synth.make_tree(f"tn{n_nodes}", 62 + n_nodes, base=2077, n_nodes=max(n_nodes, 1), n_rows=n_rows)
    if n_nodes == 0:
        w.parents = []
        w.masks = torch.zeros(n_rows, dtype=torch.int32)
    got = run_tree(w, n_splits=9)
    if n_nodes == 0:
        assert got["status"] == 0
        assert np.all(got["out_bits"] == 0) and np.all(np.isneginf(got["out_lse"]))
        assert np.all(np.isneginf(got["part_lse"])) and np.all(got["part_o"] == 0)
        return
    _assert_parity(got, expected_tree(w, 9), w)


@pytest.mark.parametrize("shape", ["chain", "star", "best_first"])
def test_tree_shapes_16k_auto_splits(shape):
    w = synth.make_tree(f"t16k_{shape}", 70, base=16384 - 16, n_nodes=16, shape=shape, slots=65536)
    got = run_tree(w, n_splits=0)
    _assert_parity(got, expected_tree(w, got["n_splits"]), w)


def test_chain_tree_matches_chain_kernel_bit_for_bit():
    # a chain of 8 nodes is the causal verify of 8 consecutive rows: same kernel, same plan, same bits
    w = synth.make_tree("tchain", 71, base=5000, n_nodes=8, shape="chain", n_rows=8)
    got = run_tree(w, n_splits=11)
    cw = synth.Workload(name="chain", seed=71, q=w.q, k_hist=w.k_hist, v_hist=w.v_hist, pos=w.node_pos, n_live=8,
                        sink=w.sink, scale=w.scale, window=0, slots=w.slots, n_splits=11, poison_tail=True)
    from gpu_cases import run_step
    chain = run_step(cw, n_splits=11)
    assert chain["status"] == 0 and got["status"] == 0
    assert np.array_equal(got["out_bits"], chain["out_bits"])
    assert np.array_equal(got["part_lse"], chain["part_lse"])


@pytest.mark.parametrize("base", [39984, 4096 - 16, 100, 4160 * 3 + 30])
def test_tree_sliding_window_ring(base):
    w = synth.make_tree(f"tswa{base}", 72, base=base, n_nodes=16, window=synth.WINDOW, slots=synth.RING_SLOTS)
    got = run_tree(w, n_splits=0)
    _assert_parity(got, expected_tree(w, got["n_splits"]), w)


def test_tree_192k_all_nodes():
    w = synth.tree_192k()
    got = run_tree(w, n_splits=0)
    _assert_parity(got, expected_tree(w, got["n_splits"]), w)


def test_tree_bad_mask_sets_status_and_writes_empty_partials():
    w = synth.make_tree("tbad", 73, base=500, n_nodes=6, n_rows=8)
    bad = w.tree.clone()
    bad[1 + 3] &= ~(1 << 3)     # node 3 without its own bit
    got = run_tree(w, n_splits=4, tree=bad)
    assert got["status"] & 32
    assert np.all(np.isneginf(got["part_lse"])) and np.all(got["part_o"] == 0)
    bad = w.tree.clone()
    bad[1 + 2] |= 1 << 7        # a node that does not exist
    got = run_tree(w, n_splits=4, tree=bad)
    assert got["status"] & 32


def test_tree_beyond_cache_sets_status():
    w = synth.make_tree("tbeyond", 74, base=500, n_nodes=6, n_rows=8)
    bad = w.tree.clone()
    bad[0] = w.slots - 3        # nodes would run past the capacity
    got = run_tree(w, n_splits=4, tree=bad, append=False)
    assert got["status"] & 4
