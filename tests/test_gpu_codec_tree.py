"""GPU parity of tree verification over the quantised K/V cache (verify_attn_q8_tree) against the FP64
tree oracle over the decoded cache.

"Qwen3.8-27B on one RTX 4090": the 16-node verify trees of section "More tokens per round: verify trees"
read the cache of section "A cheaper cache and state".  The committed prefix is encoded on the host by the
oracle's encoder (the append kernel matches it bit for bit, tests/test_gpu_codec.py), the nodes' K/V are
encoded into slots base .. base + n_nodes - 1 by kv_ring_append_q8, then verify_attn_q8_tree +
attn_split_combine run through the C ABI.  Bars as for the bf16 path (tests/parity.py), against the
oracle's attention over the decoded keys and values rounded once to bf16.  Slots the kernel must not use
hold NaN codes and NaN scales.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from oracle import kv_codec as C
from speculative_decode_verify_gb300 import synth
from test_gpu_codec import DEV, _encoded_cache, run_q8

pytestmark = pytest.mark.gpu


def run_q8_tree(w: synth.TreeWorkload, n_splits: int = 0, tree=None):
    w.slots = -(-w.slots // 64) * 64   # the quantised cache holds a multiple of 64 slots
    kc, vc, ks, vs = _encoded_cache(w, w.slots, w.base)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if w.n_nodes > 0:
        idx = torch.arange(w.base, w.base + w.n_nodes)
        va.kv_ring_append_q8(synth.bits(w.k_hist)[idx].contiguous().to(DEV),
                             synth.bits(w.v_hist)[idx].contiguous().to(DEV), w.n_nodes, kc, vc, ks, vs,
                             w.node_pos.to(DEV), dev_status=status)
    cap = n_splits if n_splits else torch.cuda.get_device_properties(0).multi_processor_count
    part_o = torch.full((cap, w.n_rows, 6, 128), float("nan"), device=DEV)
    part_lse = torch.full((cap, w.n_rows, 6), float("nan"), device=DEV)
    used = va.verify_attn_q8_tree(synth.bits(w.q).to(DEV), w.n_nodes, kc, vc, ks, vs,
                                  (w.tree if tree is None else tree).to(DEV), w.scale, part_o, part_lse,
                                  window=w.window, n_splits=n_splits, dev_status=status)
    assert used >= 1 and (n_splits == 0 or used == n_splits)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), device=DEV)
    va.attn_split_combine(part_o[:used], part_lse[:used], used, w.sink.to(DEV), w.n_nodes, out, out_lse)
    torch.cuda.synchronize()
    return dict(out=oracle.bf16_bits_to_f64(out.cpu().numpy()), out_bits=out.cpu().numpy().view(np.uint16),
                out_lse=out_lse.cpu().numpy().astype(np.float64),
                part_o=part_o[:used].cpu().numpy().astype(np.float64),
                part_lse=part_lse[:used].cpu().numpy().astype(np.float64), n_splits=used,
                status=int(status.item()))


def expected_q8_tree(w: synth.TreeWorkload, n_splits: int):
    kcodes, kscale = C.encode_k(synth.bits(w.k_hist).numpy())
    vcodes, vscale = C.encode_v(synth.bits(w.v_hist).numpy())
    res = C.verify_attn_tree_decoded(synth.bits(w.q).numpy(), C.decode_k(kcodes, kscale),
                                     C.decode_v(vcodes, vscale), w.base, w.masks.numpy(), w.n_nodes, w.sink.numpy(),
                                     w.scale, window=w.window, n_splits=n_splits, n_threads=8)
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
def test_q8_tree16_small_context_split_counts(S):
    w = synth.make_tree("q8t1k", 161, base=1000, n_nodes=16)
    _assert_parity(run_q8_tree(w, S), expected_q8_tree(w, S), w)


@pytest.mark.parametrize("n_nodes,n_rows", [(1, 16), (5, 16), (8, 8), (8, 16), (9, 16), (12, 16), (16, 16),
                                            (3, 4), (0, 16)])
def test_q8_tree_node_counts_and_padding(n_nodes, n_rows):
    w = synth.make_tree(f"q8tn{n_nodes}", 162 + n_nodes, base=2077, n_nodes=max(n_nodes, 1), n_rows=n_rows)
    if n_nodes == 0:
        w.parents = []
        w.masks = torch.zeros(n_rows, dtype=torch.int32)
    got = run_q8_tree(w, n_splits=9)
    if n_nodes == 0:
        assert got["status"] == 0
        assert np.all(got["out_bits"] == 0) and np.all(np.isneginf(got["out_lse"]))
        assert np.all(np.isneginf(got["part_lse"])) and np.all(got["part_o"] == 0)
        return
    _assert_parity(got, expected_q8_tree(w, 9), w)


@pytest.mark.parametrize("shape", ["chain", "star", "best_first"])
def test_q8_tree_shapes_16k_auto_splits(shape):
    w = synth.make_tree(f"q8t16k_{shape}", 170, base=16384 - 16, n_nodes=16, shape=shape, slots=65536)
    got = run_q8_tree(w, n_splits=0)
    _assert_parity(got, expected_q8_tree(w, got["n_splits"]), w)


def test_q8_chain_tree_matches_the_q8_chain_kernel_bit_for_bit():
    # a chain of 8 nodes is the causal verify of 8 consecutive rows: same kernel, same plan, same bits
    w = synth.make_tree("q8tchain", 171, base=5000, n_nodes=8, shape="chain", n_rows=8)
    got = run_q8_tree(w, n_splits=11)
    cw = synth.Workload(name="chain", seed=171, q=w.q, k_hist=w.k_hist, v_hist=w.v_hist, pos=w.node_pos, n_live=8,
                        sink=w.sink, scale=w.scale, window=0, slots=w.slots, n_splits=11, poison_tail=True)
    chain = run_q8(cw, n_splits=11)
    assert chain["status"] == 0 and got["status"] == 0
    assert np.array_equal(got["out_bits"], chain["out_bits"])
    assert np.array_equal(got["part_lse"], chain["part_lse"].astype(np.float64))


@pytest.mark.parametrize("base", [39984, 4096 - 16, 100, 4160 * 3 + 30])
def test_q8_tree_sliding_window_ring(base):
    w = synth.make_tree(f"q8tswa{base}", 172, base=base, n_nodes=16, window=synth.WINDOW, slots=synth.RING_SLOTS)
    got = run_q8_tree(w, n_splits=0)
    _assert_parity(got, expected_q8_tree(w, got["n_splits"]), w)


def test_q8_tree_192k_all_nodes():
    w = synth.tree_192k()
    got = run_q8_tree(w, n_splits=0)
    _assert_parity(got, expected_q8_tree(w, got["n_splits"]), w)


def test_q8_tree_bad_masks_set_status_and_write_empty_partials():
    w = synth.make_tree("q8tbad", 173, base=500, n_nodes=6, n_rows=8)
    bad = w.tree.clone()
    bad[1 + 3] &= ~(1 << 3)     # node 3 without its own bit
    got = run_q8_tree(w, n_splits=4, tree=bad)
    assert got["status"] & 32
    assert np.all(np.isneginf(got["part_lse"])) and np.all(got["part_o"] == 0)
    bad = w.tree.clone()
    bad[1 + 2] |= 1 << 7        # a node that does not exist
    got = run_q8_tree(w, n_splits=4, tree=bad)
    assert got["status"] & 32


def test_q8_tree_rejects_bad_arguments():
    q = torch.zeros(16, 6, 128, dtype=torch.int16, device=DEV)
    kc = torch.zeros(128, 128, dtype=torch.uint8, device=DEV)
    vc = torch.zeros(128, 128, dtype=torch.int8, device=DEV)
    s = torch.zeros(128, device=DEV)
    po = torch.empty(4, 16, 6, 128, device=DEV)
    pl = torch.empty(4, 16, 6, device=DEV)
    tree = torch.tensor([0] + [1 << i for i in range(16)], dtype=torch.int32, device=DEV)
    with pytest.raises(va.VerifyAttnError):      # 17 nodes
        va.verify_attn_q8_tree(torch.zeros(17, 6, 128, dtype=torch.int16, device=DEV), 17, kc, vc, s, s, tree, 0.088,
                               torch.empty(4, 17, 6, 128, device=DEV), torch.empty(4, 17, 6, device=DEV), n_splits=4)
    with pytest.raises(va.VerifyAttnError):      # a window smaller than the tree
        va.verify_attn_q8_tree(q, 16, kc, vc, s, s, tree, 0.088, po, pl, window=8, n_splits=4)
    with pytest.raises(va.VerifyAttnError):      # slots not a multiple of 64
        va.verify_attn_q8_tree(q, 16, kc[:100], vc[:100], s[:100], s[:100], tree, 0.088, po, pl, n_splits=4)
