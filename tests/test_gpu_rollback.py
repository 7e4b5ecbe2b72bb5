"""Two speculative rounds through the CUDA library: windows stay valid after partial acceptance.

IQuestRT report, "Include sampling and acceptance in the execution path" (acceptance and KV rollback are
part of the step), "Keep the request loop on the GPU" (the step settles the caches; positions stay on the
device) and "Let correctness checks change the design" (the 4,160-slot sliding-window ring).

Round 1: verify_attn_step appends the committed row and 7 drafts at P0 .. P0 + 7 and verifies them (or, for
a tree, kv_ring_append + verify_attn_tree + attn_split_combine over 16 nodes); va_accept_chain accepts
exactly k drafts (or va_tree_accept_settle walks the tree and moves the accepted path) and writes next_pos
on the device; round 2's positions are next_pos + r, built on the device; verify_attn_step appends round 2's
rows over the rejected drafts' slots and verifies.  Checked against the oracle over the linear history of
the accepted tokens only: round 1's and round 2's outputs and LSEs within the parity bars, the acceptance
count and next position exactly, and the cache bytes of every position a round-2 row can see bit for bit.
tests/test_rollback_model.py shows on the CPU that these checks fail for next_pos off by one, a ring one
slot short of W + n - 1, and a tree whose settlement is skipped.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from rollback_cases import N_DRAFTS, N_ROWS, Scenario, forced_chain_acceptance, ring_view
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
W, RING = synth.WINDOW, synth.RING_SLOTS


def _dev(t):
    return synth.bits(t).contiguous().to(DEV) if t.dtype == torch.bfloat16 else t.contiguous().to(DEV)


def _check_out(out, out_lse, ref, n):
    got = oracle.bf16_bits_to_f64(out.cpu().numpy())
    rb = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(ref["out"]))
    m = parity.out_metrics(got, rb, n, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(out_lse.cpu().numpy()[:n], ref["lse"][:n]) <= parity.LSE_ABS


def _step(sc, q, kn, vn, k, v, slots, pos_dev, n_splits, status):
    ws = torch.zeros(va.va_workspace_bytes(n_splits) // 4, dtype=torch.float32, device=DEV)
    out = torch.full((N_ROWS, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    lse = torch.full((N_ROWS, 6), float("nan"), dtype=torch.float32, device=DEV)
    va.verify_attn_step(q, kn, vn, N_ROWS, k, v, pos_dev, sc.scale, _dev(sc.sink), ws, out, lse, window=sc.window,
                        n_splits=n_splits, dev_status=status)
    return out, lse


def _round2(sc, k, v, slots, accepted_rows, nxt_dev, n_splits, status):
    pos2 = nxt_dev + torch.arange(N_ROWS, dtype=torch.int32, device=DEV)   # the next round's positions
    out, lse = _step(sc, _dev(sc.q2), _dev(sc.r2_k), _dev(sc.r2_v), k, v, slots, pos2, n_splits, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"
    nxt = int(nxt_dev.item())
    assert nxt == sc.p0 + len(accepted_rows)
    hk, hv = (x.numpy() for x in sc.history_round2(accepted_rows, nxt))
    p2 = nxt + np.arange(N_ROWS)
    ref = oracle.verify_attn(synth.bits(sc.q2).numpy(), hk, hv, p2, N_ROWS, sc.sink.numpy(), sc.scale, sc.window,
                             n_threads=8)
    _check_out(out, lse, ref, N_ROWS)
    lo, hi = oracle.read_extent(p2, N_ROWS, sc.window)
    vk, vv = ring_view(k.cpu().numpy(), v.cpu().numpy(), hi)
    assert np.array_equal(vk[lo:hi], hk[lo:hi]) and np.array_equal(vv[lo:hi], hv[lo:hi])


def _case(layer, seed):
    if layer == "full":
        return Scenario(seed, 3000), 3100
    if layer == "ring":
        return Scenario(seed, 40000, window=W), RING
    return Scenario(seed, 10 * RING - 4, window=W), RING   # round 1 straddles the end of the ring


@pytest.mark.parametrize("k_accept", range(N_DRAFTS + 1))
@pytest.mark.parametrize("layer", ["full", "ring", "ring_wrap"])
def test_chain_accept_then_next_round(layer, k_accept):
    sc, slots = _case(layer, 100 + k_accept)
    k0, v0 = sc.initial_cache(slots)
    k, v = k0.to(DEV), v0.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    n_splits = 5
    # round 1: the committed row and 7 drafts
    pos1 = (sc.p0 + torch.arange(N_ROWS, dtype=torch.int32)).to(DEV)
    out1, lse1 = _step(sc, _dev(sc.q1[:N_ROWS]), _dev(sc.r1_k[:N_ROWS]), _dev(sc.r1_v[:N_ROWS]), k, v, slots, pos1,
                       n_splits, status)
    h1k, h1v = (x.numpy() for x in sc.history_round1())
    ref1 = oracle.verify_attn(synth.bits(sc.q1[:N_ROWS]).numpy(), h1k, h1v, pos1.cpu().numpy(), N_ROWS,
                              sc.sink.numpy(), sc.scale, sc.window, n_threads=8)
    torch.cuda.synchronize()
    _check_out(out1, lse1, ref1, N_ROWS)
    # acceptance of exactly k_accept drafts; next_pos stays on the device
    a = {name: _dev(t) for name, t in forced_chain_acceptance(k_accept).items()}
    n_acc = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    toks = torch.full((N_DRAFTS + 1,), -7, dtype=torch.int32, device=DEV)
    nxt = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    va.va_accept_chain(a["p_ids"], a["p_probs"], a["p_counts"], a["q_ids"], a["q_probs"], a["q_counts"], a["drafts"],
                       a["target"], N_DRAFTS, a["u_accept"], a["u_replace"], pos1[:1], n_acc, toks, nxt)
    torch.cuda.synchronize()
    assert int(n_acc.item()) == k_accept
    # round 2 from next_pos, over the rejected drafts' slots
    _round2(sc, k, v, slots, list(range(k_accept + 1)), nxt, n_splits, status)


@pytest.mark.parametrize("layer", ["full", "ring", "ring_wrap"])
@pytest.mark.parametrize("seed", [200, 203, 207])
def test_tree_settle_then_next_round(layer, seed):
    sc, slots = _case(layer, seed)
    parents, tokens, target = synth.tree_round(seed)
    k0, v0 = sc.initial_cache(slots)
    k, v = k0.to(DEV), v0.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    masks = synth.ancestor_masks(parents, 16)
    tree = torch.cat([torch.tensor([sc.p0], dtype=torch.int32), masks]).to(DEV)
    # round 1: the 16 nodes appended at base .. base + 15, verified with their ancestor masks
    va.kv_ring_append(_dev(sc.r1_k), _dev(sc.r1_v), 16, k, v, (sc.p0 + torch.arange(16, dtype=torch.int32)).to(DEV),
                      dev_status=status)
    S = 4
    part_o = torch.empty(S, 16, 6, 128, dtype=torch.float32, device=DEV)
    part_lse = torch.empty(S, 16, 6, dtype=torch.float32, device=DEV)
    va.verify_attn_tree(_dev(sc.q1), 16, k, v, tree, sc.scale, part_o, part_lse, window=sc.window, n_splits=S,
                        dev_status=status)
    out1 = torch.empty(16, 6, 128, dtype=torch.int16, device=DEV)
    lse1 = torch.empty(16, 6, dtype=torch.float32, device=DEV)
    va.attn_split_combine(part_o, part_lse, S, _dev(sc.sink), 16, out1, lse1)
    h1k, h1v = (x.numpy() for x in sc.history_round1(16))
    ref1 = oracle.verify_attn_tree(synth.bits(sc.q1).numpy(), h1k, h1v, sc.p0, masks.numpy(), 16, sc.sink.numpy(),
                                   sc.scale, window=sc.window)
    torch.cuda.synchronize()
    _check_out(out1, lse1, ref1, 16)
    # acceptance walk and settlement of the accepted path; next_pos on the device
    path = torch.full((16,), -7, dtype=torch.int32, device=DEV)
    emitted = torch.full((16,), -7, dtype=torch.int32, device=DEV)
    n_acc = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    nxt = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    va.va_tree_accept_settle(k, v, tree, 16, tokens.to(DEV), target.to(DEV), path, emitted, n_acc, nxt, status)
    torch.cuda.synchronize()
    L = int(n_acc.item()) + 1
    accepted = path.cpu().numpy().tolist()[:L]
    _round2(sc, k, v, slots, accepted, nxt, 5, status)
