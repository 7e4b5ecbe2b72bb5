"""Two speculative rounds on one layer's cache: verify, accept part of the drafts, verify the next round.

IQuestRT report, "Include sampling and acceptance in the execution path" (acceptance and KV rollback are
part of the step) and "Keep the request loop on the GPU" (the step settles the caches before the next
round); "Let correctness checks change the design" (a sliding-window ring of 4,096 + 64 slots, because
the next round's rows are written before any row reads its window).

Round 1 verifies the committed token and 7 drafts at positions P0 .. P0 + 7 (their K/V appended first),
then accepts k of the drafts; round 2 verifies 8 new rows from next_pos = P0 + k + 1 on.  Round 2's rows
overwrite the slots of the 7 - k rejected drafts.  The result must equal attention over the linear history
of the ACCEPTED tokens only: positions < P0 from the original history, P0 .. P0 + k round 1's rows 0..k,
then round 2's rows.  For a draft tree, round 1 verifies 16 nodes at base .. base + 15, settlement moves
the accepted path to base .. base + L - 1, and round 2 starts at base + L.

Only the seeded draws and the expected linear histories live here (no attention arithmetic).
"""
import numpy as np
import torch

from speculative_decode_verify_gb300 import synth

N_ROWS = 8
N_DRAFTS = 7


class Scenario:
    """Seeded inputs of a two-round chain (or tree + chain) on one layer."""

    def __init__(self, seed: int, p0: int, window: int = 0):
        self.p0, self.window = p0, window
        g = synth.generator(seed)
        n_hist = p0 + 2 * 16 + 8
        self.k_hist = synth.normal_bf16((n_hist, 128), g)    # positions < p0 are the committed history
        self.v_hist = synth.normal_bf16((n_hist, 128), g)
        self.r1_k = synth.normal_bf16((16, 128), g)           # round 1's rows (8 chain rows or 16 tree nodes)
        self.r1_v = synth.normal_bf16((16, 128), g)
        self.r2_k = synth.normal_bf16((N_ROWS, 128), g)       # round 2's rows
        self.r2_v = synth.normal_bf16((N_ROWS, 128), g)
        self.q1 = synth.normal_bf16((16, 6, 128), g)
        self.q2 = synth.normal_bf16((N_ROWS, 6, 128), g)
        self.sink = torch.randn(6, generator=g, dtype=torch.float32)
        self.scale = synth.SCALE

    def history_round1(self, n1: int = N_ROWS):
        """Linear history seen by round 1 (bf16 bits): the committed history, then round 1's rows."""
        k = synth.bits(self.k_hist[:self.p0 + n1]).clone()
        v = synth.bits(self.v_hist[:self.p0 + n1]).clone()
        k[self.p0:self.p0 + n1] = synth.bits(self.r1_k[:n1])
        v[self.p0:self.p0 + n1] = synth.bits(self.r1_v[:n1])
        return k, v

    def history_round2(self, accepted_rows, next_pos: int):
        """Linear history seen by round 2: the committed history, the accepted round-1 rows (in order, at
        p0, p0 + 1, ..), then round 2's rows from next_pos on."""
        end = next_pos + N_ROWS
        k = torch.zeros(end, 128, dtype=torch.int16)
        v = torch.zeros(end, 128, dtype=torch.int16)
        k[:self.p0] = synth.bits(self.k_hist[:self.p0])
        v[:self.p0] = synth.bits(self.v_hist[:self.p0])
        for d, row in enumerate(accepted_rows):
            k[self.p0 + d] = synth.bits(self.r1_k[row])
            v[self.p0 + d] = synth.bits(self.r1_v[row])
        assert self.p0 + len(accepted_rows) == next_pos
        k[next_pos:end] = synth.bits(self.r2_k)
        v[next_pos:end] = synth.bits(self.r2_v)
        return k, v

    def initial_cache(self, slots: int):
        """The device-side cache before round 1 (bf16 bits, host): history positions < p0 in slot p mod slots
        (a ring keeps the last `slots` of them; other slots hold the finite sentinels K = 64, V = 1000); a full
        cache holds NaN at and beyond p0."""
        if self.window == 0:
            k = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
            v = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
            k[:self.p0] = synth.bits(self.k_hist[:self.p0])
            v[:self.p0] = synth.bits(self.v_hist[:self.p0])
            return k, v
        k = torch.full((slots, 128), synth.BF16_K_SENTINEL, dtype=torch.int16)
        v = torch.full((slots, 128), synth.BF16_V_SENTINEL, dtype=torch.int16)
        first = max(0, self.p0 - slots)
        p = torch.arange(first, self.p0)
        k[p % slots] = synth.bits(self.k_hist[first:self.p0])
        v[p % slots] = synth.bits(self.v_hist[first:self.p0])
        return k, v


def forced_chain_acceptance(k_accept: int, top_k: int = 4):
    """Target / draft distributions and uniforms under which exactly k_accept of the 7 drafts pass the
    rejection test: for i <= k_accept, p_{i-1} and q_i both put all mass on draft i (u q < p holds); draft
    k_accept + 1 is absent from p_{k_accept}, so it fails and the replacement is p's own token 900.
    Returns host tensors (ids/probs/counts of p and q with row stride top_k, drafts, target tokens, uniforms)."""
    drafts = torch.tensor([7] + [100 + i for i in range(1, N_DRAFTS + 1)], dtype=torch.int32)
    p_ids = torch.full((N_ROWS, top_k), -1, dtype=torch.int32)
    p_probs = torch.zeros(N_ROWS, top_k, dtype=torch.float32)
    q_ids = torch.full((N_ROWS, top_k), -1, dtype=torch.int32)
    q_probs = torch.zeros(N_ROWS, top_k, dtype=torch.float32)
    for r in range(N_ROWS):
        nxt = r + 1
        tok = int(drafts[nxt]) if nxt <= k_accept and nxt <= N_DRAFTS else 900 + r
        p_ids[r, 0], p_probs[r, 0] = tok, 1.0
        if 1 <= r <= N_DRAFTS:
            q_ids[r, 0], q_probs[r, 0] = int(drafts[r]), 1.0
    counts = torch.ones(N_ROWS, dtype=torch.int32)
    target = torch.tensor([800 + r for r in range(N_ROWS)], dtype=torch.int32)
    u_accept = torch.full((N_ROWS,), 0.5, dtype=torch.float32)
    u_replace = torch.tensor([0.25], dtype=torch.float32)
    return dict(p_ids=p_ids, p_probs=p_probs, p_counts=counts, q_ids=q_ids, q_probs=q_probs, q_counts=counts.clone(),
                drafts=drafts, target=target, u_accept=u_accept, u_replace=u_replace)


def dists(ids, probs, counts):
    """(ids, probs) lists per row, as oracle.sampling takes them."""
    return [(ids[r, :int(counts[r])].tolist(), probs[r, :int(counts[r])].tolist()) for r in range(ids.shape[0])]


def ring_view(k_ring, v_ring, upto: int):
    """Linear view [0, upto) of what a ring holds for each position: slot p mod slots (only the positions
    still held are meaningful)."""
    slots = k_ring.shape[0]
    idx = np.arange(upto) % slots
    return np.asarray(k_ring)[idx], np.asarray(v_ring)[idx]
