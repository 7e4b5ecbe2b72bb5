"""Seeded synthetic inputs for verify attention.

This module only draws numbers and lays down the workload recipes (shapes, seeds,
positions, value distributions).  It holds none of the attention arithmetic, so the
CUDA path and the CPU oracle can both be fed from it without sharing any method code.

Recipes (IQuestRT technical report: 8 verify rows x 6 query heads per KV head,
head_dim 128, 1K-192K context sweep with synthetic KV, sliding window 4,096 in a
4,160-slot ring):

  tiny      capacity 1,024, rows at positions 1016..1023, 5 live rows, 4 splits
  16k       capacity 65,536, 16,384 valid positions, 8 live rows, 5 % of keys x4
  swa       window 4,096, ring 4,160, context 40,000 (ring wrapped), 7 live rows
  192k      196,608 positions (about 100 MB of K/V), n_live 4..8
  sweep     {1K,4K,16K,32K,64K,128K,192K} x {full, swa} x n_live 4..8
  trees     16-node draft trees grown best-first ("Qwen3.8-27B on one RTX 4090", section "More
            tokens per round: verify trees"), verified at the same contexts; node i at slot base + i

Q, K, V ~ N(0, 1) drawn in float32 by a seeded CPU torch generator and rounded to
bf16; sink ~ N(0, 1) float32; scale = 1/sqrt(128).
"""
from __future__ import annotations

import dataclasses
import math

import torch

HEAD_DIM = 128
Q_HEADS = 6
N_ROWS = 8
SCALE = 1.0 / math.sqrt(128.0)
WINDOW = 4096
RING_SLOTS = 4160
SWEEP_CONTEXTS = (1024, 4096, 16384, 32768, 65536, 131072, 196608)

# bf16 bit patterns used to poison cache slots the kernels must not use
BF16_NAN = 0x7FC0
BF16_K_SENTINEL = 0x4280   # 64.0
BF16_V_SENTINEL = 0x447A   # 1000.0


@dataclasses.dataclass
class Workload:
    """One verify call.  Tensors are CPU tensors; bf16 data is stored as torch.bfloat16."""
    name: str
    seed: int
    q: torch.Tensor            # [n_rows, 6, 128] bf16
    k_hist: torch.Tensor       # [ctx, 128] bf16, row j = absolute position j
    v_hist: torch.Tensor       # [ctx, 128] bf16
    pos: torch.Tensor          # [n_rows] int32, 0-based absolute positions
    n_live: int
    sink: torch.Tensor         # [6] float32
    scale: float
    window: int                # 0 = full attention
    slots: int                 # full: cache capacity; swa: ring slots
    n_splits: int              # 0 = auto
    poison_tail: bool = True   # full cache: slots at and beyond the valid extent hold NaN

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def ctx(self) -> int:
        return int(self.k_hist.shape[0])


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, g: torch.Generator, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def tail_positions(ctx: int, n_live: int, n_rows: int = N_ROWS) -> torch.Tensor:
    """Rows at the end of the context: pos[r] = ctx - n_live + r (padding rows continue past it)."""
    return torch.tensor([ctx - n_live + r for r in range(n_rows)], dtype=torch.int32)


def make(name: str, seed: int, ctx: int, n_live: int, window: int = 0, slots: int = 0,
         n_splits: int = 0, peaky_frac: float = 0.0, pos: torch.Tensor | None = None,
         n_rows: int = N_ROWS, poison_tail: bool = True) -> Workload:
    """Draw one workload.  `ctx` positions of history are generated (the live rows' own K/V
    included, at their positions)."""
    g = generator(seed)
    q = normal_bf16((n_rows, Q_HEADS, HEAD_DIM), g)
    k = torch.randn(ctx, HEAD_DIM, generator=g, dtype=torch.float32)
    if peaky_frac > 0.0:
        n_peaky = int(round(peaky_frac * ctx))
        idx = torch.randperm(ctx, generator=g)[:n_peaky]
        k[idx] *= 4.0
    k = k.to(torch.bfloat16)
    v = normal_bf16((ctx, HEAD_DIM), g)
    sink = torch.randn(Q_HEADS, generator=g, dtype=torch.float32)
    if pos is None:
        pos = tail_positions(ctx, n_live, n_rows)
    if slots <= 0:
        slots = RING_SLOTS if window > 0 else ctx
    return Workload(name=name, seed=seed, q=q, k_hist=k, v_hist=v, pos=pos.to(torch.int32), n_live=n_live,
                    sink=sink, scale=SCALE, window=window, slots=slots, n_splits=n_splits,
                    poison_tail=poison_tail)


def tiny(poison_tail: bool = False) -> Workload:
    """Context 1,024, rows at 1-based positions 1017..1024 (0-based 1016..1023), 5 live, 4 splits."""
    pos = torch.arange(1016, 1024, dtype=torch.int32)
    return make("tiny", 1, ctx=1024, n_live=5, slots=1024, n_splits=4, pos=pos, poison_tail=poison_tail)


def full_16k() -> Workload:
    """Capacity 65,536, 16,384 valid positions, 8 live rows at the tail, 5 % of keys x4."""
    w = make("16k", 2, ctx=16384, n_live=8, slots=65536, n_splits=0, peaky_frac=0.05)
    return w


def swa_40k() -> Workload:
    """Window 4,096 in a 4,160-slot ring at absolute context 40,000; 7 live rows at 39,993..39,999."""
    pos = torch.tensor([39993 + r for r in range(N_ROWS)], dtype=torch.int32)
    return make("swa", 3, ctx=40000, n_live=7, window=WINDOW, slots=RING_SLOTS, n_splits=0, pos=pos)


def full_192k(n_live: int) -> Workload:
    """196,608 positions, capacity 196,672 (NaN tail), rows at the tail."""
    return make(f"192k_n{n_live}", 4 + n_live, ctx=196608, n_live=n_live, slots=196672, n_splits=0)


def sweep_points():
    """(index, ctx, window, n_live) of the 70 sweep points."""
    pts = []
    idx = 0
    for ctx in SWEEP_CONTEXTS:
        for window in (0, WINDOW):
            for n_live in (4, 5, 6, 7, 8):
                pts.append((idx, ctx, window, n_live))
                idx += 1
    return pts


def sweep(idx: int, ctx: int, window: int, n_live: int) -> Workload:
    slots = RING_SLOTS if window > 0 else ctx + 64
    kind = "swa" if window > 0 else "full"
    return make(f"sweep_{kind}_{ctx}_n{n_live}", 100 + idx, ctx=ctx, n_live=n_live, window=window,
                slots=slots, n_splits=0)


# ----------------------------------------------------------------------------- draft trees
TREE_NODES = 16
TREE_TEMPERATURE = 1.25


def best_first_tree(g: torch.Generator, n_nodes: int, branch: int = 4, temperature: float = TREE_TEMPERATURE):
    """Parent array of a synthetic draft tree grown best-first: every node offers `branch` candidate
    children whose probabilities are a softmax of N(0, 2) logits divided by `temperature`; the candidate
    with the highest path probability joins the tree next.  parents[0] = -1, parents[i] < i."""
    parents = [-1]
    path_logp = [0.0]
    frontier = []   # (path log-probability, parent)

    def offer(node):
        logits = torch.randn(branch, generator=g, dtype=torch.float64) * 2.0 / temperature
        logp = torch.log_softmax(logits, dim=0)
        for c in range(branch):
            frontier.append((path_logp[node] + float(logp[c]), node))

    offer(0)
    while len(parents) < n_nodes:
        best = max(range(len(frontier)), key=lambda i: frontier[i][0])
        lp, par = frontier.pop(best)
        parents.append(par)
        path_logp.append(lp)
        offer(len(parents) - 1)
    return parents


def chain_parents(n_nodes: int):
    return [i - 1 for i in range(n_nodes)]


def star_parents(n_nodes: int):
    return [-1] + [0] * (n_nodes - 1)


def ancestor_masks(parents, n_rows: int = TREE_NODES) -> torch.Tensor:
    """[n_rows] int32: bit k of entry i set iff node k is node i or one of its ancestors (0 past the nodes)."""
    m = [0] * n_rows
    for i, par in enumerate(parents):
        m[i] = (1 << i) | (m[par] if par >= 0 else 0)
    return torch.tensor(m, dtype=torch.int32)


@dataclasses.dataclass
class TreeWorkload:
    """One tree verify call: nodes 0..n_nodes-1 at slots base..base+n_nodes-1 (their K/V are the last
    n_nodes rows of the history); rows n_nodes..n_rows-1 are padding."""
    name: str
    seed: int
    q: torch.Tensor            # [n_rows, 6, 128] bf16
    k_hist: torch.Tensor       # [base + n_nodes, 128] bf16
    v_hist: torch.Tensor
    base: int
    parents: list
    masks: torch.Tensor        # [n_rows] int32 ancestor-or-self masks
    sink: torch.Tensor
    scale: float
    window: int
    slots: int
    n_splits: int

    @property
    def n_nodes(self) -> int:
        return len(self.parents)

    @property
    def n_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def ctx(self) -> int:
        return int(self.k_hist.shape[0])

    @property
    def node_pos(self) -> torch.Tensor:
        """[n_rows] int32 slots of the nodes (padding rows continue past them), for the append."""
        return torch.tensor([self.base + i for i in range(self.n_rows)], dtype=torch.int32)

    @property
    def tree(self) -> torch.Tensor:
        """[1 + n_rows] int32: base, then the masks (the verify call's tree descriptor)."""
        return torch.cat([torch.tensor([self.base], dtype=torch.int32), self.masks])


def make_tree(name: str, seed: int, base: int, n_nodes: int = TREE_NODES, shape: str = "best_first",
              window: int = 0, slots: int = 0, n_splits: int = 0, n_rows: int = TREE_NODES) -> TreeWorkload:
    g = generator(seed)
    q = normal_bf16((n_rows, Q_HEADS, HEAD_DIM), g)
    ctx = base + n_nodes
    k = normal_bf16((ctx, HEAD_DIM), g)
    v = normal_bf16((ctx, HEAD_DIM), g)
    sink = torch.randn(Q_HEADS, generator=g, dtype=torch.float32)
    if shape == "best_first":
        parents = best_first_tree(g, n_nodes)
    elif shape == "chain":
        parents = chain_parents(n_nodes)
    elif shape == "star":
        parents = star_parents(n_nodes)
    else:
        raise ValueError(shape)
    if slots <= 0:
        slots = RING_SLOTS if window > 0 else ctx + 64
    return TreeWorkload(name=name, seed=seed, q=q, k_hist=k, v_hist=v, base=base, parents=parents,
                        masks=ancestor_masks(parents, n_rows), sink=sink, scale=SCALE, window=window, slots=slots,
                        n_splits=n_splits)


def tree_192k(n_nodes: int = TREE_NODES, shape: str = "best_first") -> TreeWorkload:
    """A 16-node tree whose last slot is position 196,607: the same 196,608-position extent as the
    192K chain workload."""
    return make_tree(f"tree192k_{shape}_n{n_nodes}", 20 + n_nodes, base=196608 - n_nodes, n_nodes=n_nodes,
                     shape=shape, slots=196672)


# ----------------------------------------------------------------------------- sampling inputs
VOCAB = 160000


def logits(seed: int, n_rows: int, vocab: int = VOCAB, head: int = 40) -> torch.Tensor:
    """[n_rows, vocab] float32 logits: N(0, 2) everywhere plus a head of `head` tokens per row raised by
    U(6, 14), so that top-k 20 / top-p 0.95 cut inside a realistic peaked distribution."""
    g = generator(seed)
    x = torch.randn(n_rows, vocab, generator=g, dtype=torch.float32) * 2.0
    for r in range(n_rows):
        idx = torch.randperm(vocab, generator=g)[:head]
        x[r, idx] += 6.0 + 8.0 * torch.rand(head, generator=g)
    return x


def uniforms(seed: int, n: int) -> torch.Tensor:
    """n float32 uniforms in [0, 1)."""
    return torch.rand(n, generator=generator(seed), dtype=torch.float32)


def sparse_distribution(g: torch.Generator, k: int, support, boost=None):
    """A distribution over k distinct token ids drawn from `support`, probabilities from exp(N(0, 1.5))
    (optionally raised on `boost` ids), sorted descending.  Returns (ids int32 [k], probs float32 [k])."""
    support = torch.as_tensor(support)
    ids = support[torch.randperm(support.numel(), generator=g)[:k]]
    w = torch.exp(torch.randn(k, generator=g, dtype=torch.float64) * 1.5)
    if boost is not None:
        for b in boost:
            w[ids == int(b)] *= 4.0
    order = torch.argsort(-w, stable=True)
    ids, w = ids[order], w[order]
    return ids.to(torch.int32), (w / w.sum()).to(torch.float32)


def chain_round(seed: int, n_drafts: int, k: int = 20, vocab_span: int = 60):
    """Synthetic inputs of one chain acceptance: per verify row r a target distribution p_r, per draft
    i a proposal distribution q_i (overlapping p_{i-1}'s ids), the draft token d_i drawn from q_i, the
    uniforms and the target's own draw per row.  Distributions are padded to k entries (-1 / 0)."""
    g = generator(seed)
    rows = n_drafts + 1
    p_ids = torch.full((rows, k), -1, dtype=torch.int32)
    p_pr = torch.zeros(rows, k, dtype=torch.float32)
    q_ids = torch.full((rows, k), -1, dtype=torch.int32)
    q_pr = torch.zeros(rows, k, dtype=torch.float32)
    p_cnt = torch.zeros(rows, dtype=torch.int32)
    q_cnt = torch.zeros(rows, dtype=torch.int32)
    drafts = torch.zeros(rows, dtype=torch.int32)
    target = torch.zeros(rows, dtype=torch.int32)
    drafts[0] = 7
    for r in range(rows):
        kp = int(torch.randint(1, k + 1, (1,), generator=g))
        ids, pr = sparse_distribution(g, kp, torch.arange(vocab_span))
        p_ids[r, :kp], p_pr[r, :kp], p_cnt[r] = ids, pr, kp
        target[r] = int(ids[int(torch.multinomial(pr.double(), 1, generator=g))])
    for i in range(1, rows):
        kq = int(torch.randint(1, k + 1, (1,), generator=g))
        ids, pr = sparse_distribution(g, kq, torch.arange(vocab_span), boost=p_ids[i - 1, :2].tolist())
        q_ids[i, :kq], q_pr[i, :kq], q_cnt[i] = ids, pr, kq
        drafts[i] = int(ids[int(torch.multinomial(pr.double(), 1, generator=g))])
    return dict(p_ids=p_ids, p_pr=p_pr, p_cnt=p_cnt, q_ids=q_ids, q_pr=q_pr, q_cnt=q_cnt, drafts=drafts,
                target=target, u_accept=torch.rand(rows, generator=g), u_replace=torch.rand(1, generator=g),
                pos=torch.tensor([int(torch.randint(0, 1 << 20, (1,), generator=g))], dtype=torch.int32))


def tree_round(seed: int, n_nodes: int = TREE_NODES, follow: float = 0.75, vocab_span: int = 1000):
    """Synthetic inputs of one tree acceptance: a best-first tree, distinct sibling tokens, and at each
    node a target token that equals one of its children's tokens with probability `follow`."""
    g = generator(seed)
    parents = best_first_tree(g, n_nodes)
    tokens = torch.randperm(vocab_span, generator=g)[:n_nodes].to(torch.int32)
    target = torch.zeros(n_nodes, dtype=torch.int32)
    for v in range(n_nodes):
        kids = [c for c in range(n_nodes) if parents[c] == v]
        if kids and float(torch.rand(1, generator=g)) < follow:
            target[v] = tokens[kids[int(torch.randint(0, len(kids), (1,), generator=g))]]
        else:
            target[v] = vocab_span + v   # a token no child carries
    return parents, tokens, target


def random_partials(seed: int, n_splits: int, n_rows: int, n_live: int, empty_frac: float = 0.1):
    """Synthetic split partials for testing the merge on its own: o ~ N(0,1) fp32,
    lse ~ N(0, 3) fp32 with a fraction set to -inf (empty splits), sink ~ N(0, 1)."""
    g = generator(seed)
    part_o = torch.randn(n_splits, n_rows, Q_HEADS, HEAD_DIM, generator=g, dtype=torch.float32)
    part_lse = torch.randn(n_splits, n_rows, Q_HEADS, generator=g, dtype=torch.float32) * 3.0
    empty = torch.rand(n_splits, n_rows, Q_HEADS, generator=g) < empty_frac
    part_lse[empty] = float("-inf")
    part_o[empty] = 0.0
    sink = torch.randn(Q_HEADS, generator=g, dtype=torch.float32)
    return part_o, part_lse, sink


def bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor -> its int16 bit patterns (same storage size)."""
    return t.contiguous().view(torch.int16)
