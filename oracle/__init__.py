"""FP64 CPU oracle for speculative-decoding verify attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference arm may import this package.  It shares
no code with the CUDA library (``speculative_decode_verify_gb300``) and imports
nothing from it; the two meet only in the seeded input generator module.

Sources (IQuestRT technical report):
  * section "Read only the KV tiles needed by the current positions": 8 verify rows
    x 6 query heads share one KV head; work is partitioned along the sequence; the
    read extent comes from the current positions, with a causal mask at the
    boundary; the learned sink has a zero value and only enters the denominator;
    sliding-window layers keep a physical ring of the 4,096-position window plus
    one 64-slot tile, and the verify rows are written before they are read.
  * section "Expose more parallelism in attention": split-KV partials are merged
    with their log-sum-exp values; the combine applies the sink correction.
  * section "Let correctness checks change the design": the ring bug was found with
    independent position labels and visible-position sets.

Readings taken where the pages are silent:
  * positions are 0-based; a row at position p sees keys j <= p;
  * the read extent comes from the live rows only: hi = max live position + 1;
  * a sliding window of W covers [p - W + 1, p] for a row at p;
  * the sink is a logit in the post-scale score domain, natural-log LSE;
  * sequence splits are made of 64-position tiles aligned to absolute position;
    with T tiles between the extent's first and last tile, split s takes tiles
    [t_lo + floor(s*T/S), t_lo + floor((s+1)*T/S));
  * partials are normalised (o_s) with a natural-log lse_s; empty -> 0 / -inf;
  * padding rows and rows with nothing visible give a zero output and LSE -inf.

The floating-point attention and the combine run in C (``verify_attn_oracle.c``,
compiled with gcc on first use); the integer models (extent, split plan, ring
slots, ring append, position labels) are plain Python/numpy here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "HEAD_DIM", "Q_HEADS", "TILE", "build", "read_extent", "split_plan", "split_position_ranges",
    "verify_attn", "combine", "ring_slot", "ring_append", "ring_labels", "rows_window_complete",
    "visible_positions", "visible_slot_counts", "bf16_bits_to_f64", "f64_to_bf16_bits",
    "tree_masks_from_parents", "tree_depths", "tree_extent", "tree_visible_positions", "verify_attn_tree",
]

HEAD_DIM = 128
Q_HEADS = 6
TILE = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math); returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                        "-o", tmp, _SRC, "-lm", "-lpthread"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            lib.oracle_verify_attn.restype = ctypes.c_int
            lib.oracle_verify_attn.argtypes = [p, p, p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int, p,
                                               ctypes.c_double, ctypes.c_int64, ctypes.c_int, p, p,
                                               p, p, p, p, ctypes.c_int]
            lib.oracle_verify_attn_tree.restype = ctypes.c_int
            lib.oracle_verify_attn_tree.argtypes = [p, p, p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int, p,
                                                    ctypes.c_double, ctypes.c_int64, ctypes.c_int, p, p,
                                                    p, p, p, p, ctypes.c_int]
            lib.oracle_verify_attn_f64kv.restype = ctypes.c_int
            lib.oracle_verify_attn_f64kv.argtypes = [p, p, p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int, p,
                                                     ctypes.c_double, ctypes.c_int64, ctypes.c_int, p, p,
                                                     p, p, p, p, ctypes.c_int]
            lib.oracle_verify_attn_tree_f64kv.restype = ctypes.c_int
            lib.oracle_verify_attn_tree_f64kv.argtypes = [p, p, p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int,
                                                          p, ctypes.c_double, ctypes.c_int64, ctypes.c_int, p, p,
                                                          p, p, p, p, ctypes.c_int]
            lib.oracle_combine.restype = ctypes.c_int
            lib.oracle_combine.argtypes = [p, p, ctypes.c_int, p, ctypes.c_int, ctypes.c_int, p, p]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------- bf16 helpers
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16/int16 array) to float64."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values once to bf16 (round to nearest, ties to even); returns uint16 bits.

    Rounds straight from the double (no float32 step, so no double rounding): a bf16
    number has 8 significant bits, so x = m * 2**e is rounded to a multiple of 2**(e-8)
    with ``np.rint`` (ties to even); below the normal range the spacing stays 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        e = np.maximum(e, -125)
        y = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
        f = y.astype(np.float32)                      # exact: at most 8 significant bits
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits[np.isnan(x)] = 0x7FC0
    return bits


# ----------------------------------------------------------------------------- integer models
def read_extent(pos, n_live: int, window: int = 0):
    """[lo, hi): the positions the live rows can see.  hi = max live position + 1; lo = 0 for
    full attention, max(0, min live position - W + 1) for a sliding window W."""
    live = [int(p) for p in list(pos)[:n_live]]
    if not live:
        return 0, 0
    hi = max(live) + 1
    lo = max(0, min(live) - window + 1) if window > 0 else 0
    return lo, hi


def split_plan(lo: int, hi: int, n_splits: int):
    """64-position tiles of [lo, hi) dealt to n_splits splits: list of (first_tile, end_tile)."""
    if hi <= lo:
        return [(0, 0)] * n_splits
    t_lo = lo // TILE
    t_hi = -(-hi // TILE) - 1
    T = t_hi - t_lo + 1
    return [(t_lo + (s * T) // n_splits, t_lo + ((s + 1) * T) // n_splits) for s in range(n_splits)]


def split_position_ranges(lo: int, hi: int, n_splits: int):
    """Per split the absolute position range [a, b) it owns, clipped to [lo, hi)."""
    out = []
    for first, end in split_plan(lo, hi, n_splits):
        a, b = max(lo, first * TILE), min(hi, end * TILE)
        out.append((a, b) if (end > first and b > a) else (0, 0))
    return out


def visible_positions(p: int, window: int = 0):
    """Positions a row at p sees: range(first, p + 1)."""
    first = max(0, p - window + 1) if window > 0 else 0
    return range(first, p + 1)


def ring_slot(p, slots: int):
    """Physical slot of absolute position p in a ring (or a linear cache) of `slots` rows."""
    return np.asarray(p, dtype=np.int64) % slots


def ring_append(k_cache, v_cache, k_new, v_new, pos, n_live: int):
    """Model of the append: row r of the new K/V goes to slot pos[r] mod slots, in row order.
    Works on copies (numpy arrays [slots, 128]); returns the new caches."""
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    slots = k.shape[0]
    for r in range(n_live):
        s = int(ring_slot(int(pos[r]), slots))
        k[s] = k_new[r]
        v[s] = v_new[r]
    return k, v


def ring_labels(history_positions, pos, n_live: int, slots: int):
    """Position label held by each slot after the history positions are placed in the given
    order and the live rows are appended; -1 where nothing was written."""
    label = np.full(slots, -1, dtype=np.int64)
    for p in history_positions:
        label[int(p) % slots] = int(p)
    for r in range(n_live):
        label[int(pos[r]) % slots] = int(pos[r])
    return label


def rows_window_complete(label, pos, n_live: int, window: int):
    """For each live row: True iff every position of its visible set is still held by its slot."""
    slots = label.shape[0]
    res = []
    for r in range(n_live):
        vis = np.arange(visible_positions(int(pos[r]), window).start, int(pos[r]) + 1, dtype=np.int64)
        res.append(bool(np.all(label[vis % slots] == vis)))
    return res


def visible_slot_counts(pos, n_live: int, n_rows: int, window: int, slots: int):
    """[n_rows, slots] int64: how many times each row's visible set touches each slot
    (one count per visible position; padding rows stay zero)."""
    cnt = np.zeros((n_rows, slots), dtype=np.int64)
    for r in range(n_live):
        vis = np.arange(visible_positions(int(pos[r]), window).start, int(pos[r]) + 1, dtype=np.int64)
        np.add.at(cnt[r], vis % slots, 1)
    return cnt


# ----------------------------------------------------------------------------- verify trees
# "Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify trees": the draft is a tree
# verified in one pass with a tree attention mask.  Node i's K/V sit in slot base + i; node i sees the
# committed prefix and its ancestors (and itself).
def tree_masks_from_parents(parents):
    """Ancestor-or-self bitmasks from a parent array (parents[0] = -1 for the root, parents[i] < i)."""
    masks = []
    for i, par in enumerate(parents):
        par = int(par)
        assert par < i, "nodes are listed parents first"
        masks.append((1 << i) | (masks[par] if par >= 0 else 0))
    return np.array(masks, dtype=np.int32)


def tree_depths(masks):
    """Depth of each node: the number of its strict ancestors."""
    return np.array([bin(int(m) & 0x7FFFFFFF).count("1") - 1 for m in masks], dtype=np.int64)


def tree_extent(base: int, masks, n_nodes: int, window: int = 0):
    """[lo, hi): the slots the live nodes can see.  hi = base + n_nodes (the node slots); lo = 0 for full
    attention, else the earliest window start over the nodes (a node at depth d has logical position
    base + d and a window of W positions ending there), never above base."""
    if n_nodes <= 0:
        return 0, 0
    hi = base + n_nodes
    if window <= 0:
        return 0, hi
    d_min = int(tree_depths(masks[:n_nodes]).min())
    return min(base, max(0, base + d_min - window + 1)), hi


def tree_visible_positions(base: int, masks, n_nodes: int, i: int, window: int = 0):
    """Sorted slot positions node i sees: its window of the prefix, then its in-window ancestors' slots."""
    depth = tree_depths(masks[:n_nodes])
    first = max(0, base + int(depth[i]) - window + 1) if window > 0 else 0
    out = list(range(min(first, base), base))
    for k in range(n_nodes):
        if (int(masks[i]) >> k) & 1 and (window <= 0 or depth[k] >= depth[i] - window + 1):
            out.append(base + k)
    return out


def verify_attn_tree(q_bits, k_hist_bits, v_hist_bits, base: int, masks, n_nodes: int, sink, scale: float,
                     window: int = 0, n_splits: int = 0, split_ranges=None, n_threads: int = 1):
    """FP64 tree verify attention over the linear history (slot j of the history = position j; the nodes
    at base .. base + n_nodes - 1).  q_bits [n_rows, 6, 128]; masks [>= n_nodes] ancestor-or-self masks.
    With n_splits > 0 the partials follow ``split_ranges`` (default: the tile plan of ``tree_extent``).
    Returns dict(out, lse, part_o, part_lse, ranges)."""
    q = _bits16(q_bits)
    kh = _bits16(k_hist_bits)
    vh = _bits16(v_hist_bits)
    n_rows = q.shape[0]
    assert q.shape == (n_rows, Q_HEADS, HEAD_DIM) and kh.shape == vh.shape and kh.shape[1] == HEAD_DIM
    tree = np.zeros(1 + n_rows, dtype=np.int32)
    tree[0] = base
    tree[1:1 + n_nodes] = np.asarray(masks, dtype=np.int64)[:n_nodes]
    sk = None if sink is None else np.ascontiguousarray(np.asarray(sink, dtype=np.float64))
    if n_splits > 0 and split_ranges is None:
        lo, hi = tree_extent(base, tree[1:], n_nodes, window)
        split_ranges = split_position_ranges(lo, hi, n_splits)
    if split_ranges is None:
        split_ranges = []
    S = len(split_ranges)
    sa = np.ascontiguousarray(np.array([a for a, _ in split_ranges] or [0], dtype=np.int64))
    sb = np.ascontiguousarray(np.array([b for _, b in split_ranges] or [0], dtype=np.int64))
    out = np.zeros((n_rows, Q_HEADS, HEAD_DIM), dtype=np.float64)
    lse = np.zeros((n_rows, Q_HEADS), dtype=np.float64)
    part_o = np.zeros((max(S, 1), n_rows, Q_HEADS, HEAD_DIM), dtype=np.float64)
    part_lse = np.zeros((max(S, 1), n_rows, Q_HEADS), dtype=np.float64)
    rc = _load().oracle_verify_attn_tree(_ptr(q), _ptr(kh), _ptr(vh), kh.shape[0], _ptr(tree), n_rows, n_nodes,
                                         _ptr(sk), float(scale), int(window), S, _ptr(sa), _ptr(sb),
                                         _ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attn_tree rejected its arguments (rc={rc})")
    return dict(out=out, lse=lse, part_o=part_o[:S], part_lse=part_lse[:S], ranges=list(split_ranges))


def _bits16(a):
    a = np.asarray(a)
    return np.ascontiguousarray(a.view(np.uint16) if a.dtype == np.int16 else a.astype(np.uint16))


# ----------------------------------------------------------------------------- fp64 attention
def verify_attn(q_bits, k_hist_bits, v_hist_bits, pos, n_live: int, sink, scale: float,
                window: int = 0, n_splits: int = 0, split_ranges=None, n_threads: int = 1):
    """FP64 verify attention over the linear history.

    q_bits [n_rows, 6, 128] and k/v_hist_bits [ctx, 128]: bf16 bit patterns (uint16/int16).
    pos [n_rows] int; sink [6] float or None; window 0 = full attention.
    With n_splits > 0 the partials follow ``split_ranges`` (default: the tile plan of the
    live rows' extent).  Returns dict(out, lse, part_o, part_lse, ranges).
    """
    q = np.ascontiguousarray(np.asarray(q_bits).view(np.uint16) if np.asarray(q_bits).dtype == np.int16
                             else np.asarray(q_bits, dtype=np.uint16))
    kh = np.ascontiguousarray(np.asarray(k_hist_bits).view(np.uint16) if np.asarray(k_hist_bits).dtype == np.int16
                              else np.asarray(k_hist_bits, dtype=np.uint16))
    vh = np.ascontiguousarray(np.asarray(v_hist_bits).view(np.uint16) if np.asarray(v_hist_bits).dtype == np.int16
                              else np.asarray(v_hist_bits, dtype=np.uint16))
    n_rows = q.shape[0]
    assert q.shape == (n_rows, Q_HEADS, HEAD_DIM) and kh.shape == vh.shape and kh.shape[1] == HEAD_DIM
    posa = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    sk = None if sink is None else np.ascontiguousarray(np.asarray(sink, dtype=np.float64))
    if n_splits > 0 and split_ranges is None:
        lo, hi = read_extent(posa, n_live, window)
        split_ranges = split_position_ranges(lo, hi, n_splits)
    if split_ranges is None:
        split_ranges = []
    S = len(split_ranges)
    sa = np.ascontiguousarray(np.array([a for a, _ in split_ranges] or [0], dtype=np.int64))
    sb = np.ascontiguousarray(np.array([b for _, b in split_ranges] or [0], dtype=np.int64))
    out = np.zeros((n_rows, Q_HEADS, HEAD_DIM), dtype=np.float64)
    lse = np.zeros((n_rows, Q_HEADS), dtype=np.float64)
    part_o = np.zeros((max(S, 1), n_rows, Q_HEADS, HEAD_DIM), dtype=np.float64)
    part_lse = np.zeros((max(S, 1), n_rows, Q_HEADS), dtype=np.float64)
    rc = _load().oracle_verify_attn(_ptr(q), _ptr(kh), _ptr(vh), kh.shape[0], _ptr(posa), n_rows, n_live,
                                     _ptr(sk), float(scale), int(window), S, _ptr(sa), _ptr(sb),
                                     _ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attn rejected its arguments (rc={rc})")
    return dict(out=out, lse=lse, part_o=part_o[:S], part_lse=part_lse[:S], ranges=list(split_ranges))


def combine(part_o, part_lse, sink, n_live: int):
    """FP64 log-sum-exp merge of partials [S, n_rows, 6, 128] / [S, n_rows, 6] with the sink."""
    po = np.ascontiguousarray(np.asarray(part_o, dtype=np.float64))
    pl = np.ascontiguousarray(np.asarray(part_lse, dtype=np.float64))
    S, n_rows = pl.shape[0], pl.shape[1]
    sk = None if sink is None else np.ascontiguousarray(np.asarray(sink, dtype=np.float64))
    out = np.zeros((n_rows, Q_HEADS, HEAD_DIM), dtype=np.float64)
    out_lse = np.zeros((n_rows, Q_HEADS), dtype=np.float64)
    rc = _load().oracle_combine(_ptr(po), _ptr(pl), S, _ptr(sk), n_rows, n_live, _ptr(out), _ptr(out_lse))
    if rc != 0:
        raise ValueError(f"oracle_combine rejected its arguments (rc={rc})")
    return out, out_lse
