"""CPU oracle of the quantised K/V cache codec and of verify attention over it.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rules as the rest of ``oracle/``).

Source: "Qwen3.8-27B on one RTX 4090", section "A cheaper cache and state": cache values move to INT8;
keys stay FP8 after a Hadamard rotation; verify attention gets faster.  Where the page leaves the codec
open, the plainest reading is taken:

  * one scale per cached position and tensor (per row of K and per row of V), fp32;
  * keys: k' = H k with H the 128 x 128 Sylvester Hadamard matrix of +-1 entries, evaluated by the fast
    Walsh-Hadamard butterfly in float32 (stages of width 1, 2, 4, .., 64; a pair (a, b) becomes
    (a + b, a - b)); s_k = max_i |k'_i| / 448 (float32); code_i = E4M3(k'_i / s_k) rounded to nearest,
    ties to even, saturating at +-448 (float32 division); a value that rounds to zero is coded +0;
  * values: s_v = max_i |v_i| / 127 (float32); code_i = round-half-even(v_i / s_v) in [-127, 127];
  * an all-zero row gets scale 0 and codes 0;
  * decoding: v^ = s_v * code; k^ = H^T (s_k * code) / 128 (H^T H = 128 I), so that
    q . k^ = (H q) . (s_k * code) / 128: attention over the decoded cache is attention in the rotated space.

Where floating point decides a code (the butterfly sums, the scale, the division, the rounding), the
oracle takes the same float32 steps as the encoder, so codes must match bit for bit.  The attention over
the decoded history is computed in float64 by the C oracle.
"""
from __future__ import annotations

import numpy as np

from . import _load, _ptr, split_position_ranges, read_extent, tree_extent, Q_HEADS, HEAD_DIM

__all__ = ["E4M3_MAX", "fwht_f32", "e4m3_round", "e4m3_decode", "e4m3_encode_bits", "encode_k", "encode_v",
           "decode_k", "decode_v", "verify_attn_decoded", "verify_attn_tree_decoded"]

E4M3_MAX = 448.0


def fwht_f32(x):
    """Unnormalised Walsh-Hadamard transform of the last axis (length 128) by the butterfly, in float32."""
    y = np.array(x, dtype=np.float32, copy=True)
    n = y.shape[-1]
    h = 1
    while h < n:
        y = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (n,))
        h *= 2
    return y


def _e4m3_grid():
    """The finite non-negative E4M3 values (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; the
    pattern S.1111.111 is NaN, there are no infinities): subnormals m 2^-9, normals (1 + m/8) 2^(e-7)."""
    vals = [m * 2.0 ** -9 for m in range(8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_GRID = _e4m3_grid()           # 127 values: index = the code's low 7 bits


def e4m3_round(x):
    """Round float values to the nearest E4M3 value (ties to the even code), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(_GRID, a)                 # first grid value >= a
    idx = np.clip(idx, 1, len(_GRID) - 1)
    lo, hi = _GRID[idx - 1], _GRID[idx]
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & ((idx % 2) == 0))   # tie: the even code
    code = np.where(pick_hi, idx, idx - 1)
    code = np.where(a <= 0.0, 0, code)
    neg = (x < 0) & (code > 0)          # a value that rounds to zero gets the code +0
    return np.where(neg, -_GRID[code], _GRID[code]), code.astype(np.uint8) | np.where(neg, 0x80, 0).astype(np.uint8)


def e4m3_encode_bits(x):
    """E4M3 bit patterns (uint8) of float values, rounding as e4m3_round."""
    return e4m3_round(x)[1]


def e4m3_decode(bits):
    b = np.asarray(bits, dtype=np.uint8)
    v = _GRID[np.minimum(b & 0x7F, len(_GRID) - 1)]
    return np.where(b & 0x80, -v, v)


def encode_k(k_bits):
    """bf16 keys [n, 128] (bit patterns) -> (codes uint8 [n, 128], scales float32 [n])."""
    from . import bf16_bits_to_f64
    k = bf16_bits_to_f64(k_bits).astype(np.float32)
    kr = fwht_f32(k)
    m = np.max(np.abs(kr), axis=-1).astype(np.float32)
    s = (m / np.float32(E4M3_MAX)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s[:, None] > 0, (kr / s[:, None]).astype(np.float32), np.float32(0))
    codes = e4m3_encode_bits(ratio.astype(np.float64))
    return codes, s


def encode_v(v_bits):
    """bf16 values [n, 128] -> (codes int8 [n, 128], scales float32 [n])."""
    from . import bf16_bits_to_f64
    v = bf16_bits_to_f64(v_bits).astype(np.float32)
    m = np.max(np.abs(v), axis=-1).astype(np.float32)
    s = (m / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s[:, None] > 0, (v / s[:, None]).astype(np.float32), np.float32(0))
    codes = np.clip(np.rint(ratio.astype(np.float64)), -127, 127).astype(np.int8)
    return codes, s


def decode_k(codes, scales):
    """k^ = H^T (s * e4m3(code)) / 128 in float64 (H symmetric, so H^T = H)."""
    y = e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]
    n = y.shape[-1]
    h = 1
    while h < n:   # exact in float64 for these magnitudes: the butterfly is only used as the matrix H
        y = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(y.shape[:-3] + (n,))
        h *= 2
    return y / 128.0


def decode_v(codes, scales):
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[:, None]


def verify_attn_decoded(q_bits, k_dec, v_dec, pos, n_live: int, sink, scale: float, window: int = 0,
                        n_splits: int = 0, split_ranges=None, n_threads: int = 1):
    """FP64 verify attention over a decoded (float64) linear history k_dec, v_dec [ctx, 128]; arguments and
    result as oracle.verify_attn."""
    q = np.ascontiguousarray(np.asarray(q_bits).view(np.uint16) if np.asarray(q_bits).dtype == np.int16
                             else np.asarray(q_bits, dtype=np.uint16))
    kd = np.ascontiguousarray(np.asarray(k_dec, dtype=np.float64))
    vd = np.ascontiguousarray(np.asarray(v_dec, dtype=np.float64))
    n_rows = q.shape[0]
    assert q.shape == (n_rows, Q_HEADS, HEAD_DIM) and kd.shape == vd.shape and kd.shape[1] == HEAD_DIM
    posa = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    sk = None if sink is None else np.ascontiguousarray(np.asarray(sink, dtype=np.float64))
    if n_splits > 0 and split_ranges is None:
        lo, hi = read_extent(posa, n_live, window)
        split_ranges = split_position_ranges(lo, hi, n_splits)
    split_ranges = split_ranges or []
    S = len(split_ranges)
    sa = np.ascontiguousarray(np.array([a for a, _ in split_ranges] or [0], dtype=np.int64))
    sb = np.ascontiguousarray(np.array([b for _, b in split_ranges] or [0], dtype=np.int64))
    out = np.zeros((n_rows, Q_HEADS, HEAD_DIM))
    lse = np.zeros((n_rows, Q_HEADS))
    part_o = np.zeros((max(S, 1), n_rows, Q_HEADS, HEAD_DIM))
    part_lse = np.zeros((max(S, 1), n_rows, Q_HEADS))
    rc = _load().oracle_verify_attn_f64kv(_ptr(q), _ptr(kd), _ptr(vd), kd.shape[0], _ptr(posa), n_rows, n_live,
                                          _ptr(sk), float(scale), int(window), S, _ptr(sa), _ptr(sb), _ptr(out),
                                          _ptr(lse), _ptr(part_o), _ptr(part_lse), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attn_f64kv rejected its arguments (rc={rc})")
    return dict(out=out, lse=lse, part_o=part_o[:S], part_lse=part_lse[:S], ranges=list(split_ranges))


def verify_attn_tree_decoded(q_bits, k_dec, v_dec, base: int, masks, n_nodes: int, sink, scale: float,
                             window: int = 0, n_splits: int = 0, split_ranges=None, n_threads: int = 1):
    """FP64 tree verify attention ("Qwen3.8-27B on one RTX 4090", section "More tokens per round: verify
    trees") over a decoded (float64) linear history k_dec, v_dec [ctx, 128]: the nodes at base ..
    base + n_nodes - 1 under their ancestor-or-self masks.  Arguments and result as oracle.verify_attn_tree."""
    q = np.ascontiguousarray(np.asarray(q_bits).view(np.uint16) if np.asarray(q_bits).dtype == np.int16
                             else np.asarray(q_bits, dtype=np.uint16))
    kd = np.ascontiguousarray(np.asarray(k_dec, dtype=np.float64))
    vd = np.ascontiguousarray(np.asarray(v_dec, dtype=np.float64))
    n_rows = q.shape[0]
    assert q.shape == (n_rows, Q_HEADS, HEAD_DIM) and kd.shape == vd.shape and kd.shape[1] == HEAD_DIM
    tree = np.zeros(1 + n_rows, dtype=np.int32)
    tree[0] = base
    tree[1:1 + n_nodes] = np.asarray(masks, dtype=np.int64)[:n_nodes]
    sk = None if sink is None else np.ascontiguousarray(np.asarray(sink, dtype=np.float64))
    if n_splits > 0 and split_ranges is None:
        lo, hi = tree_extent(base, tree[1:], n_nodes, window)
        split_ranges = split_position_ranges(lo, hi, n_splits)
    split_ranges = split_ranges or []
    S = len(split_ranges)
    sa = np.ascontiguousarray(np.array([a for a, _ in split_ranges] or [0], dtype=np.int64))
    sb = np.ascontiguousarray(np.array([b for _, b in split_ranges] or [0], dtype=np.int64))
    out = np.zeros((n_rows, Q_HEADS, HEAD_DIM))
    lse = np.zeros((n_rows, Q_HEADS))
    part_o = np.zeros((max(S, 1), n_rows, Q_HEADS, HEAD_DIM))
    part_lse = np.zeros((max(S, 1), n_rows, Q_HEADS))
    rc = _load().oracle_verify_attn_tree_f64kv(_ptr(q), _ptr(kd), _ptr(vd), kd.shape[0], _ptr(tree), n_rows,
                                               n_nodes, _ptr(sk), float(scale), int(window), S, _ptr(sa), _ptr(sb),
                                               _ptr(out), _ptr(lse), _ptr(part_o), _ptr(part_lse), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attn_tree_f64kv rejected its arguments (rc={rc})")
    return dict(out=out, lse=lse, part_o=part_o[:S], part_lse=part_lse[:S], ranges=list(split_ranges))
