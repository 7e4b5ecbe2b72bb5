"""Parity metrics shared by the tests (numpy only).

Bars (one KV head, 48 matrix rows, bf16 output):
  * output: max |out - ref| <= 1e-2 and relative RMS ||out - ref|| / ||ref|| <= 2e-3 over the
    live rows, where ref is the FP64 oracle rounded once to bf16 (round to nearest even).  Where one
    bf16 step at |ref| is wider than 1e-2 (|ref| >= 2), an element may differ from ref by that one
    step: the kernel's fp32 result and the exact one can lie on the two sides of a rounding midpoint,
    and the output format cannot hold a closer value;
  * output against the unrounded FP64 result `exact`: |out - exact| <= 1e-2 + one half bf16 step at
    max(|exact|, |out|), element by element.  This is the 1e-2 bar plus exactly the one rounding to bf16
    that the output format forces, so a one-step allowance above can only cover a rounding flip, never a
    kernel error of more than 1e-2;
  * per-split LSE: |lse_s - ref| <= 1e-3 over non-empty splits (both -inf counts as equal);
  * padding rows: exactly zero output, LSE -inf.
"""
import numpy as np

OUT_MAX_ABS = 1e-2
OUT_REL_RMS = 2e-3
LSE_ABS = 1e-3


def bf16_step(x):
    """Spacing of bf16 values at |x| (2^(e - 7) for |x| in [2^e, 2^(e+1)); the subnormal spacing below)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def out_metrics(out, ref, n_live, exact=None):
    """out, ref: float arrays [n_rows, 6, 128]; metrics over live rows.  over_bar: the largest amount by
    which an element exceeds its bar max(1e-2, one bf16 step at |ref|) (<= 0 when every element passes).
    exact (the unrounded FP64 oracle output, same shape): max_abs_exact = max |out - exact| and
    over_exact, the largest amount by which an element exceeds 1e-2 + half a bf16 step at
    max(|exact|, |out|)."""
    o = np.asarray(out, dtype=np.float64)[:n_live]
    r = np.asarray(ref, dtype=np.float64)[:n_live]
    diff = o - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    over = float(np.max(np.abs(diff) - np.maximum(OUT_MAX_ABS, bf16_step(r)))) if diff.size else 0.0
    denom = float(np.linalg.norm(r))
    rel_rms = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    m = dict(max_abs=max_abs, over_bar=over, rel_rms=rel_rms, nan=bool(np.isnan(o).any()))
    if exact is not None:
        e = np.asarray(exact, dtype=np.float64)[:n_live]
        de = np.abs(o - e)
        bar = OUT_MAX_ABS + 0.5 * bf16_step(np.maximum(np.abs(e), np.abs(o)))
        m["max_abs_exact"] = float(de.max()) if de.size else 0.0
        m["over_exact"] = float(np.max(de - bar)) if de.size else 0.0
    return m


def out_ok(m):
    return (not m["nan"]) and m["over_bar"] <= 0.0 and m["rel_rms"] <= OUT_REL_RMS and \
        m.get("over_exact", 0.0) <= 0.0


def lse_err(lse, ref):
    """Max |lse - ref| where both are finite; inf if exactly one side is -inf (or NaN)."""
    a = np.asarray(lse, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    if np.isnan(a).any():
        return float("inf")
    both_empty = np.isneginf(a) & np.isneginf(b)
    one_empty = np.isneginf(a) ^ np.isneginf(b)
    if one_empty.any():
        return float("inf")
    d = np.abs(np.where(both_empty, 0.0, a - np.where(both_empty, 0.0, b)))
    return float(d.max()) if d.size else 0.0
