"""Parity metrics shared by the tests (numpy only).

Bars (one KV head, 48 matrix rows, bf16 output):
  * output: max |out - ref| <= 1e-2 and relative RMS ||out - ref|| / ||ref|| <= 2e-3 over the
    live rows, where ref is the FP64 oracle rounded once to bf16 (round to nearest even);
  * per-split LSE: |lse_s - ref| <= 1e-3 over non-empty splits (both -inf counts as equal);
  * padding rows: exactly zero output, LSE -inf.
"""
import numpy as np

OUT_MAX_ABS = 1e-2
OUT_REL_RMS = 2e-3
LSE_ABS = 1e-3


def out_metrics(out, ref, n_live):
    """out, ref: float arrays [n_rows, 6, 128]; metrics over live rows."""
    o = np.asarray(out, dtype=np.float64)[:n_live]
    r = np.asarray(ref, dtype=np.float64)[:n_live]
    diff = o - r
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(r))
    rel_rms = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return dict(max_abs=max_abs, rel_rms=rel_rms, nan=bool(np.isnan(o).any()))


def out_ok(m):
    return (not m["nan"]) and m["max_abs"] <= OUT_MAX_ABS and m["rel_rms"] <= OUT_REL_RMS


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
