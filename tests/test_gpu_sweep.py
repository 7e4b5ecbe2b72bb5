"""GPU parity over the context sweep: {1K, 4K, 16K, 32K, 64K, 128K, 192K} x {full, sliding window} x
n_live 4..8 (70 points), automatic split counts, rows at the tail of the context."""
import pytest

import parity
from gpu_cases import expected, run_step
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("idx,ctx,window,n_live", synth.sweep_points(),
                         ids=[f"{'swa' if p[2] else 'full'}-{p[1]}-n{p[3]}" for p in synth.sweep_points()])
def test_sweep_point(idx, ctx, window, n_live):
    w = synth.sweep(idx, ctx, window, n_live)
    got = run_step(w, n_splits=0)
    assert got["status"] == 0
    ref = expected(w, got["n_splits"], n_threads=16)
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:w.n_live], ref["lse"][:w.n_live]) <= parity.LSE_ABS
    assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS
    assert (got["out_bits"][w.n_live:] == 0).all()
