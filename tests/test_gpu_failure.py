"""Failure detection on the GPU without a fault: the bounded wait every kernel of the library uses gives
up on a barrier that nothing completes, reports VA_DEV_TIMEOUT in the status word, returns early when a
warp of its CTA raises the abort flag, and leaves the context usable (a verify call right after still
matches the oracle)."""
import numpy as np
import pytest
import torch

import parity
import speculative_decode_verify_gb300 as va
from gpu_cases import DEV, expected, run_step
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(limit_ns, abort_after_ns=0):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    va.va_selftest_bounded_wait(limit_ns, abort_after_ns, dev_status=status, elapsed_ns=elapsed)
    torch.cuda.synchronize()
    return int(status.item()), int(elapsed.item())


def test_a_wait_on_a_barrier_nothing_completes_gives_up_after_its_limit():
    status, elapsed = _run(20_000_000)
    assert status & 16   # VA_DEV_TIMEOUT
    assert 20_000_000 <= elapsed < 500_000_000


def test_the_abort_flag_ends_the_wait_early():
    status, elapsed = _run(500_000_000, abort_after_ns=5_000_000)
    assert status & 16
    assert 5_000_000 <= elapsed < 100_000_000


def test_the_context_stays_usable_after_a_timed_out_wait():
    _run(10_000_000)
    w = synth.make("after_timeout", 3, ctx=1024, n_live=5, slots=1088,
                   pos=torch.arange(1016, 1024, dtype=torch.int32))
    got = run_step(w, n_splits=4)
    assert got["status"] == 0
    ref = expected(w, 4)
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert np.all(got["out_bits"][w.n_live:] == 0)
