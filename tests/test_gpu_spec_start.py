"""The split kernel's speculative start (build option VA_SPEC): q and the first ring fill are requested from
the positions read before the launch dependency resolves, and checked against the positions read after it.

The build must give the default build's bytes exactly: the same plan, the same tiles, the same arithmetic.
The VA_SPEC_SKEW test build shifts the early positions by one tile, so that every launch whose first fill
was requested from them takes the stale-hint path (wait for the copies, re-arm the stage barriers, request
the real tiles); its outputs must be the same bytes too.  Parity with the FP64 oracle under the bars of
tests/parity.py, for separate calls and for verify_attn_step (IQuestRT report, "Read only the KV tiles
needed by the current positions"; "Let correctness checks change the design").
"""
import numpy as np
import pytest
import torch

import parity
from gpu_cases import expected, run_step, run_step_fused
from speculative_decode_verify_gb300 import build, synth

pytestmark = pytest.mark.gpu
VARIANTS = {"_spec": ["VA_SPEC=1", "VA_EARLY=0"], "_specskew": ["VA_SPEC=1", "VA_SPEC_SKEW=1", "VA_EARLY=0"]}


@pytest.fixture(scope="module", params=sorted(VARIANTS))
def variant(request):
    build.build(variant=request.param, defines=VARIANTS[request.param])
    return request.param


def _case(name):
    if name == "tiny":
        return synth.tiny()
    if name == "inv":
        return synth.make("inv", 7, ctx=3000, n_live=6, slots=3100)
    if name == "16k":
        return synth.full_16k()
    return synth.swa_40k()


def _check(got, base, w):
    assert got["status"] == 0, f"device status {got['status']:#x}"
    ref = expected(w, got["n_splits"])
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:w.n_live], ref["lse"][:w.n_live]) <= parity.LSE_ABS
    assert np.array_equal(got["out_bits"], base["out_bits"])
    assert np.array_equal(got["out_lse"], base["out_lse"], equal_nan=True)
    assert np.array_equal(got["part_o"], base["part_o"], equal_nan=True)
    assert torch.equal(got["k"], base["k"]) and torch.equal(got["v"], base["v"])


@pytest.mark.parametrize("name,S,wrap", [("tiny", 1, 0), ("tiny", 4, 0), ("tiny", 7, 0), ("inv", 1, 0),
                                         ("inv", 16, 0), ("inv", 400, 0), ("16k", 0, 0), ("swa", 0, 0),
                                         ("swa", 5, 1000)])
def test_separate_calls(variant, name, S, wrap):
    w = _case(name)
    got = run_step(w, n_splits=S, wrap_offset=wrap, variant=variant)
    _check(got, run_step(w, n_splits=got["n_splits"], wrap_offset=wrap), w)


@pytest.mark.parametrize("name,S,wrap", [("tiny", 1, 0), ("tiny", 2, 0), ("tiny", 7, 0), ("inv", 3, 0),
                                         ("inv", 47, 0), ("16k", 0, 0), ("swa", 0, 0), ("swa", 5, 4159)])
def test_step(variant, name, S, wrap):
    w = _case(name)
    got = run_step_fused(w, n_splits=S, wrap_offset=wrap, variant=variant)
    _check(got, run_step_fused(w, n_splits=got["n_splits"], wrap_offset=wrap), w)
