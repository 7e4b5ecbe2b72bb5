"""GPU parity of the whole verify call verify_attn_step (the append inside the attention launch, then the
combine) against the FP64 oracle, and against the separate calls bit for bit.

Same bars and caches as tests/test_gpu_parity.py.  The step runs the separate calls' attention kernel with
the same plan and the same combine kernel, so its output, output LSE, partials and cache bytes must equal
those of kv_ring_append + verify_attn_full / verify_attn_swa + attn_split_combine exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from gpu_cases import DEV, expected, run_step, run_step_fused
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _assert_parity(got, ref, w):
    assert got["status"] == 0, f"device status {got['status']:#x}"
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:w.n_live], ref["lse"][:w.n_live]) <= parity.LSE_ABS
    assert np.all(got["out_bits"][w.n_live:] == 0)
    assert np.all(np.isneginf(got["out_lse"][w.n_live:]))
    assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS
    assert np.abs(got["part_o"] - ref["part_o"]).max() <= parity.OUT_MAX_ABS
    return m


def _assert_same_as_separate(got, sep):
    assert np.array_equal(got["out_bits"], sep["out_bits"])
    assert np.array_equal(got["out_lse"], sep["out_lse"], equal_nan=True)
    assert np.array_equal(got["part_lse"], sep["part_lse"], equal_nan=True)
    assert np.array_equal(got["part_o"], sep["part_o"], equal_nan=True)
    assert torch.equal(got["k"], sep["k"]) and torch.equal(got["v"], sep["v"])


@pytest.mark.parametrize("poison", [False, True])
@pytest.mark.parametrize("S", [1, 2, 4, 7])
def test_tiny_step(poison, S):
    w = synth.tiny(poison_tail=poison)
    got = run_step_fused(w, n_splits=S)
    _assert_parity(got, expected(w, S), w)
    _assert_same_as_separate(got, run_step(w, n_splits=S))


@pytest.mark.parametrize("S", [1, 3, 16, 47, 0, 400])
def test_step_split_counts(S):
    w = synth.make("inv", 7, ctx=3000, n_live=6, slots=3100)
    got = run_step_fused(w, n_splits=S)
    _assert_parity(got, expected(w, got["n_splits"]), w)
    _assert_same_as_separate(got, run_step(w, n_splits=got["n_splits"]))


def test_step_16k_peaky_auto():
    w = synth.full_16k()
    got = run_step_fused(w)
    _assert_parity(got, expected(w, got["n_splits"]), w)


@pytest.mark.parametrize("placement", ["all", "window"])
def test_step_swa_ring_wrapped(placement):
    w = synth.swa_40k()
    got = run_step_fused(w, placement=placement)
    _assert_parity(got, expected(w, got["n_splits"]), w)
    _assert_same_as_separate(got, run_step(w, n_splits=got["n_splits"], placement=placement))


@pytest.mark.parametrize("off", [64, 1000, 4159])
def test_step_swa_ring_placement(off):
    w = synth.swa_40k()
    got = run_step_fused(w, n_splits=5, wrap_offset=off)
    ref = expected(w, 5)
    assert got["status"] == 0
    assert parity.out_ok(parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"]))
    _assert_same_as_separate(got, run_step(w, n_splits=5, wrap_offset=off))


@pytest.mark.parametrize("n_live", [4, 5, 6, 7, 8])
def test_step_192k(n_live):
    w = synth.full_192k(n_live)
    got = run_step_fused(w)
    _assert_parity(got, expected(w, got["n_splits"]), w)


@pytest.mark.parametrize("n_rows,n_live", [(1, 1), (3, 2), (8, 0), (8, 8)])
def test_step_row_counts(n_rows, n_live):
    w = synth.make("rows", 50 + n_rows, ctx=2000, n_live=n_live, n_rows=n_rows, slots=2048)
    got = run_step_fused(w, n_splits=6)
    assert got["status"] == 0
    if n_live:
        _assert_parity(got, expected(w, 6), w)
    else:
        assert np.all(got["out_bits"] == 0) and np.all(np.isneginf(got["out_lse"]))


def test_step_reuses_one_workspace_across_calls_and_split_counts():
    ws = torch.empty(va.va_workspace_bytes(_sms()) // 4, dtype=torch.float32, device=DEV)
    for i, S in enumerate([4, 4, 9, 1, _sms(), 3]):
        w = synth.make("reuse", 60 + i, ctx=2500, n_live=1 + i % 8, slots=2560)
        got = run_step_fused(w, n_splits=S, workspace=ws)
        _assert_parity(got, expected(w, S), w)


def test_step_in_a_cuda_graph():
    w = synth.make("graph", 70, ctx=5000, n_live=8, slots=5120)
    S = 12
    ref = run_step(w, n_splits=S)
    k, v = ref["k"].clone(), ref["v"].clone()
    # the caches as before the append (the graph call appends the same rows again: same bytes)
    q = synth.bits(w.q).to(DEV)
    idx = w.pos[:8].to(torch.int64)
    kn, vn = synth.bits(w.k_hist)[idx].contiguous().to(DEV), synth.bits(w.v_hist)[idx].contiguous().to(DEV)
    pos, sink = w.pos.to(DEV), w.sink.to(DEV)
    ws = torch.empty(va.va_workspace_bytes(S) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty(8, 6, 128, dtype=torch.int16, device=DEV)
    lse = torch.empty(8, 6, dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        va.verify_attn_step(q, kn, vn, 8, k, v, pos, w.scale, sink, ws, out, lse, n_splits=S, stream=s)   # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            va.verify_attn_step(q, kn, vn, 8, k, v, pos, w.scale, sink, ws, out, lse, n_splits=S, stream=s)
    for _ in range(3):
        out.fill_(0x7FC0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), ref["out_bits"])
    assert torch.equal(k, ref["k"]) and torch.equal(v, ref["v"])


def test_step_argument_errors():
    w = synth.tiny()
    q = synth.bits(w.q).to(DEV)
    k = torch.zeros(w.slots, 128, dtype=torch.int16, device=DEV)
    v = torch.zeros_like(k)
    kn = torch.zeros(8, 128, dtype=torch.int16, device=DEV)
    pos, sink = w.pos.to(DEV), w.sink.to(DEV)
    out = torch.empty(8, 6, 128, dtype=torch.int16, device=DEV)
    ws = torch.zeros(va.va_workspace_bytes(8) // 4, dtype=torch.float32, device=DEV)
    with pytest.raises(va.VerifyAttnError) as e:       # workspace not 16-byte aligned
        va.verify_attn_step(q, kn, kn, 5, k, v, pos, w.scale, sink, ws[1:], out, n_splits=4)
    assert e.value.status == va.VA_INVALID_ARG
    with pytest.raises(va.VerifyAttnError) as e:       # live rows without their K/V
        va.verify_attn_step(q, None, None, 5, k, v, pos, w.scale, sink, ws, out, n_splits=4)
    assert e.value.status == va.VA_INVALID_ARG
    ring = torch.zeros(4096, 128, dtype=torch.int16, device=DEV)
    with pytest.raises(va.VerifyAttnError) as e:
        va.verify_attn_step(q, kn, kn, 8, ring, ring, pos, w.scale, sink, ws, out, window=4096, n_splits=4)
    assert e.value.status == va.VA_RING_TOO_SMALL
    ring = torch.zeros(4200, 128, dtype=torch.int16, device=DEV)
    with pytest.raises(va.VerifyAttnError) as e:
        va.verify_attn_step(q, kn, kn, 8, ring, ring, pos, w.scale, sink, ws, out, window=4096, n_splits=4)
    assert e.value.status == va.VA_UNSUPPORTED


def test_step_append_with_repeated_positions_matches_row_order():
    # rows sharing a position: the last of them is the one left in the cache, as kv_ring_append leaves it
    w = synth.make("dup", 80, ctx=700, n_live=5, slots=768,
                   pos=torch.tensor([600, 601, 601, 602, 602, 603, 604, 605], dtype=torch.int32))
    kn = torch.randint(-2000, 2000, (5, 128), dtype=torch.int16, generator=synth.generator(81))
    vn = torch.randint(-2000, 2000, (5, 128), dtype=torch.int16, generator=synth.generator(82))
    k0 = torch.zeros(768, 128, dtype=torch.int16)
    k0[:w.ctx] = synth.bits(w.k_hist)
    v0 = torch.zeros(768, 128, dtype=torch.int16)
    v0[:w.ctx] = synth.bits(w.v_hist)
    pos = w.pos.to(DEV)
    ka, va_ = k0.to(DEV), v0.to(DEV)
    va.kv_ring_append(kn.to(DEV), vn.to(DEV), 5, ka, va_, pos)
    kb, vb = k0.to(DEV), v0.to(DEV)
    ws = torch.empty(va.va_workspace_bytes(3) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty(8, 6, 128, dtype=torch.int16, device=DEV)
    va.verify_attn_step(synth.bits(w.q).to(DEV), kn.to(DEV), vn.to(DEV), 5, kb, vb, pos, w.scale, w.sink.to(DEV), ws,
                        out, n_splits=3)
    torch.cuda.synchronize()
    ek, ev = oracle.ring_append(k0.numpy(), v0.numpy(), kn.numpy(), vn.numpy(), w.pos.numpy(), 5)
    np.testing.assert_array_equal(kb.cpu().numpy(), ek)
    np.testing.assert_array_equal(vb.cpu().numpy(), ev)
    assert torch.equal(ka, kb) and torch.equal(va_, vb)
    assert torch.equal(kb[601].cpu(), kn[2]) and torch.equal(kb[602].cpu(), kn[4])
