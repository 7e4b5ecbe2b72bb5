"""GPU checks of verify_attn_q8_step: the whole verify call over the quantised cache in one call (the
encoding append, the split kernel, the combine).  It must equal kv_ring_append_q8 + verify_attn_q8 +
attn_split_combine called one by one, bit for bit (codes, scales, partials, output, LSE), and so the FP64
oracle over the decoded cache within the parity bars ("Qwen3.8-27B on one RTX 4090", section "A cheaper
cache and state"; IQuestRT report, "Read only the KV tiles needed by the current positions": the new rows
are written before they are read)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from speculative_decode_verify_gb300 import synth
from test_gpu_codec import DEV, _assert, _encoded_cache, expected_q8

pytestmark = pytest.mark.gpu


def _live(w):
    idx = w.pos[:w.n_live].to(torch.int64)
    return (synth.bits(w.k_hist)[idx].contiguous().to(DEV), synth.bits(w.v_hist)[idx].contiguous().to(DEV))


def _splits(w, n_splits):
    if n_splits:
        return n_splits
    return va.va_auto_splits(w.window + w.n_live - 1 if w.window else w.slots, w.window)


def run_separate(w, n_splits=0, live=None):
    S = _splits(w, n_splits)
    kc, vc, ks, vs = _encoded_cache(w, w.slots, int(w.pos[0]))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kn, vn = live or _live(w)
    va.kv_ring_append_q8(kn, vn, w.n_live, kc, vc, ks, vs, w.pos.to(DEV), dev_status=status)
    part_o = torch.full((S, w.n_rows, 6, 128), float("nan"), device=DEV)
    part_lse = torch.full((S, w.n_rows, 6), float("nan"), device=DEV)
    used = va.verify_attn_q8(synth.bits(w.q).to(DEV), w.n_live, kc, vc, ks, vs, w.pos.to(DEV), w.scale, part_o,
                             part_lse, window=w.window, n_splits=S, dev_status=status)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), device=DEV)
    va.attn_split_combine(part_o, part_lse, used, w.sink.to(DEV), w.n_live, out, out_lse)
    torch.cuda.synchronize()
    return dict(out_bits=out.cpu().numpy().view(np.uint16), out_lse=out_lse.cpu().numpy(), part_o=part_o.cpu().numpy(),
                part_lse=part_lse.cpu().numpy(), status=int(status.item()), n_splits=used,
                caches=[t.cpu().numpy() for t in (kc, vc, ks, vs)])


def run_step(w, n_splits=0, workspace=None, live=None):
    S = _splits(w, n_splits)
    kc, vc, ks, vs = _encoded_cache(w, w.slots, int(w.pos[0]))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    kn, vn = live or _live(w)
    if workspace is None:
        workspace = torch.full((va.va_workspace_bytes(S) // 4,), float("nan"), device=DEV)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), device=DEV)
    used = va.verify_attn_q8_step(synth.bits(w.q).to(DEV), kn, vn, w.n_live, kc, vc, ks, vs, w.pos.to(DEV), w.scale,
                                  w.sink.to(DEV), workspace, out, out_lse, window=w.window, n_splits=S,
                                  dev_status=status)
    torch.cuda.synchronize()
    n_o = used * 8 * 6 * 128
    part_o = workspace[:used * w.n_rows * 6 * 128].view(used, w.n_rows, 6, 128)
    part_lse = workspace[n_o:n_o + used * w.n_rows * 6].view(used, w.n_rows, 6)
    return dict(out_bits=out.cpu().numpy().view(np.uint16), out_lse=out_lse.cpu().numpy(), part_o=part_o.cpu().numpy(),
                part_lse=part_lse.cpu().numpy(), status=int(status.item()), n_splits=used,
                caches=[t.cpu().numpy() for t in (kc, vc, ks, vs)])


def _same(a, b):
    assert a["status"] == 0 and b["status"] == 0, (a["status"], b["status"])
    assert a["n_splits"] == b["n_splits"]
    for x, y in zip(a["caches"], b["caches"]):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))   # NaN sentinels compare by bits
    assert np.array_equal(a["out_bits"], b["out_bits"])
    assert np.array_equal(a["out_lse"].view(np.uint32), b["out_lse"].view(np.uint32))
    assert np.array_equal(a["part_o"].view(np.uint32), b["part_o"].view(np.uint32))
    assert np.array_equal(a["part_lse"].view(np.uint32), b["part_lse"].view(np.uint32))


@pytest.mark.parametrize("S", [1, 3, 4, 16])
def test_q8_step_small_full_equals_separate_calls(S):
    w = synth.make("q8s", 231, ctx=1024, n_live=5, slots=1088, pos=torch.arange(1016, 1024, dtype=torch.int32))
    _same(run_step(w, S), run_separate(w, S))


@pytest.mark.parametrize("n_live", [1, 4, 8])
def test_q8_step_16k_auto_splits_equals_separate_calls_and_the_oracle(n_live):
    w = synth.make("q8s16k", 232 + n_live, ctx=16384, n_live=n_live, slots=65536, peaky_frac=0.05)
    got = run_step(w)
    _same(got, run_separate(w))
    ref = expected_q8(w, got["n_splits"])
    out = oracle.bf16_bits_to_f64(got["out_bits"].view(np.int16))
    m = parity.out_metrics(out, ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS


@pytest.mark.parametrize("ctx,n_live", [(40000, 7), (4200, 8), (300, 3)])
def test_q8_step_sliding_window_ring_equals_separate_calls(ctx, n_live):
    pos = torch.tensor([ctx - n_live + r for r in range(8)], dtype=torch.int32)
    w = synth.make("q8s_swa", 240 + n_live, ctx=ctx, n_live=n_live, window=synth.WINDOW, slots=synth.RING_SLOTS,
                   pos=pos)
    _same(run_step(w), run_separate(w))


def test_q8_step_192k_equals_separate_calls():
    w = synth.full_192k(8)
    w.slots = 196672
    _same(run_step(w), run_separate(w))


@pytest.mark.parametrize("n_live", [0, 2, 8])
def test_q8_step_row_counts(n_live):
    pos = torch.tensor([3000 + r for r in range(8)], dtype=torch.int32)
    w = synth.make("q8srows", 250 + n_live, ctx=3008, n_live=max(n_live, 1), slots=3072, pos=pos)
    w.n_live = n_live
    got = run_step(w, 7)
    _same(got, run_separate(w, 7))
    if n_live == 0:
        assert np.all(got["out_bits"] == 0) and np.all(np.isneginf(got["out_lse"]))


def test_q8_step_rows_sharing_a_position_land_in_row_order():
    # rows 1, 2 share position 2001 and rows 4, 5, 6 share 2003, with different K/V: the slot keeps the
    # last row's codes, in the step as in the separate append
    pos = torch.tensor([2000, 2001, 2001, 2002, 2003, 2003, 2003, 2004], dtype=torch.int32)
    w = synth.make("q8sdup", 260, ctx=2005, n_live=8, slots=2048, pos=pos)
    g = synth.generator(261)
    kb = synth.bits(synth.normal_bf16((8, 128), g))
    vb = synth.bits(synth.normal_bf16((8, 128), g))
    live = (kb.to(DEV), vb.to(DEV))
    a, b = run_step(w, 5, live=live), run_separate(w, 5, live=live)
    _same(a, b)
    from oracle import kv_codec as C
    rk, rks = C.encode_k(kb.numpy())
    rv, rvs = C.encode_v(vb.numpy())
    for r in range(8):
        if r + 1 < 8 and int(pos[r + 1]) == int(pos[r]):
            continue   # a later row owns the slot
        p = int(pos[r])
        assert np.array_equal(a["caches"][0][p], rk[r]) and np.array_equal(a["caches"][1][p], rv[r])
        assert a["caches"][2][p].view(np.uint32) == rks[r].view(np.uint32)
        assert a["caches"][3][p].view(np.uint32) == rvs[r].view(np.uint32)


def test_q8_step_workspace_reuse_and_graph_capture():
    w = synth.make("q8sgraph", 270, ctx=8192, n_live=6, slots=8256)
    S = _splits(w, 0)
    ws = torch.full((va.va_workspace_bytes(S) // 4,), float("nan"), device=DEV)
    first = run_step(w, 0, workspace=ws)
    again = run_step(w, 0, workspace=ws)
    _same(first, again)
    kc, vc, ks, vs = _encoded_cache(w, w.slots, int(w.pos[0]))
    kn, vn = _live(w)
    q, pos, sink = synth.bits(w.q).to(DEV), w.pos.to(DEV), w.sink.to(DEV)
    out = torch.empty(w.n_rows, 6, 128, dtype=torch.int16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            va.verify_attn_q8_step(q, kn, vn, w.n_live, kc, vc, ks, vs, pos, w.scale, sink, ws, out, n_splits=S,
                                   stream=s)
        g.replay()
    s.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), first["out_bits"])
