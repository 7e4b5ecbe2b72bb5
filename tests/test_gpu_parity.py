"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the same seeded inputs.

Bars (tests/parity.py): output within 1e-2 max-abs and 2e-3 relative RMS of the oracle rounded
once to bf16; per-split LSE within 1e-3; padding rows exactly 0 / -inf; ring and cache bytes
bit-exact.  Caches are poisoned where the kernels must not read: NaN beyond the valid extent of a
full cache, finite sentinels (K = 64, V = 1000) in stale ring slots.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from gpu_cases import DEV, expected, run_step
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu


def _assert_parity(got, ref, w, check_partials=True):
    assert got["status"] == 0, f"device status {got['status']:#x}"
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:w.n_live], ref["lse"][:w.n_live]) <= parity.LSE_ABS
    # padding rows: exactly zero, LSE -inf
    assert np.all(got["out_bits"][w.n_live:] == 0)
    assert np.all(np.isneginf(got["out_lse"][w.n_live:]))
    if check_partials:
        assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS
        # partial outputs are fp32: compare where the split saw something
        po_err = np.abs(got["part_o"] - ref["part_o"]).max()
        assert po_err <= parity.OUT_MAX_ABS, po_err
    return m


@pytest.mark.parametrize("poison", [False, True])
def test_tiny_full_four_splits(poison):
    w = synth.tiny(poison_tail=poison)
    got = run_step(w, n_splits=4)
    assert got["status"] == 0
    ref = expected(w, 4)
    _assert_parity(got, ref, w)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 7, 16, 0, "T", "T+5"])
def test_split_count_invariance(S):
    w = synth.make("inv", 7, ctx=3000, n_live=6, slots=3100)
    lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, 0)
    T = -(-hi // 64) - lo // 64
    S = {"T": T, "T+5": T + 5}.get(S, S)
    got = run_step(w, n_splits=S)
    ref = expected(w, got["n_splits"])
    _assert_parity(got, ref, w)


def test_full_16k_peaky_auto_splits():
    w = synth.full_16k()
    got = run_step(w, n_splits=0)
    ref = expected(w, got["n_splits"])
    _assert_parity(got, ref, w)


@pytest.mark.parametrize("placement", ["all", "window"])
def test_swa_ring_wrapped_append_then_read(placement):
    w = synth.swa_40k()
    got = run_step(w, n_splits=0, placement=placement)
    assert got["status"] == 0
    ref = expected(w, got["n_splits"])
    _assert_parity(got, ref, w)


def test_swa_ring_placement_invariance():
    w = synth.swa_40k()
    base = run_step(w, n_splits=5)
    ref = expected(w, 5)
    for off in (64, 1000, 4159):
        got = run_step(w, n_splits=5, wrap_offset=off)
        m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
        assert parity.out_ok(m), (off, m)
        assert parity.lse_err(got["out_lse"][:w.n_live], base["out_lse"][:w.n_live]) <= 1e-5


@pytest.mark.parametrize("S", [1, 3, 33])
def test_swa_short_history_and_split_counts(S):
    # context shorter than the window: lo = 0, ring not yet wrapped
    w = synth.make("swa_short", 9, ctx=1500, n_live=8, window=4096, slots=4160)
    got = run_step(w, n_splits=S)
    ref = expected(w, S)
    _assert_parity(got, ref, w)


@pytest.mark.parametrize("n_live", [4, 5, 6, 7, 8])
def test_full_192k(n_live):
    w = synth.full_192k(n_live)
    got = run_step(w, n_splits=0)
    ref = expected(w, got["n_splits"], n_threads=16)
    _assert_parity(got, ref, w)


def test_short_context_sink_carries_weight():
    # few keys, so the sink matters: a dropped sink would fail here
    w = synth.make("short", 13, ctx=40, n_live=8, slots=64)
    got = run_step(w, n_splits=2)
    ref = expected(w, 2)
    _assert_parity(got, ref, w)


@pytest.mark.parametrize("n_live,n_rows", [(1, 1), (1, 8), (3, 4), (8, 8)])
def test_row_counts(n_live, n_rows):
    w = synth.make("rows", 17 + n_live, ctx=777, n_live=n_live, slots=800, n_rows=n_rows)
    got = run_step(w, n_splits=3)
    ref = expected(w, 3)
    _assert_parity(got, ref, w)


def test_no_live_rows_gives_zero():
    w = synth.make("empty", 19, ctx=200, n_live=1, slots=256)
    w.n_live = 0
    q = synth.bits(w.q).to(DEV)
    k = torch.zeros(256, 128, dtype=torch.int16, device=DEV)
    part_o = torch.full((2, 8, 6, 128), float("nan"), device=DEV)
    part_lse = torch.full((2, 8, 6), float("nan"), device=DEV)
    va.verify_attn_full(q, 0, k, k, w.pos.to(DEV), w.scale, part_o, part_lse, 2)
    out = torch.full((8, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    va.attn_split_combine(part_o, part_lse, 2, w.sink.to(DEV), 0, out)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(part_lse)) and torch.all(part_o == 0)


@pytest.mark.parametrize("pos", [[5, 7, 7, 9, 9, 9, 12, 13], [3, 259, 4, 515, 6, 6, 100, 3],
                                 list(range(16)), [40] * 16])
def test_append_rows_sharing_a_slot_land_in_row_order(pos):
    # repeated positions, and positions a multiple of the slot count apart: the last row wins
    slots = 256
    g = synth.generator(24)
    n = len(pos)
    k0 = torch.randint(-30000, 30000, (slots, 128), generator=g, dtype=torch.int16)
    v0 = torch.randint(-30000, 30000, (slots, 128), generator=g, dtype=torch.int16)
    kn = torch.randint(-30000, 30000, (n, 128), generator=g, dtype=torch.int16)
    vn = torch.randint(-30000, 30000, (n, 128), generator=g, dtype=torch.int16)
    p = torch.tensor(pos, dtype=torch.int32)
    for _ in range(3):
        k, v = k0.clone().to(DEV), v0.clone().to(DEV)
        va.kv_ring_append(kn.to(DEV), vn.to(DEV), n, k, v, p.to(DEV))
        ek, ev = oracle.ring_append(k0.numpy(), v0.numpy(), kn.numpy(), vn.numpy(), p.numpy(), n)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(k.cpu().numpy(), ek)
        np.testing.assert_array_equal(v.cpu().numpy(), ev)


def test_append_bytes_bit_exact_with_wrap():
    slots = 256
    g = synth.generator(23)
    k0 = torch.randint(-30000, 30000, (slots, 128), generator=g, dtype=torch.int16)
    v0 = torch.randint(-30000, 30000, (slots, 128), generator=g, dtype=torch.int16)
    kn = torch.randint(-30000, 30000, (8, 128), generator=g, dtype=torch.int16)
    vn = torch.randint(-30000, 30000, (8, 128), generator=g, dtype=torch.int16)
    pos = torch.arange(1020, 1028, dtype=torch.int32)         # wraps around slot 255 -> 0
    for n_live in (1, 5, 8):
        k, v = k0.clone().to(DEV), v0.clone().to(DEV)
        va.kv_ring_append(kn[:n_live].to(DEV), vn[:n_live].to(DEV), n_live, k, v, pos.to(DEV))
        ek, ev = oracle.ring_append(k0.numpy(), v0.numpy(), kn.numpy(), vn.numpy(), pos.numpy(), n_live)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(k.cpu().numpy(), ek)
        np.testing.assert_array_equal(v.cpu().numpy(), ev)


def test_device_status_for_bad_positions():
    w = synth.make("bad", 29, ctx=500, n_live=4, slots=512)
    q = synth.bits(w.q).to(DEV)
    k = synth.bits(w.k_hist).to(DEV)
    cases = [([10, 11, -1, 13, 0, 0, 0, 0], 0, va.VA_OK, 1),       # negative
             ([10, 11, 9, 13, 0, 0, 0, 0], 0, va.VA_OK, 2),        # decreasing
             ([497, 498, 499, 500, 0, 0, 0, 0], 0, va.VA_OK, 4)]   # beyond a 500-row cache
    for pos, window, _, bit in cases:
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        part_o = torch.full((3, 8, 6, 128), float("nan"), device=DEV)
        part_lse = torch.full((3, 8, 6), float("nan"), device=DEV)
        va.verify_attn_full(q, 4, k[:500], k[:500], torch.tensor(pos, dtype=torch.int32, device=DEV), w.scale,
                            part_o, part_lse, 3, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & bit
        assert torch.all(torch.isneginf(part_lse)) and torch.all(part_o == 0)
    # sliding window: positions spread wider than the ring allows
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ring = torch.zeros(4160, 128, dtype=torch.int16, device=DEV)
    part_o = torch.full((3, 8, 6, 128), float("nan"), device=DEV)
    part_lse = torch.full((3, 8, 6), float("nan"), device=DEV)
    pos = torch.tensor([5000, 5001, 5100, 5200, 0, 0, 0, 0], dtype=torch.int32, device=DEV)
    va.verify_attn_swa(q, 4, ring, ring, 4096, pos, w.scale, part_o, part_lse, 3, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 8
    assert torch.all(torch.isneginf(part_lse))
    # append with a negative position writes nothing and flags it
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ring2 = ring.clone()
    va.kv_ring_append(k[:2], k[:2], 2, ring2, ring2, torch.tensor([-3, 7], dtype=torch.int32, device=DEV),
                      dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 1
    assert torch.equal(ring2[7].cpu(), k[1].cpu()) and int((ring2 != 0).any(dim=1).sum()) == 1


# every shape of the combine: one warp a CTA with 1, 2, 3, 6, 9 or 12 splits a lane (S <= 48), 128 threads x 5
# (49..80), 128 threads x 10 in one round (81..160) or more rounds; above 8 rows (trees) one warp a CTA up to 48
# splits, else 128 threads x 5 in one or more rounds
@pytest.mark.parametrize("n_rows,n_live,S", [(8, 7, 0), (8, 7, 1), (8, 7, 3), (8, 7, 4), (8, 7, 5), (8, 7, 9),
                                             (8, 7, 20), (8, 7, 33), (8, 7, 48), (8, 7, 64), (8, 7, 152),
                                             (8, 7, 160), (8, 7, 161), (8, 7, 4096), (16, 13, 17), (16, 13, 76),
                                             (16, 16, 100)])
def test_combine_alone_on_synthetic_partials(n_rows, n_live, S):
    po, pl, sink = synth.random_partials(31 + S, max(S, 1), n_rows, n_live)
    po, pl = po[:S], pl[:S]
    ref_out, ref_lse = oracle.combine(po.numpy(), pl.numpy(), sink.numpy(), n_live)
    out = torch.full((n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((n_rows, 6), float("nan"), device=DEV)
    va.attn_split_combine(po.to(DEV) if S else None, pl.to(DEV) if S else None, S, sink.to(DEV), n_live, out,
                          out_lse)
    torch.cuda.synchronize()
    got = oracle.bf16_bits_to_f64(out.cpu().numpy())
    m = parity.out_metrics(got, oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(ref_out)), n_live, exact=ref_out)
    assert parity.out_ok(m), m
    assert parity.lse_err(out_lse.cpu().numpy()[:n_live], ref_lse[:n_live]) <= 1e-5
    assert torch.all(out[n_live:] == 0)


def test_graph_capture_of_the_step_replays_identically():
    w = synth.make("graph", 37, ctx=5000, n_live=8, slots=5120)
    q = synth.bits(w.q).to(DEV)
    k = synth.bits(w.k_hist).to(DEV)
    v = synth.bits(w.v_hist).to(DEV)
    kc = torch.zeros(5120, 128, dtype=torch.int16, device=DEV)
    vc = torch.zeros(5120, 128, dtype=torch.int16, device=DEV)
    kc[:5000] = k
    vc[:5000] = v
    pos = w.pos.to(DEV)
    S = 9
    part_o = torch.empty(S, 8, 6, 128, device=DEV)
    part_lse = torch.empty(S, 8, 6, device=DEV)
    out = torch.empty(8, 6, 128, dtype=torch.int16, device=DEV)
    sink = w.sink.to(DEV)
    idx = w.pos.to(torch.int64)
    k_new, v_new = synth.bits(w.k_hist)[idx].to(DEV), synth.bits(w.v_hist)[idx].to(DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        def step():
            va.kv_ring_append(k_new, v_new, 8, kc, vc, pos, stream=s)
            va.verify_attn_full(q, 8, kc, vc, pos, w.scale, part_o, part_lse, S, stream=s)
            va.attn_split_combine(part_o, part_lse, S, sink, 8, out, stream=s)
        step()
        s.synchronize()
        eager = out.clone()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        out.zero_()
        g.replay()
        s.synchronize()
    assert torch.equal(out, eager)
    ref = expected(w, S)
    m = parity.out_metrics(oracle.bf16_bits_to_f64(out.cpu().numpy()), ref["out_bf16"], 8, exact=ref["out"])
    assert parity.out_ok(m), m


def test_stability_one_vs_eight_live_rows():
    # row 0 must not depend on how many drafts ride along with it
    w8 = synth.make("stab", 41, ctx=9000, n_live=8, slots=9100)
    w1 = synth.make("stab", 41, ctx=9000, n_live=8, slots=9100)
    w1.n_live = 1
    a = run_step(w8, n_splits=0)
    b = run_step(w1, n_splits=0)
    ref = expected(w1, b["n_splits"])
    for got in (a, b):
        m = parity.out_metrics(got["out"][:1], ref["out_bf16"][:1], 1, exact=ref["out"][:1])
        assert parity.out_ok(m), m
