"""Pins of the FP64 oracle against things other than itself (no GPU).

Each check ties the oracle to the pages' definition through an independent route:
a library routine (torch's scaled_dot_product_attention in float64, torch.logsumexp),
a closed form, an invariant, or brute force.  Planted mistakes (window off by one,
sink dropped, extent from padding rows, shifted split boundaries, a 4,096-slot ring)
must fail the same bars the GPU parity tests use.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import parity
from speculative_decode_verify_gb300 import synth

D, H = 128, 6


def _f64(t):
    return oracle.bf16_bits_to_f64(synth.bits(t).numpy())


def _run(w, n_splits=0, ranges=None, **over):
    args = dict(q_bits=synth.bits(w.q).numpy(), k_hist_bits=synth.bits(w.k_hist).numpy(),
                v_hist_bits=synth.bits(w.v_hist).numpy(), pos=w.pos.numpy(), n_live=w.n_live,
                sink=w.sink.numpy(), scale=w.scale, window=w.window, n_splits=n_splits,
                split_ranges=ranges, n_threads=4)
    args.update(over)
    return oracle.verify_attn(**args)


def _sdpa(w, with_sink=True, window=None):
    """Library route: torch SDPA (float64, CPU math kernel) with the sink as one extra key whose
    K and V are zero and whose additive mask value is the sink logit."""
    window = w.window if window is None else window
    q = torch.from_numpy(_f64(w.q))             # [R, 6, 128]
    K = torch.from_numpy(_f64(w.k_hist))        # [ctx, 128]
    V = torch.from_numpy(_f64(w.v_hist))
    R, ctx = q.shape[0], K.shape[0]
    Kx = torch.cat([K, torch.zeros(1, D, dtype=torch.float64)])
    Vx = torch.cat([V, torch.zeros(1, D, dtype=torch.float64)])
    j = torch.arange(ctx)
    outs, lses = [], []
    for h in range(H):
        mask = torch.full((R, ctx + 1), float("-inf"), dtype=torch.float64)
        for r in range(R):
            p = int(w.pos[r])
            first = max(0, p - window + 1) if window > 0 else 0
            vis = (j >= first) & (j <= p) if r < w.n_live else torch.ones(ctx, dtype=torch.bool)
            mask[r, :ctx] = torch.where(vis, 0.0, float("-inf"))
        mask[:, ctx] = float(w.sink[h]) if with_sink else float("-inf")
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None, None, :, h, :], Kx[None, None], Vx[None, None], attn_mask=mask[None, None], scale=w.scale)
        outs.append(o[0, 0])
        scores = (q[:, h, :] @ Kx.T) * w.scale + mask
        lses.append(torch.logsumexp(scores, dim=-1))
    return torch.stack(outs, 1).numpy(), torch.stack(lses, 1).numpy()


def _small(seed, ctx, n_live, window=0, n_rows=8, pos=None, sink_shift=0.0):
    w = synth.make("pin", seed, ctx=ctx, n_live=n_live, window=window, n_rows=n_rows, pos=pos)
    if sink_shift:
        w.sink = w.sink + sink_shift
    return w


# ----------------------------------------------------------------------------- library routine pins
@pytest.mark.parametrize("ctx,n_live,window,seed", [
    (1, 1, 0, 11), (7, 3, 0, 12), (64, 8, 0, 13), (65, 5, 0, 14), (300, 8, 0, 15),
    (300, 6, 37, 16), (200, 8, 1, 17), (129, 2, 64, 18)])
def test_oracle_matches_sdpa_with_sink_key(ctx, n_live, window, seed):
    w = _small(seed, ctx, n_live, window)
    res = _run(w)
    ref_out, ref_lse = _sdpa(w)
    np.testing.assert_allclose(res["out"][:n_live], ref_out[:n_live], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["lse"][:n_live], ref_lse[:n_live], rtol=1e-12, atol=1e-12)
    assert np.all(res["out"][n_live:] == 0.0) and np.all(np.isneginf(res["lse"][n_live:]))


def test_no_sink_is_textbook_sdpa():
    w = _small(21, 250, 8)
    res = _run(w, sink=None)
    ref_out, ref_lse = _sdpa(w, with_sink=False)
    np.testing.assert_allclose(res["out"], ref_out, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["lse"], ref_lse, rtol=1e-12, atol=1e-12)
    w.sink[:] = float("-inf")
    res2 = _run(w)
    np.testing.assert_allclose(res2["out"], ref_out, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------- closed forms
def test_uniform_scores_give_mean_of_visible_values():
    w = _small(31, 300, 8, window=50)
    w.q = torch.zeros_like(w.q)
    Vf = _f64(w.v_hist)
    for with_sink in (False, True):
        res = _run(w, sink=(w.sink.numpy() if with_sink else None))
        for r in range(w.n_live):
            p = int(w.pos[r])
            vis = np.arange(max(0, p - 49), p + 1)
            n = vis.size
            mean = Vf[vis].mean(axis=0)
            for h in range(H):
                f = n / (n + math.exp(float(w.sink[h]))) if with_sink else 1.0
                np.testing.assert_allclose(res["out"][r, h], f * mean, rtol=1e-12, atol=1e-14)
                lz = math.log(n + math.exp(float(w.sink[h]))) if with_sink else math.log(n)
                assert abs(res["lse"][r, h] - lz) < 1e-12


def test_single_visible_key():
    # full attention at position 0, and a window of 1 at any position: one key each
    for window, pos0 in ((0, 0), (1, 77)):
        w = _small(41, 100, 1, window=window, pos=torch.tensor([pos0] * 8, dtype=torch.int32))
        res = _run(w)
        q, K, V = _f64(w.q), _f64(w.k_hist), _f64(w.v_hist)
        for h in range(H):
            s = w.scale * float(np.dot(q[0, h], K[pos0]))
            sink = float(w.sink[h])
            np.testing.assert_allclose(res["out"][0, h], V[pos0] / (1.0 + math.exp(sink - s)), rtol=1e-12)
            assert abs(res["lse"][0, h] - (s + math.log1p(math.exp(sink - s)))) < 1e-12


def test_window_covering_history_equals_full():
    # every live row sees its whole history once W >= its position + 1
    w = _small(51, 400, 6)
    full = _run(w)
    for W in (int(w.pos[w.n_live - 1]) + 1, int(w.pos[7]) + 1, 4096):
        sw = _run(w, window=W)
        np.testing.assert_array_equal(sw["out"], full["out"])
        np.testing.assert_array_equal(sw["lse"], full["lse"])
    # W = pos[0] + 1 covers row 0 only; the later rows lose their oldest keys
    sw = _run(w, window=int(w.pos[0]) + 1)
    np.testing.assert_array_equal(sw["out"][0], full["out"][0])
    assert np.all(sw["lse"][1:w.n_live] < full["lse"][1:w.n_live])


def test_scale_multiplies_the_dot_product():
    # doubling q (exact in bf16) equals doubling the scale
    w = _small(61, 180, 8)
    a = _run(w, scale=2.0 * w.scale)
    q2 = (w.q.to(torch.float32) * 2.0).to(torch.bfloat16)
    b = _run(w, q_bits=synth.bits(q2).numpy())
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-13, atol=1e-13)


def test_rows_are_independent_of_each_other():
    # permuting which row sits where only permutes the outputs
    w = _small(71, 260, 8)
    res = _run(w)
    perm = np.array([3, 1, 7, 0, 6, 2, 5, 4])
    w2 = _small(71, 260, 8)
    w2.q = w.q[perm]
    w2.pos = w.pos[perm]
    res2 = _run(w2)
    np.testing.assert_array_equal(res2["out"], res["out"][perm])


# ----------------------------------------------------------------------------- split invariants
@pytest.mark.parametrize("window", [0, 100])
def test_split_partials_merge_to_the_direct_result(window):
    w = _small(81, 700, 7, window=window)
    direct = _run(w)
    lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, window)
    T = -(-hi // 64) - lo // 64
    for S in (1, 2, 3, 4, 7, 16, T, T + 5):
        res = _run(w, n_splits=S)
        out, lse = oracle.combine(res["part_o"], res["part_lse"], w.sink.numpy(), w.n_live)
        np.testing.assert_allclose(out, direct["out"], rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(lse[:w.n_live], direct["lse"][:w.n_live], rtol=1e-12, atol=1e-12)
        # without the sink, the log-sum-exp of the split LSEs is the whole-extent LSE
        nosink = _run(w, sink=None)
        tot = torch.logsumexp(torch.from_numpy(res["part_lse"]), dim=0).numpy()
        np.testing.assert_allclose(tot[:w.n_live], nosink["lse"][:w.n_live], rtol=1e-12, atol=1e-12)
        # exactly max(0, S - T) splits own no tile: -inf / 0 for every row
        empty = [s for s, (a, b) in enumerate(res["ranges"]) if b <= a]
        assert len(empty) == max(0, S - T)
        for s in empty:
            assert np.all(np.isneginf(res["part_lse"][s])) and np.all(res["part_o"][s] == 0.0)


def test_combine_single_split_without_sink_is_identity():
    po, pl, _ = synth.random_partials(5, 1, 8, 8, empty_frac=0.0)
    out, lse = oracle.combine(po.numpy(), pl.numpy(), None, 8)
    np.testing.assert_array_equal(out, po.numpy()[0].astype(np.float64))
    np.testing.assert_array_equal(lse, pl.numpy()[0].astype(np.float64))


def test_combine_all_empty_gives_zero():
    po = np.zeros((3, 8, H, D))
    pl = np.full((3, 8, H), -np.inf)
    out, lse = oracle.combine(po, pl, None, 8)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))
    out, lse = oracle.combine(po, pl, np.zeros(H), 8)      # only the sink: zero value
    assert np.all(out == 0.0) and np.allclose(lse, 0.0)


# ----------------------------------------------------------------------------- integer models
def test_split_plan_brute_force():
    rng = np.random.default_rng(0)
    for _ in range(300):
        lo = int(rng.integers(0, 5000))
        hi = lo + int(rng.integers(1, 20000))
        S = int(rng.integers(1, 200))
        plan = oracle.split_plan(lo, hi, S)
        t_lo, t_hi = lo // 64, (hi - 1) // 64
        T = t_hi - t_lo + 1
        tiles = [t for a, b in plan for t in range(a, b)]
        assert tiles == list(range(t_lo, t_hi + 1))                 # ordered, disjoint, complete
        sizes = [b - a for a, b in plan]
        assert max(sizes) - min(sizes) <= 1 and sum(sizes) == T
        assert sum(1 for x in sizes if x > 0) == min(S, T)
        ranges = oracle.split_position_ranges(lo, hi, S)
        covered = sorted(p for a, b in ranges for p in range(a, b))
        assert covered == list(range(lo, hi))


def test_read_extent_uses_live_rows_only():
    pos = np.arange(1016, 1024)
    assert oracle.read_extent(pos, 5) == (0, 1021)
    assert oracle.read_extent(pos, 5, window=4096) == (0, 1021)
    pos = np.arange(39993, 40001)
    assert oracle.read_extent(pos, 7, window=4096) == (39993 - 4095, 40000)


def test_ring_of_window_plus_one_tile_keeps_every_window():
    pos = np.arange(39993, 40001)
    hist = range(0, 39993)
    label = oracle.ring_labels(hist, pos, 8, 4160)
    assert all(oracle.rows_window_complete(label, pos, 8, 4096))
    # placement order of older history does not matter once it is out of every window
    label2 = oracle.ring_labels(list(range(30000, 39993)), pos, 8, 4160)
    assert all(oracle.rows_window_complete(label2, pos, 8, 4096))


def test_negative_control_ring_of_window_loses_history():
    pos = np.arange(39993, 40001)
    label = oracle.ring_labels(range(0, 39993), pos, 8, 4096)
    complete = oracle.rows_window_complete(label, pos, 8, 4096)
    assert not complete[0] and not all(complete)
    # the smallest ring that keeps every window for n live rows is W + n - 1
    for n in range(1, 9):
        lab = oracle.ring_labels(range(0, 39993), pos, n, 4096 + n - 1)
        assert all(oracle.rows_window_complete(lab, pos, n, 4096))
        if n > 1:
            lab = oracle.ring_labels(range(0, 39993), pos, n, 4096 + n - 2)
            assert not all(oracle.rows_window_complete(lab, pos, n, 4096))


def test_ring_append_model():
    k = np.arange(20 * D, dtype=np.uint16).reshape(20, D)
    v = k + 7
    kn = np.full((3, D), 0xAAAA, dtype=np.uint16)
    vn = np.full((3, D), 0xBBBB, dtype=np.uint16)
    k2, v2 = oracle.ring_append(k, v, kn, vn, np.array([18, 19, 20, 21]), 3)
    assert np.all(k2[18] == 0xAAAA) and np.all(k2[19] == 0xAAAA) and np.all(k2[0] == 0xAAAA)
    assert np.all(k2[1] == k[1]) and np.all(v2[0] == 0xBBBB)


def test_visible_slot_counts_wrap():
    cnt = oracle.visible_slot_counts(np.array([69, 70]), 2, 3, window=8, slots=64)
    assert cnt[0].sum() == 8 and cnt[1].sum() == 8 and cnt[2].sum() == 0
    assert cnt[0, 62] == 1 and cnt[0, 5] == 1 and cnt[0, 6] == 0 and cnt[1, 6] == 1 and cnt[1, 62] == 0


# ----------------------------------------------------------------------------- bf16 rounding helper
def test_bf16_rounding_against_brute_force_nearest():
    allbits = np.arange(0, 0x7F80, dtype=np.uint16)           # all finite non-negative bf16
    vals = oracle.bf16_bits_to_f64(allbits)
    rng = np.random.default_rng(3)
    x = rng.uniform(0, 1, 20000) * np.exp2(rng.integers(-140, 120, 20000))
    x = np.concatenate([x, (vals[1:200] + vals[:199]) / 2, (vals[1000:1200] + vals[999:1199]) / 2])
    got = oracle.f64_to_bf16_bits(x)
    i = np.searchsorted(vals, x)
    i = np.clip(i, 1, vals.size - 1)
    lo_err, hi_err = x - vals[i - 1], vals[i] - x
    pick = np.where(hi_err < lo_err, i, np.where(lo_err < hi_err, i - 1, np.where(i % 2 == 0, i, i - 1)))
    np.testing.assert_array_equal(got, allbits[pick])
    np.testing.assert_array_equal(oracle.f64_to_bf16_bits(-x), allbits[pick] | 0x8000)


# ----------------------------------------------------------------------------- negative controls
def _bf16_ref(out):
    return oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(out))


def test_negative_control_window_off_by_one_fails_the_bar():
    w = synth.swa_40k()
    good = _run(w)
    for W in (w.window - 1, w.window + 1):
        bad = _run(w, window=W)
        assert not parity.out_ok(parity.out_metrics(_bf16_ref(bad["out"]), _bf16_ref(good["out"]), w.n_live))


def test_negative_control_dropped_sink_fails_the_bar():
    # short context, where the sink carries real weight
    w = _small(91, 40, 8)
    good = _run(w)
    bad = _run(w, sink=None)
    assert not parity.out_ok(parity.out_metrics(_bf16_ref(bad["out"]), _bf16_ref(good["out"]), w.n_live))
    assert parity.lse_err(bad["lse"][:w.n_live], good["lse"][:w.n_live]) > parity.LSE_ABS


def test_negative_control_extent_from_padding_rows_fails():
    w = synth.tiny()
    good = _run(w)
    bad = _run(w, n_live=w.n_rows)
    assert np.any(bad["out"][w.n_live:] != 0.0)            # padding rows must stay exactly zero
    np.testing.assert_array_equal(bad["out"][:w.n_live], good["out"][:w.n_live])


def test_negative_control_shifted_split_boundaries_fail():
    w = synth.tiny()
    lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, 0)
    good = _run(w, n_splits=4)
    shifted = [(a + 64 if a > 0 else a, b + 64 if b < hi else b) for a, b in good["ranges"]]
    bad = _run(w, ranges=shifted)
    assert parity.lse_err(bad["part_lse"], good["part_lse"]) > parity.LSE_ABS


def test_bars_accept_the_oracle_itself():
    w = synth.tiny()
    res = _run(w)
    m = parity.out_metrics(_bf16_ref(res["out"]), _bf16_ref(res["out"]), w.n_live)
    assert parity.out_ok(m) and m["max_abs"] == 0.0


def test_parity_bar_allows_one_bf16_step_only_where_the_step_exceeds_the_bar():
    import parity
    assert parity.bf16_step(1.5) == 2.0 ** -7 and parity.bf16_step(3.0) == 2.0 ** -6 and parity.bf16_step(-5.0) == 2.0 ** -5
    ref = np.full((8, 6, 128), 0.5)
    out = ref.copy()
    ref[0, 0, 0], out[0, 0, 0] = 3.0, 3.0 + 2.0 ** -6          # one step at |ref| in [2, 4): allowed
    assert parity.out_ok(parity.out_metrics(out, ref, 8))
    out[0, 0, 0] = 3.0 + 2.0 ** -5                             # two steps: not
    assert not parity.out_ok(parity.out_metrics(out, ref, 8))
    out[0, 0, 0] = 3.0
    ref[1, 0, 0], out[1, 0, 0] = 1.5, 1.5 + 0.011              # below 2 the bar stays 1e-2
    assert not parity.out_ok(parity.out_metrics(out, ref, 8))


def test_unrounded_bar_admits_a_rounding_flip_but_not_a_one_and_a_half_step_error():
    # against the unrounded result the bar is 1e-2 plus the half step the bf16 output itself costs
    exact = np.full((8, 6, 128), 0.5)
    exact[0, 0, 0] = 3.0 + 0.45 * 2.0 ** -6          # |exact| in [2, 4): one bf16 step is 2^-6
    ref = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(exact))
    assert ref[0, 0, 0] == 3.0
    out = ref.copy()
    out[0, 0, 0] = 3.0 + 2.0 ** -6                    # the neighbouring value: a rounding flip, allowed
    m = parity.out_metrics(out, ref, 8, exact=exact)
    assert parity.out_ok(m) and m["max_abs_exact"] < 1e-2 + 0.5 * 2.0 ** -6
    out[0, 0, 0] = 3.0 + 1.5 * 2.0 ** -6 + 1e-2       # 1.5 steps + 1e-2 beyond the rounded reference: rejected
    assert not parity.out_ok(parity.out_metrics(out, ref, 8, exact=exact))
    # in [4, 8) one step is 2^-5: the grid bar admits a step on either side of the rounded reference, the
    # unrounded bar only the side a rounding flip can reach
    exact[0, 0, 0] = 5.0 + 0.4 * 2.0 ** -5
    ref = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(exact))
    assert ref[0, 0, 0] == 5.0
    out = ref.copy()
    out[0, 0, 0] = 5.0 + 2.0 ** -5                    # flip upwards: 0.6 step from exact, allowed
    assert parity.out_ok(parity.out_metrics(out, ref, 8, exact=exact))
    out[0, 0, 0] = 5.0 - 2.0 ** -5                    # one step down: 1.4 steps (0.044) from exact, rejected
    m = parity.out_metrics(out, ref, 8, exact=exact)
    assert m["over_bar"] <= 0.0 and not parity.out_ok(m)
    exact[0, 0, 0] = 5.0                              # on the grid: a one-step output is a 0.031 error
    ref = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(exact))
    out = ref.copy()
    out[0, 0, 0] = 5.0 + 2.0 ** -5
    assert not parity.out_ok(parity.out_metrics(out, ref, 8, exact=exact))
