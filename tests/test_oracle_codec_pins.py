"""Pins of the quantised-KV codec oracle (oracle/kv_codec.py; no GPU).

"Qwen3.8-27B on one RTX 4090", section "A cheaper cache and state": keys FP8 after a Hadamard rotation,
values INT8.  The codec's pieces are pinned by other routes: the butterfly against the Sylvester matrix
(scipy.linalg.hadamard) in float64, E4M3 rounding against a brute-force nearest search with the format's
bit layout, INT8 against a brute-force nearest integer, decode(encode(x)) within the formats' error
bounds, the rotated-space identity q . k^ = (H q) . (s c) / 128, and attention over the decoded cache
against torch's float64 SDPA.
"""
import numpy as np
import pytest
import torch
from scipy.linalg import hadamard

import oracle
from oracle import kv_codec as C
from speculative_decode_verify_gb300 import synth


def _bits(t):
    return synth.bits(t).numpy()


def test_butterfly_is_the_sylvester_hadamard_matrix():
    H = hadamard(128).astype(np.float64)
    rng = np.random.default_rng(1)
    x = rng.integers(-50, 50, size=(7, 128)).astype(np.float32)   # small integers: float32 sums are exact
    np.testing.assert_array_equal(C.fwht_f32(x).astype(np.float64), x.astype(np.float64) @ H.T)
    y = rng.standard_normal((5, 128)).astype(np.float32)
    np.testing.assert_allclose(C.fwht_f32(y), y.astype(np.float64) @ H.T, rtol=0, atol=1e-4)


def _e4m3_value_of_bits(b):
    s, e, m = (b >> 7) & 1, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return None                     # NaN
    v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def test_e4m3_rounding_brute_force():
    table = [(b, _e4m3_value_of_bits(b)) for b in range(256)]
    finite = [(b, v) for b, v in table if v is not None and not (v == 0 and b == 0x80)]
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000) * 50, rng.standard_normal(1000) * 0.01,
                         np.array([v for _, v in finite]), np.array([(a + b) / 2 for (_, a), (_, b) in
                                                                    zip(sorted(finite, key=lambda t: t[1])[:-1],
                                                                        sorted(finite, key=lambda t: t[1])[1:])]),
                         np.array([448.0, 449.0, 460.0, 1000.0, -1000.0, 0.0, 2.0 ** -10, 3 * 2.0 ** -10])])
    got = C.e4m3_encode_bits(xs)
    for x, g in zip(xs, got):
        cx = min(abs(x), 448.0)
        best = min((abs(v - cx), b & 0x7F) for b, v in finite if v >= 0)
        cands = [b & 0x7F for b, v in finite if v >= 0 and abs(v - cx) == best[0]]
        want = min(cands, key=lambda c: (c % 2, c)) if len(cands) > 1 else cands[0]   # ties: even code
        if x < 0 and want != 0:      # values rounding to zero are coded +0
            want |= 0x80
        assert int(g) == want, (x, int(g), want)
    assert np.array_equal(C.e4m3_decode(C.e4m3_encode_bits(np.array([v for _, v in finite]))),
                          np.array([v for _, v in finite]))


def test_int8_values_brute_force_and_error_bound():
    w = synth.make("codec", 3, ctx=500, n_live=4)
    codes, s = C.encode_v(_bits(w.v_hist))
    v = oracle.bf16_bits_to_f64(_bits(w.v_hist))
    for r in range(0, 500, 37):
        for d in range(0, 128, 11):
            ratio = np.float32(np.float32(v[r, d]) / s[r])
            cand = np.arange(-127, 128)
            dist = np.abs(cand - float(ratio))
            best = cand[dist == dist.min()]
            want = best[np.argmin(best % 2)] if len(best) > 1 else best[0]
            assert codes[r, d] == want
    dec = C.decode_v(codes, s)
    assert np.all(np.abs(dec - v) <= 0.5 * s[:, None] * (1 + 1e-4) + 1e-30)   # float32 quotient
    assert np.all(np.abs(codes).max(axis=1) == 127)


def test_keys_decode_within_the_e4m3_bound_and_rotated_identity():
    w = synth.make("codec", 4, ctx=300, n_live=4)
    codes, s = C.encode_k(_bits(w.k_hist))
    k = oracle.bf16_bits_to_f64(_bits(w.k_hist))
    kd = C.decode_k(codes, s)
    H = hadamard(128).astype(np.float64)
    # in the rotated space every element is within half an E4M3 step (relative 2^-4, absolute 2^-10 s)
    rot = k @ H.T
    rot_dec = C.e4m3_decode(codes) * s[:, None].astype(np.float64)
    bound = np.maximum(np.abs(rot) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * 1.0001 + 1e-4 * s[:, None]
    assert np.all(np.abs(rot_dec - rot) <= bound)
    np.testing.assert_allclose(kd, rot_dec @ H / 128.0, rtol=1e-12, atol=1e-12)
    q = np.random.default_rng(5).standard_normal(128)
    np.testing.assert_allclose(kd @ q, rot_dec @ (H @ q) / 128.0, rtol=1e-10, atol=1e-10)
    assert np.all(np.max(np.abs(rot_dec / s[:, None]), axis=1) <= 448.0)


def test_zero_rows_encode_to_zero():
    z = np.zeros((3, 128), dtype=np.uint16)
    kc, ks = C.encode_k(z)
    vc, vs = C.encode_v(z)
    assert np.all(kc == 0) and np.all(ks == 0) and np.all(vc == 0) and np.all(vs == 0)
    assert np.all(C.decode_k(kc, ks) == 0) and np.all(C.decode_v(vc, vs) == 0)


@pytest.mark.parametrize("window", [0, 37])
def test_attention_over_the_decoded_cache_matches_sdpa(window):
    w = synth.make("codec", 6, ctx=260, n_live=6, window=window)
    kc, ks = C.encode_k(_bits(w.k_hist))
    vc, vs = C.encode_v(_bits(w.v_hist))
    kd, vd = C.decode_k(kc, ks), C.decode_v(vc, vs)
    res = C.verify_attn_decoded(_bits(w.q), kd, vd, w.pos.numpy(), w.n_live, w.sink.numpy(), w.scale, window,
                                n_splits=3)
    q = torch.from_numpy(oracle.bf16_bits_to_f64(_bits(w.q)))
    K = torch.cat([torch.from_numpy(kd), torch.zeros(1, 128, dtype=torch.float64)])
    V = torch.cat([torch.from_numpy(vd), torch.zeros(1, 128, dtype=torch.float64)])
    j = torch.arange(w.ctx)
    for r in range(w.n_live):
        p = int(w.pos[r])
        first = max(0, p - window + 1) if window else 0
        for h in range(6):
            mask = torch.full((w.ctx + 1,), float("-inf"), dtype=torch.float64)
            mask[:w.ctx] = torch.where((j >= first) & (j <= p), 0.0, float("-inf"))
            mask[w.ctx] = float(w.sink[h])
            o = torch.nn.functional.scaled_dot_product_attention(q[None, None, r:r + 1, h], K[None, None], V[None, None],
                                                                 attn_mask=mask[None, None, None], scale=w.scale)
            np.testing.assert_allclose(res["out"][r, h], o[0, 0, 0].numpy(), rtol=1e-11, atol=1e-13)
    out, lse = oracle.combine(res["part_o"], res["part_lse"], w.sink.numpy(), w.n_live)
    np.testing.assert_allclose(out[:w.n_live], res["out"][:w.n_live], rtol=1e-10, atol=1e-13)


def test_quantised_attention_stays_near_the_bf16_attention():
    # the codec's own error, for scale: not a kernel bar
    w = synth.make("codec", 7, ctx=2000, n_live=8)
    kc, ks = C.encode_k(_bits(w.k_hist))
    vc, vs = C.encode_v(_bits(w.v_hist))
    exact = oracle.verify_attn(_bits(w.q), _bits(w.k_hist), _bits(w.v_hist), w.pos.numpy(), 8, w.sink.numpy(), w.scale)
    quant = C.verify_attn_decoded(_bits(w.q), C.decode_k(kc, ks), C.decode_v(vc, vs), w.pos.numpy(), 8,
                                  w.sink.numpy(), w.scale)
    rel = np.linalg.norm(quant["out"] - exact["out"]) / np.linalg.norm(exact["out"])
    assert rel < 0.05


def test_the_key_scale_maps_each_row_maximum_to_the_largest_e4m3_value():
    w = synth.make("codec", 8, ctx=400, n_live=4)
    codes, s = C.encode_k(_bits(w.k_hist))
    dec = np.abs(C.e4m3_decode(codes))
    assert np.all(dec.max(axis=1) == C.E4M3_MAX)
    vcodes, _ = C.encode_v(_bits(w.v_hist))
    assert np.all(np.abs(vcodes.astype(np.int64)).max(axis=1) == 127)


def test_an_exactly_representable_cache_reduces_to_the_bf16_oracle():
    # rotated keys r = a e_i + b e_j with a = +-448 and b a small E4M3 value: k = H r / 128 is exact in bf16,
    # the float32 butterfly gives r back exactly, the scale is 1 and the codes are exact, so attention over
    # the decoded cache must equal the bf16-path oracle on the same keys; values are integers with a row
    # maximum of 127 (scale 1, exact codes)
    rng = np.random.default_rng(9)
    ctx, H = 180, hadamard(128).astype(np.float64)
    r = np.zeros((ctx, 128))
    i = rng.integers(0, 128, ctx)
    j = (i + 1 + rng.integers(0, 127, ctx)) % 128
    r[np.arange(ctx), i] = rng.choice([-448.0, 448.0], ctx)
    r[np.arange(ctx), j] = rng.choice([-8.0, -4.0, 2.0, 6.0, 12.0], ctx)
    k = r @ H / 128.0
    v = rng.integers(-126, 127, (ctx, 128)).astype(np.float64)
    v[np.arange(ctx), rng.integers(0, 128, ctx)] = 127.0
    kb, vb = oracle.f64_to_bf16_bits(k), oracle.f64_to_bf16_bits(v)
    assert np.array_equal(oracle.bf16_bits_to_f64(kb), k) and np.array_equal(oracle.bf16_bits_to_f64(vb), v)
    kc, ks = C.encode_k(kb)
    vc, vs = C.encode_v(vb)
    assert np.all(ks == 1.0) and np.all(vs == 1.0)
    np.testing.assert_array_equal(C.decode_k(kc, ks), k)
    np.testing.assert_array_equal(C.decode_v(vc, vs), v)
    w = synth.make("codec", 10, ctx=ctx, n_live=5)
    q = _bits(w.q)
    sink = w.sink.numpy()
    pos = w.pos.numpy()
    got = C.verify_attn_decoded(q, C.decode_k(kc, ks), C.decode_v(vc, vs), pos, 5, sink, 0.01, n_splits=2)
    ref = oracle.verify_attn(q, kb, vb, pos, 5, sink, 0.01)
    np.testing.assert_allclose(got["out"], ref["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["lse"][:5], ref["lse"][:5], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- planted mistakes
def test_planted_codec_mistakes_fail_the_pins(monkeypatch):
    """Each plausible mistake in the codec oracle (planted on the CPU) fails at least one pin above."""
    def no_rotation_on_decode(codes, scales):
        return C.e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]

    def key_scale_by_127(k_bits):
        k = oracle.bf16_bits_to_f64(k_bits).astype(np.float32)
        kr = C.fwht_f32(k)
        s = (np.max(np.abs(kr), axis=-1) / np.float32(127.0)).astype(np.float32)
        return C.e4m3_encode_bits(np.where(s[:, None] > 0, kr / s[:, None], 0).astype(np.float64)), s

    def int8_truncation(v_bits):
        v = oracle.bf16_bits_to_f64(v_bits).astype(np.float32)
        s = (np.max(np.abs(v), axis=-1) / np.float32(127.0)).astype(np.float32)
        ratio = np.where(s[:, None] > 0, (v / s[:, None]).astype(np.float32), np.float32(0))
        return np.clip(np.trunc(ratio), -127, 127).astype(np.int8), s

    real_round = C.e4m3_round

    def e4m3_ties_away(x):
        # round half away from zero instead of half to even
        x = np.asarray(x, dtype=np.float64)
        v, code = real_round(x)
        up, _ = real_round(np.nextafter(np.abs(x), np.inf) * np.sign(x))
        return np.where(np.abs(up) > np.abs(v), up, v), real_round(np.where(np.abs(up) > np.abs(v), up, v))[1]

    cases = [("decode_k", no_rotation_on_decode, test_keys_decode_within_the_e4m3_bound_and_rotated_identity),
             ("encode_k", key_scale_by_127, test_the_key_scale_maps_each_row_maximum_to_the_largest_e4m3_value),
             ("encode_v", int8_truncation, test_int8_values_brute_force_and_error_bound),
             ("e4m3_round", e4m3_ties_away, test_e4m3_rounding_brute_force)]
    for name, wrong, pin in cases:
        with monkeypatch.context() as m:
            m.setattr(C, name, wrong)
            with pytest.raises(AssertionError):
                pin()
