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
