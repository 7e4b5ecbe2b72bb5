"""GPU parity of the quantised K/V cache: the encoding append bit for bit, and verify attention over the
cache against the FP64 oracle over the decoded cache ("Qwen3.8-27B on one RTX 4090", section "A cheaper
cache and state").

The history is encoded on the host by the oracle's encoder (the append kernel matches it bit for bit, see
the first tests), the live rows are appended by kv_ring_append_q8, then verify_attn_q8 + attn_split_combine
run through the C ABI.  Bars as for the bf16 path (tests/parity.py), against the oracle's attention over the
decoded keys and values rounded once to bf16.  Slots the kernel must not use hold NaN codes and NaN scales.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from oracle import kv_codec as C
from speculative_decode_verify_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAN_CODE = 0x7F


def _rows(seed, n):
    """bf16 rows with the cases the encoder must get right: ordinary, large, tiny, zero, signed zeros."""
    g = synth.generator(seed)
    x = torch.randn(n, 128, generator=g, dtype=torch.float32)
    x[1] *= 300.0
    x[2] *= 1e-6
    x[3] = 0.0
    x[4, ::2] = -0.0
    x[5, :64] = 0.0
    x[6] = torch.where(torch.rand(128, generator=g) < 0.5, 1e-3, -2.5)
    return synth.bits(x.to(torch.bfloat16))


@pytest.mark.parametrize("slots", [64, 4160])
def test_append_encodes_bit_for_bit(slots):
    n = 16
    kb, vb = _rows(1, n), _rows(2, n)
    pos = torch.tensor([slots * 3 + 5 + i for i in range(n)], dtype=torch.int32)   # wraps the ring
    kc = torch.full((slots, 128), NAN_CODE, dtype=torch.uint8, device=DEV)
    vc = torch.full((slots, 128), -1, dtype=torch.int8, device=DEV)
    ks = torch.full((slots,), float("nan"), device=DEV)
    vs = torch.full((slots,), float("nan"), device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    va.kv_ring_append_q8(kb.to(DEV), vb.to(DEV), n, kc, vc, ks, vs, pos.to(DEV), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rk, rks = C.encode_k(kb.numpy())
    rv, rvs = C.encode_v(vb.numpy())
    slot = (pos.numpy().astype(np.int64) % slots)
    np.testing.assert_array_equal(kc.cpu().numpy()[slot], rk)
    np.testing.assert_array_equal(vc.cpu().numpy()[slot], rv)
    np.testing.assert_array_equal(ks.cpu().numpy()[slot].view(np.uint32), rks.view(np.uint32))
    np.testing.assert_array_equal(vs.cpu().numpy()[slot].view(np.uint32), rvs.view(np.uint32))
    untouched = np.setdiff1d(np.arange(slots), slot)
    assert np.all(kc.cpu().numpy()[untouched] == NAN_CODE)


def test_append_encodes_a_large_random_batch_bit_for_bit():
    for seed in range(20):
        kb = synth.bits(synth.normal_bf16((16, 128), synth.generator(100 + seed), scale=float(10 ** (seed % 5 - 2))))
        vb = synth.bits(synth.normal_bf16((16, 128), synth.generator(200 + seed)))
        kc = torch.zeros(64, 128, dtype=torch.uint8, device=DEV)
        vc = torch.zeros(64, 128, dtype=torch.int8, device=DEV)
        ks = torch.zeros(64, device=DEV)
        vs = torch.zeros(64, device=DEV)
        pos = torch.arange(16, dtype=torch.int32, device=DEV)
        va.kv_ring_append_q8(kb.to(DEV), vb.to(DEV), 16, kc, vc, ks, vs, pos)
        torch.cuda.synchronize()
        rk, rks = C.encode_k(kb.numpy())
        rv, rvs = C.encode_v(vb.numpy())
        np.testing.assert_array_equal(kc.cpu().numpy()[:16], rk)
        np.testing.assert_array_equal(vc.cpu().numpy()[:16], rv)
        np.testing.assert_array_equal(ks.cpu().numpy()[:16], rks)
        np.testing.assert_array_equal(vs.cpu().numpy()[:16], rvs)


def _encoded_cache(w, slots, upto):
    """Host-encoded cache holding positions [first, upto) (full: from 0) at slot p mod slots; NaN codes
    and scales elsewhere."""
    kc = np.full((slots, 128), NAN_CODE, dtype=np.uint8)
    vc = np.full((slots, 128), -128, dtype=np.int8)
    ks = np.full(slots, np.nan, dtype=np.float32)
    vs = np.full(slots, np.nan, dtype=np.float32)
    first = max(0, upto - slots) if w.window else 0
    if upto > first:
        k_codes, k_s = C.encode_k(synth.bits(w.k_hist[first:upto]).numpy())
        v_codes, v_s = C.encode_v(synth.bits(w.v_hist[first:upto]).numpy())
        sl = np.arange(first, upto) % slots
        kc[sl], vc[sl], ks[sl], vs[sl] = k_codes, v_codes, k_s, v_s
    return [torch.from_numpy(a).to(DEV) for a in (kc, vc, ks, vs)]


def run_q8(w, n_splits=0):
    slots = w.slots
    p0 = int(w.pos[0])
    kc, vc, ks, vs = _encoded_cache(w, slots, p0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = w.pos[:w.n_live].to(torch.int64)
    va.kv_ring_append_q8(synth.bits(w.k_hist)[idx].contiguous().to(DEV), synth.bits(w.v_hist)[idx].contiguous().to(DEV),
                         w.n_live, kc, vc, ks, vs, w.pos.to(DEV), dev_status=status)
    cap = n_splits if n_splits else torch.cuda.get_device_properties(0).multi_processor_count
    part_o = torch.full((cap, w.n_rows, 6, 128), float("nan"), device=DEV)
    part_lse = torch.full((cap, w.n_rows, 6), float("nan"), device=DEV)
    used = va.verify_attn_q8(synth.bits(w.q).to(DEV), w.n_live, kc, vc, ks, vs, w.pos.to(DEV), w.scale, part_o,
                             part_lse, window=w.window, n_splits=n_splits, dev_status=status)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), device=DEV)
    va.attn_split_combine(part_o[:used], part_lse[:used], used, w.sink.to(DEV), w.n_live, out, out_lse)
    torch.cuda.synchronize()
    return dict(out=oracle.bf16_bits_to_f64(out.cpu().numpy()), out_bits=out.cpu().numpy().view(np.uint16),
                out_lse=out_lse.cpu().numpy().astype(np.float64), part_lse=part_lse[:used].cpu().numpy(),
                part_o=part_o[:used].cpu().numpy(), n_splits=used, status=int(status.item()))


def expected_q8(w, n_splits):
    kcodes, kscale = C.encode_k(synth.bits(w.k_hist).numpy())
    vcodes, vscale = C.encode_v(synth.bits(w.v_hist).numpy())
    res = C.verify_attn_decoded(synth.bits(w.q).numpy(), C.decode_k(kcodes, kscale), C.decode_v(vcodes, vscale),
                                w.pos.numpy(), w.n_live, w.sink.numpy(), w.scale, w.window, n_splits=n_splits,
                                n_threads=8)
    res["out_bf16"] = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(res["out"]))
    return res


def _assert(got, ref, w):
    assert got["status"] == 0, hex(got["status"])
    m = parity.out_metrics(got["out"], ref["out_bf16"], w.n_live, exact=ref["out"])
    assert parity.out_ok(m), m
    assert parity.lse_err(got["out_lse"][:w.n_live], ref["lse"][:w.n_live]) <= parity.LSE_ABS
    assert np.all(got["out_bits"][w.n_live:] == 0)
    assert parity.lse_err(got["part_lse"], ref["part_lse"]) <= parity.LSE_ABS
    assert np.abs(got["part_o"] - ref["part_o"]).max() <= parity.OUT_MAX_ABS
    return m


@pytest.mark.parametrize("S", [1, 3, 4, 16])
def test_q8_small_full(S):
    w = synth.make("q8", 31, ctx=1024, n_live=5, slots=1088, pos=torch.arange(1016, 1024, dtype=torch.int32))
    _assert(run_q8(w, S), expected_q8(w, S), w)


@pytest.mark.parametrize("n_live", [1, 4, 8])
def test_q8_16k_peaky_auto_splits(n_live):
    w = synth.make("q8_16k", 32 + n_live, ctx=16384, n_live=n_live, slots=65536, peaky_frac=0.05)
    got = run_q8(w)
    _assert(got, expected_q8(w, got["n_splits"]), w)


@pytest.mark.parametrize("ctx,n_live", [(40000, 7), (4200, 8), (300, 3)])
def test_q8_sliding_window_ring(ctx, n_live):
    pos = torch.tensor([ctx - n_live + r for r in range(8)], dtype=torch.int32)
    w = synth.make("q8_swa", 40 + n_live, ctx=ctx, n_live=n_live, window=synth.WINDOW, slots=synth.RING_SLOTS, pos=pos)
    got = run_q8(w)
    _assert(got, expected_q8(w, got["n_splits"]), w)


def test_q8_192k_full():
    w = synth.full_192k(8)
    w.slots = 196672
    got = run_q8(w)
    _assert(got, expected_q8(w, got["n_splits"]), w)


def test_q8_rejects_and_flags():
    q = torch.zeros(8, 6, 128, dtype=torch.int16, device=DEV)
    kc = torch.zeros(100, 128, dtype=torch.uint8, device=DEV)     # not a multiple of 64
    vc = torch.zeros(100, 128, dtype=torch.int8, device=DEV)
    s = torch.zeros(100, device=DEV)
    po = torch.empty(4, 8, 6, 128, device=DEV)
    pl = torch.empty(4, 8, 6, device=DEV)
    pos = torch.arange(8, dtype=torch.int32, device=DEV)
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_q8(q, 8, kc, vc, s, s, pos, 0.088, po, pl, n_splits=4)
    kc = torch.zeros(128, 128, dtype=torch.uint8, device=DEV)
    vc = torch.zeros(128, 128, dtype=torch.int8, device=DEV)
    s = torch.zeros(128, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = torch.tensor([200 + i for i in range(8)], dtype=torch.int32, device=DEV)   # beyond the capacity
    va.verify_attn_q8(q, 8, kc, vc, s, s, bad, 0.088, po, pl, n_splits=4, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4
    assert torch.all(torch.isneginf(pl))
