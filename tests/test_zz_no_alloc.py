"""verify_attn_full_noalloc against the allocating entry points.

Some callers of this library cannot allocate device memory when they call it: a decode loop embedded in
another runtime that hands it only tensors and a stream (and no allocator), or a latency-critical loop
that must not call cudaMalloc because cudaMalloc can synchronise the device.  verify_attn_full_noalloc
serves them by keeping the split partials in a fixed device buffer owned by the library.  Its output
must equal that of verify_attn_full + attn_split_combine with caller-allocated partials, call after call
(the shared buffer keeps the previous call's contents).

This file is named to be collected last, so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decode_verify_gb300 as va
from speculative_decode_verify_gb300 import build as vbuild
from speculative_decode_verify_gb300 import synth


def test_noalloc_rejects_split_counts_beyond_its_buffer():
    vbuild.build()
    L = va.lib()
    fake = ctypes.c_void_p(0x1000)
    st = L.verify_attn_full_noalloc(fake, 8, 8, fake, fake, 1024, fake, ctypes.c_float(0.088),
                                    va.NOALLOC_MAX_SPLITS + 1, None, fake, None, None, None, None)
    assert st == va.VA_INVALID_ARG
    st = L.verify_attn_full_noalloc(None, 8, 8, fake, fake, 1024, fake, ctypes.c_float(0.088), 4, None, fake,
                                    None, None, None, None)
    assert st == va.VA_INVALID_ARG


def _device_case(w, dev):
    """Full cache with the history in place and NaN beyond the live extent."""
    kc = torch.full((w.slots, 128), synth.BF16_NAN, dtype=torch.int16)
    vc = torch.full((w.slots, 128), synth.BF16_NAN, dtype=torch.int16)
    lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, 0)
    kc[:hi] = synth.bits(w.k_hist)[:hi]
    vc[:hi] = synth.bits(w.v_hist)[:hi]
    return dict(q=synth.bits(w.q).to(dev), k=kc.to(dev), v=vc.to(dev), pos=w.pos.to(dev), sink=w.sink.to(dev),
                hi=hi)


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_points_on_consecutive_calls():
    vbuild.build()
    L = va.lib()
    dev = torch.device("cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    cases = [synth.full_16k(), synth.make("noalloc", 43, ctx=5000, n_live=6, slots=5120)]
    for w in cases:   # two calls in a row, different shapes: the shared buffer is reused
        c = _device_case(w, dev)
        S = va.va_auto_splits(c["hi"], 0)
        # allocating entry points
        part_o = torch.empty(S, w.n_rows, 6, 128, dtype=torch.float32, device=dev)
        part_lse = torch.empty(S, w.n_rows, 6, dtype=torch.float32, device=dev)
        ref = torch.empty(w.n_rows, 6, 128, dtype=torch.int16, device=dev)
        ref_lse = torch.empty(w.n_rows, 6, dtype=torch.float32, device=dev)
        va.verify_attn_full(c["q"], w.n_live, c["k"], c["v"], c["pos"], w.scale, part_o, part_lse, S)
        va.attn_split_combine(part_o, part_lse, S, c["sink"], w.n_live, ref, ref_lse)
        # the no-alloc entry point through the C ABI
        out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=dev)
        out_lse = torch.full((w.n_rows, 6), float("nan"), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        used = ctypes.c_int(0)
        st = L.verify_attn_full_noalloc(P(c["q"]), w.n_rows, w.n_live, P(c["k"]), P(c["v"]), w.slots, P(c["pos"]),
                                        ctypes.c_float(w.scale), S, P(c["sink"]), P(out), P(out_lse),
                                        ctypes.byref(used), P(status),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == va.VA_OK and used.value == S
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = oracle.bf16_bits_to_f64(out.cpu().numpy())
        exp = oracle.bf16_bits_to_f64(ref.cpu().numpy())
        m = parity.out_metrics(got, exp, w.n_live, exact=exp)
        assert parity.out_ok(m), m
        assert parity.lse_err(out_lse.cpu().numpy()[:w.n_live], ref_lse.cpu().numpy()[:w.n_live]) <= parity.LSE_ABS
        assert np.all(out.cpu().numpy()[w.n_live:] == 0)
        # and against the FP64 oracle directly
        o = oracle.verify_attn(synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(), synth.bits(w.v_hist).numpy(),
                               w.pos.numpy(), w.n_live, w.sink.numpy(), w.scale, 0, n_splits=S, n_threads=8)
        m = parity.out_metrics(got, oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(o["out"])), w.n_live,
                               exact=o["out"])
        assert parity.out_ok(m), m
        assert parity.lse_err(out_lse.cpu().numpy()[:w.n_live], o["lse"][:w.n_live]) <= parity.LSE_ABS


@pytest.mark.gpu
def test_noalloc_auto_split_count():
    # n_splits = 0: the library's own choice, capped at the fixed buffer's limit
    vbuild.build()
    L = va.lib()
    dev = torch.device("cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    w = synth.make("noalloc_auto", 44, ctx=3000, n_live=5, slots=9000)
    c = _device_case(w, dev)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=dev)
    out_lse = torch.full((w.n_rows, 6), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    used = ctypes.c_int(0)
    for _ in range(2):
        st = L.verify_attn_full_noalloc(P(c["q"]), w.n_rows, w.n_live, P(c["k"]), P(c["v"]), w.slots, P(c["pos"]),
                                        ctypes.c_float(w.scale), 0, P(c["sink"]), P(out), P(out_lse),
                                        ctypes.byref(used), P(status),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == va.VA_OK
        assert used.value == min(va.va_auto_splits(w.slots, 0), va.NOALLOC_MAX_SPLITS)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o = oracle.verify_attn(synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(), synth.bits(w.v_hist).numpy(),
                               w.pos.numpy(), w.n_live, w.sink.numpy(), w.scale, 0, n_splits=used.value, n_threads=8)
        got = oracle.bf16_bits_to_f64(out.cpu().numpy())
        m = parity.out_metrics(got, oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(o["out"])), w.n_live,
                               exact=o["out"])
        assert parity.out_ok(m), m
        assert np.all(out.cpu().numpy()[w.n_live:] == 0)
