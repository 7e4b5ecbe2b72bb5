"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must load, export every function include/*.h declares, reject bad arguments before
launching anything, and agree with the shapes the pages state.
"""
import ctypes
import os
import re

import pytest

import speculative_decode_verify_gb300 as va
from speculative_decode_verify_gb300 import build as vbuild
from speculative_decode_verify_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verify_attn.h")
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    vbuild.build()
    return va.lib()


def _declared():
    names = []
    for h in HEADERS:
        names += re.findall(r"VA_API\s+[\w\s\*]+?\b(\w+)\s*\(", open(h).read())
    return names


def _defines():
    src = "".join(open(h).read() for h in HEADERS)
    return {k: int(v) for k, v in re.findall(r"#define\s+(VA_\w+)\s+(-?\d+)\b", src)}


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("kv_ring_append", "verify_attn_full", "verify_attn_swa", "attn_split_combine"):
        assert n in names
    assert set(names) == set(va.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_binding_constants_match_header():
    d = _defines()
    assert (d["VA_HEAD_DIM"], d["VA_Q_HEADS"], d["VA_MAX_ROWS"], d["VA_TILE"], d["VA_MAX_SPLITS"]) == \
        (va.HEAD_DIM, va.Q_HEADS, va.MAX_ROWS, va.TILE, va.MAX_SPLITS)
    assert (d["VA_OK"], d["VA_INVALID_ARG"], d["VA_UNSUPPORTED"], d["VA_RING_TOO_SMALL"], d["VA_CUDA_ERROR"]) == \
        (va.VA_OK, va.VA_INVALID_ARG, va.VA_UNSUPPORTED, va.VA_RING_TOO_SMALL, va.VA_CUDA_ERROR)
    # the binding's copies of the other limits must not drift from the headers
    assert d["VA_NOALLOC_MAX_SPLITS"] == va.NOALLOC_MAX_SPLITS
    assert d["VA_MAX_TREE_NODES"] == va.MAX_TREE_NODES
    assert (d["VA_SAMPLE_MAX_K"], d["VA_SAMPLE_TILE"], d["VA_SAMPLE_MAX_VOCAB"]) == \
        (va.SAMPLE_MAX_K, va.SAMPLE_TILE, va.SAMPLE_MAX_VOCAB)


def test_page_constants_golden():
    g = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "page_constants.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            g[k] = int(v)
    d = _defines()
    assert d["VA_Q_HEADS"] == g["query_heads"] and d["VA_MAX_ROWS"] == g["verify_rows"]
    assert d["VA_Q_HEADS"] * d["VA_MAX_ROWS"] == g["matrix_rows"]
    assert synth.WINDOW == g["window"] and synth.RING_SLOTS == g["ring_slots"]
    assert g["ring_slots"] == g["window"] + g["ring_extra_tile"] and d["VA_TILE"] == g["ring_extra_tile"]
    # the enlarged ring keeps every live row's window when all eight rows are appended first
    assert g["ring_slots"] >= g["window"] + g["verify_rows"] - 1
    assert g["window"] < g["window"] + g["verify_rows"] - 1


# fake, never-dereferenced addresses: every call below must be rejected before any launch
FAKE = ctypes.c_void_p(0x1000)


def _full(L, **kw):
    a = dict(q=FAKE, n_rows=8, n_live=5, k=FAKE, v=FAKE, cap=1024, pos=FAKE, scale=0.088, S=4, po=FAKE, pl=FAKE)
    a.update(kw)
    return L.verify_attn_full(a["q"], a["n_rows"], a["n_live"], a["k"], a["v"], a["cap"], a["pos"], a["scale"],
                              a["S"], a["po"], a["pl"], None, None, None)


def _swa(L, **kw):
    a = dict(q=FAKE, n_rows=8, n_live=8, k=FAKE, v=FAKE, R=4160, W=4096, pos=FAKE, scale=0.088, S=4,
             po=FAKE, pl=FAKE)
    a.update(kw)
    return L.verify_attn_swa(a["q"], a["n_rows"], a["n_live"], a["k"], a["v"], a["R"], a["W"], a["pos"],
                             a["scale"], a["S"], a["po"], a["pl"], None, None, None)


@pytest.mark.parametrize("kw", [dict(q=None), dict(k=None), dict(pos=None), dict(po=None), dict(pl=None),
                                dict(n_rows=0), dict(n_rows=9), dict(n_live=-1), dict(n_live=9),
                                dict(cap=0), dict(S=-1), dict(S=4097), dict(scale=float("nan")),
                                dict(scale=float("inf"))])
def test_full_rejects_bad_arguments(L, kw):
    assert _full(L, **kw) == va.VA_INVALID_ARG


def test_misaligned_pointers_are_rejected(L):
    odd = ctypes.c_void_p(0x1002)
    assert _full(L, q=odd) == va.VA_INVALID_ARG
    assert _full(L, k=odd) == va.VA_INVALID_ARG
    assert _full(L, po=odd) == va.VA_INVALID_ARG
    assert _swa(L, v=odd) == va.VA_INVALID_ARG
    assert L.kv_ring_append(odd, FAKE, 2, FAKE, FAKE, 64, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.attn_split_combine(FAKE, FAKE, 4, None, 8, 8, odd, None, None) == va.VA_INVALID_ARG


def test_swa_ring_checks(L):
    assert _swa(L, R=4100) == va.VA_UNSUPPORTED                 # not a multiple of 64
    assert _swa(L, R=4096) == va.VA_RING_TOO_SMALL              # the ring the pages fixed
    assert _swa(L, R=4096, n_live=1, q=None) == va.VA_INVALID_ARG
    assert _swa(L, W=0) == va.VA_INVALID_ARG
    assert _swa(L, R=4160, n_live=8, W=4160 - 6) == va.VA_RING_TOO_SMALL   # needs W + 7 slots


def test_append_and_combine_reject_bad_arguments(L):
    assert L.kv_ring_append(FAKE, FAKE, 17, FAKE, FAKE, 64, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.kv_ring_append(FAKE, FAKE, 2, FAKE, FAKE, 0, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.kv_ring_append(None, FAKE, 2, FAKE, FAKE, 64, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.kv_ring_append(None, None, 0, None, None, 64, None, None, None) == va.VA_OK   # nothing to do
    assert L.attn_split_combine(FAKE, FAKE, 4, None, 8, 8, None, None, None) == va.VA_INVALID_ARG
    assert L.attn_split_combine(None, FAKE, 4, None, 8, 8, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.attn_split_combine(FAKE, FAKE, 4097, None, 8, 8, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.attn_split_combine(FAKE, FAKE, 4, None, 8, 9, FAKE, None, None) == va.VA_INVALID_ARG
    assert L.attn_split_combine(FAKE, FAKE, 4, None, 17, 8, FAKE, None, None) == va.VA_INVALID_ARG


def _tree(L, **kw):
    a = dict(q=FAKE, n_rows=16, n_nodes=16, k=FAKE, v=FAKE, slots=4160, W=4096, tree=FAKE, scale=0.088, S=4,
             po=FAKE, pl=FAKE)
    a.update(kw)
    return L.verify_attn_tree(a["q"], a["n_rows"], a["n_nodes"], a["k"], a["v"], a["slots"], a["W"], a["tree"],
                              a["scale"], a["S"], a["po"], a["pl"], None, None, None)


@pytest.mark.parametrize("kw", [dict(q=None), dict(tree=None), dict(k=None), dict(po=None), dict(n_rows=0),
                                dict(n_rows=17), dict(n_nodes=-1), dict(n_nodes=17), dict(n_rows=8, n_nodes=9),
                                dict(slots=0), dict(W=-1), dict(S=-1), dict(S=4097),
                                dict(scale=float("nan")), dict(q=ctypes.c_void_p(0x1008))])
def test_tree_rejects_bad_arguments(L, kw):
    assert _tree(L, **kw) == va.VA_INVALID_ARG


def test_tree_window_and_ring_checks(L):
    assert _tree(L, W=15) == va.VA_UNSUPPORTED            # a window shorter than the tree
    assert _tree(L, slots=4100) == va.VA_UNSUPPORTED      # ring not a multiple of 64
    assert _tree(L, slots=4096) == va.VA_RING_TOO_SMALL   # needs W + 15 slots
    assert _tree(L, W=4160 - 14) == va.VA_RING_TOO_SMALL


def test_workspace_and_status_strings(L):
    assert va.va_workspace_bytes(0) == 0 and va.va_workspace_bytes(4097) == 0
    assert va.va_workspace_bytes(152) == 4 * 152 * 8 * 6 * 129
    assert va.va_status_string(va.VA_RING_TOO_SMALL) == "VA_RING_TOO_SMALL"
    assert va.va_status_string(99) == "VA_UNKNOWN_STATUS"


def test_auto_split_policy(L):
    for sm in (148, 152):
        assert va.va_auto_splits_for(196608, 0, sm) == sm          # long context fills every SM
        prev = 0
        for ext in (1, 64, 128, 1024, 4096, 16384, 65536, 196608, 1 << 30):
            s = va.va_auto_splits_for(ext, 0, sm)
            assert 1 <= s <= sm and s >= prev
            prev = s
        s_swa = va.va_auto_splits_for(4103, 4096, sm)
        assert s_swa == va.va_auto_splits_for(10 ** 6, 4096, sm)   # a window bounds the work
        assert 1 <= s_swa <= sm


# ----------------------------------------------------------------------------- sampling, acceptance, settlement
def test_sample_workspace_and_argument_checks(L):
    # the row counters first (256 B, the same place for every shape), then 20 tiles x 20 keys x 8 B per row
    assert va.va_sample_workspace_bytes(8, 160000, 20) == 256 + 8 * 20 * 20 * 8
    assert va.va_sample_workspace_bytes(64, 160000, 20) == 256 + 64 * 20 * 20 * 8
    assert va.va_sample_workspace_bytes(65, 160000, 20) == 0
    assert va.va_sample_workspace_bytes(0, 160000, 20) == 0
    assert va.va_sample_workspace_bytes(8, 160000, 33) == 0
    assert va.va_sample_workspace_bytes(8, 262148, 20) == 0
    assert va.va_sample_workspace_bytes(8, 10, 20) == 0
    f = ctypes.c_float
    ok = dict(x=FAKE, n=8, vocab=160000, k=20, p=0.95, T=1.0, u=FAKE, ws=FAKE, wsb=25632)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return L.va_sample_topk_topp(a["x"], a["n"], a["vocab"], a["k"], f(a["p"]), f(a["T"]), a["u"], FAKE, FAKE,
                                     FAKE, FAKE, a["ws"], a["wsb"], None)
    for kw in (dict(x=None), dict(u=None), dict(ws=None), dict(wsb=25631), dict(vocab=160002), dict(p=0.0),
               dict(p=1.5), dict(T=0.0), dict(T=-1.0), dict(k=0), dict(n=65), dict(x=ctypes.c_void_p(0x1004))):
        assert call(**kw) == va.VA_INVALID_ARG, kw


def test_accept_and_settle_argument_checks(L):
    a = [FAKE] * 6 + [20, FAKE, FAKE, 7, FAKE, FAKE, FAKE, FAKE, FAKE, None, None]
    bad = list(a)
    bad[9] = 64                                                    # n_drafts out of range
    assert L.va_accept_chain(*bad) == va.VA_INVALID_ARG
    bad = list(a)
    bad[6] = 33                                                    # k_stride out of range
    assert L.va_accept_chain(*bad) == va.VA_INVALID_ARG
    bad = list(a)
    bad[3] = None                                                  # q needed when there are drafts
    assert L.va_accept_chain(*bad) == va.VA_INVALID_ARG
    s = [FAKE, FAKE, 64, FAKE, 16, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None]
    for i, v in ((4, 17), (4, 0), (3, None), (2, 0), (1, None), (0, ctypes.c_void_p(0x1008))):
        bad = list(s)
        bad[i] = v
        assert L.va_tree_accept_settle(*bad) == va.VA_INVALID_ARG, (i, v)


def _step(L, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, n_rows=8, n_live=8, k=FAKE, v=FAKE, slots=4160, W=4096, pos=FAKE, sink=None,
             scale=0.088, S=4, ws=FAKE, out=FAKE)
    a.update(kw)
    return L.verify_attn_step(a["q"], a["kn"], a["vn"], a["n_rows"], a["n_live"], a["k"], a["v"], a["slots"], a["W"],
                              a["pos"], a["sink"], a["scale"], a["S"], a["ws"], a["out"], None, None, None, None)


@pytest.mark.parametrize("kw", [dict(out=None), dict(out=ctypes.c_void_p(0x1002)), dict(kn=None), dict(vn=None),
                                dict(kn=ctypes.c_void_p(0x1004)), dict(W=-1), dict(S=-1), dict(S=4097), dict(ws=None),
                                dict(q=None), dict(k=None), dict(pos=None), dict(n_rows=0), dict(n_rows=9),
                                dict(n_live=9), dict(n_live=-1), dict(slots=0), dict(scale=float("nan"))])
def test_step_rejects_bad_arguments(L, kw):
    assert _step(L, **kw) == va.VA_INVALID_ARG


def test_step_ring_checks(L):
    assert _step(L, slots=4100) == va.VA_UNSUPPORTED            # a ring must hold whole 64-position tiles
    assert _step(L, slots=4096) == va.VA_RING_TOO_SMALL         # needs W + n_live - 1 slots
    assert _step(L, slots=4160, W=4160 - 6) == va.VA_RING_TOO_SMALL


def _q8(L, **kw):
    a = dict(q=FAKE, n_rows=8, n_live=8, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, slots=4160, W=4096, pos=FAKE,
             scale=0.088, S=4, po=FAKE, pl=FAKE)
    a.update(kw)
    return L.verify_attn_q8(a["q"], a["n_rows"], a["n_live"], a["kc"], a["vc"], a["ks"], a["vs"], a["slots"], a["W"],
                            a["pos"], a["scale"], a["S"], a["po"], a["pl"], None, None, None)


@pytest.mark.parametrize("kw", [dict(q=None), dict(kc=None), dict(vc=None), dict(ks=None), dict(vs=None),
                                dict(pos=None), dict(po=None), dict(pl=None), dict(ks=ctypes.c_void_p(0x1004)),
                                dict(n_rows=0), dict(n_rows=9), dict(n_live=9), dict(n_live=-1), dict(slots=0),
                                dict(W=-1), dict(S=-1), dict(S=4097), dict(scale=float("inf"))])
def test_q8_rejects_bad_arguments(L, kw):
    assert _q8(L, **kw) == va.VA_INVALID_ARG


def test_q8_ring_checks(L):
    assert _q8(L, slots=4100) == va.VA_UNSUPPORTED
    assert _q8(L, slots=4100, W=0) == va.VA_UNSUPPORTED           # the quantised cache is tiled in 64 rows
    assert _q8(L, slots=4096) == va.VA_RING_TOO_SMALL


def _q8_tree(L, **kw):
    a = dict(q=FAKE, n_rows=16, n_nodes=16, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, slots=4160, W=4096, tree=FAKE,
             scale=0.088, S=4, po=FAKE, pl=FAKE)
    a.update(kw)
    return L.verify_attn_q8_tree(a["q"], a["n_rows"], a["n_nodes"], a["kc"], a["vc"], a["ks"], a["vs"], a["slots"],
                                 a["W"], a["tree"], a["scale"], a["S"], a["po"], a["pl"], None, None, None)


@pytest.mark.parametrize("kw", [dict(q=None), dict(tree=None), dict(kc=None), dict(vs=None), dict(po=None),
                                dict(n_rows=0), dict(n_rows=17), dict(n_nodes=-1), dict(n_nodes=17),
                                dict(n_rows=8, n_nodes=9), dict(slots=0), dict(W=-1), dict(S=-1), dict(S=4097),
                                dict(scale=float("nan")), dict(vc=ctypes.c_void_p(0x1008))])
def test_q8_tree_rejects_bad_arguments(L, kw):
    assert _q8_tree(L, **kw) == va.VA_INVALID_ARG


def test_q8_tree_window_and_ring_checks(L):
    assert _q8_tree(L, W=15) == va.VA_UNSUPPORTED            # a window shorter than the tree
    assert _q8_tree(L, slots=4100) == va.VA_UNSUPPORTED      # not a multiple of 64
    assert _q8_tree(L, slots=4100, W=0) == va.VA_UNSUPPORTED
    assert _q8_tree(L, slots=4096) == va.VA_RING_TOO_SMALL   # needs W + 15 slots


def test_q8_append_argument_checks(L):
    def call(n=4, kn=FAKE, kc=FAKE, ks=FAKE, slots=4160, pos=FAKE):
        return L.kv_ring_append_q8(kn, FAKE, n, kc, FAKE, ks, FAKE, slots, pos, None, None)
    assert call(n=-1) == va.VA_INVALID_ARG
    assert call(n=16777217) == va.VA_INVALID_ARG
    assert call(slots=0) == va.VA_INVALID_ARG
    assert call(slots=100) == va.VA_UNSUPPORTED
    assert call(kn=None) == va.VA_INVALID_ARG
    assert call(pos=None) == va.VA_INVALID_ARG
    assert call(ks=ctypes.c_void_p(0x1004)) == va.VA_INVALID_ARG
    assert call(n=0, kn=None, kc=None, ks=None, pos=None) == va.VA_OK   # nothing to encode, nothing launched


def test_bounded_wait_selftest_argument_checks(L):
    assert L.va_selftest_bounded_wait(0, 0, None, None, None) == va.VA_INVALID_ARG
    assert L.va_selftest_bounded_wait(1_000_000_001, 0, None, None, None) == va.VA_INVALID_ARG
    assert L.va_selftest_bounded_wait(1_000_000, 1_000_001, None, None, None) == va.VA_INVALID_ARG


def _q8_step(L, **kw):
    a = dict(q=FAKE, kn=FAKE, vn=FAKE, n_rows=8, n_live=8, kc=FAKE, vc=FAKE, ks=FAKE, vs=FAKE, slots=4160, W=4096,
             pos=FAKE, sink=None, scale=0.088, S=4, ws=FAKE, out=FAKE)
    a.update(kw)
    return L.verify_attn_q8_step(a["q"], a["kn"], a["vn"], a["n_rows"], a["n_live"], a["kc"], a["vc"], a["ks"],
                                 a["vs"], a["slots"], a["W"], a["pos"], a["sink"], a["scale"], a["S"], a["ws"],
                                 a["out"], None, None, None, None)


@pytest.mark.parametrize("kw", [dict(out=None), dict(ws=None), dict(ws=ctypes.c_void_p(0x1004)), dict(kn=None),
                                dict(vn=ctypes.c_void_p(0x1008)), dict(q=None), dict(kc=None), dict(vs=None),
                                dict(pos=None), dict(ks=ctypes.c_void_p(0x1004)), dict(n_rows=0), dict(n_rows=9),
                                dict(n_live=9), dict(n_live=-1), dict(slots=0), dict(W=-1), dict(S=-1),
                                dict(S=4097), dict(scale=float("nan"))])
def test_q8_step_rejects_bad_arguments(L, kw):
    assert _q8_step(L, **kw) == va.VA_INVALID_ARG


def test_q8_step_ring_checks(L):
    assert _q8_step(L, slots=4100) == va.VA_UNSUPPORTED
    assert _q8_step(L, slots=4100, W=0) == va.VA_UNSUPPORTED
    assert _q8_step(L, slots=4096) == va.VA_RING_TOO_SMALL
