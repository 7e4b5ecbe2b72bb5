"""Bit-exact indexing of the split kernel through its debug build (VA_DEBUG_VISIT): every CTA counts each
(live row, cache slot) pair it lets into the softmax, and the map must equal, exactly, the visible-slot sets
that the positions define (IQuestRT report, "Read only the KV tiles needed by the current positions": each
row sees the valid extent up to its own position, or its window, through the ring; "Let correctness checks
change the design": position labels and visible-position sets).  Full caches, wrapped rings, split counts
with empty splits, and draft trees under their ancestor masks ("Qwen3.8-27B on one RTX 4090", section
"More tokens per round: verify trees")."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decode_verify_gb300 as va
from gpu_cases import DEV, run_step
from speculative_decode_verify_gb300 import build, synth

pytestmark = pytest.mark.gpu
V = "_visit"


@pytest.fixture(scope="module")
def L():
    build.build(variant=V, defines=["VA_DEBUG_VISIT"])
    lib = va.lib(V)
    lib.va_debug_set_visit.argtypes = [ctypes.c_void_p]
    return lib


def _visit_map(L, n_rows, slots, fn):
    buf = torch.zeros(n_rows * slots, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    assert L.va_debug_set_visit(ctypes.c_void_p(buf.data_ptr())) == 0
    try:
        res = fn()
        torch.cuda.synchronize()
    finally:
        L.va_debug_set_visit(None)
    return buf.view(n_rows, slots).cpu().numpy().astype(np.int64), res


@pytest.mark.parametrize("case,S", [("tiny", 4), ("tiny", 1), ("tiny", 40), ("16k", 0), ("swa", 0), ("swa", 9),
                                    ("swa_short", 0), ("swa_offset", 0)])
def test_visit_map_equals_the_visible_slot_sets(L, case, S):
    wrap = 0
    if case == "tiny":
        w = synth.tiny()
    elif case == "16k":
        w = synth.make("visit16k", 2, ctx=16384, n_live=8, slots=65536, peaky_frac=0.05)
    elif case in ("swa", "swa_offset"):
        pos = torch.tensor([39993 + r for r in range(8)], dtype=torch.int32)
        w = synth.make("visitswa", 3, ctx=40000, n_live=7, window=synth.WINDOW, slots=synth.RING_SLOTS, pos=pos)
        wrap = 1234 if case == "swa_offset" else 0
    else:
        pos = torch.tensor([300 + r for r in range(8)], dtype=torch.int32)
        w = synth.make("visitswa_short", 4, ctx=308, n_live=8, window=synth.WINDOW, slots=synth.RING_SLOTS, pos=pos)
    got, res = _visit_map(L, w.n_rows, w.slots, lambda: run_step(w, n_splits=S, wrap_offset=wrap, variant=V))
    assert res["status"] == 0
    ref = oracle.visible_slot_counts(w.pos.numpy().astype(np.int64) + wrap, w.n_live, w.n_rows, w.window, w.slots)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]


@pytest.mark.parametrize("window,n_nodes", [(0, 16), (0, 5), (40, 16)])
def test_tree_visit_map_equals_the_ancestor_sets(L, window, n_nodes):
    w = synth.make_tree("visittree", 5, base=3000 + n_nodes, n_nodes=n_nodes, window=window,
                        slots=synth.RING_SLOTS if window else 0)
    k = torch.full((w.slots, 128), synth.BF16_NAN if not window else synth.BF16_K_SENTINEL, dtype=torch.int16)
    v = torch.full((w.slots, 128), synth.BF16_NAN if not window else synth.BF16_V_SENTINEL, dtype=torch.int16)
    kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
    p = torch.arange(0, w.ctx)
    k[p % w.slots], v[p % w.slots] = kb, vb
    k, v = k.to(DEV), v.to(DEV)
    q = synth.bits(w.q).to(DEV)
    S = 13
    po = torch.empty(S, w.n_rows, 6, 128, device=DEV)
    pl = torch.empty(S, w.n_rows, 6, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, _ = _visit_map(L, w.n_rows, w.slots, lambda: va.verify_attn_tree(q, w.n_nodes, k, v, w.tree.to(DEV), w.scale,
                                                                          po, pl, window=window, n_splits=S,
                                                                          dev_status=status, variant=V))
    assert int(status.item()) == 0
    ref = np.zeros((w.n_rows, w.slots), dtype=np.int64)
    masks = w.masks.numpy()
    for i in range(w.n_nodes):
        for pos_ in oracle.tree_visible_positions(w.base, masks, w.n_nodes, i, window):
            ref[i, pos_ % w.slots] += 1
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]
