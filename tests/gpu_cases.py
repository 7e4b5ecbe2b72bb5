"""Helpers shared by the GPU tests: device state for a workload, the CUDA path through the C ABI,
and the oracle's expected values for the same seeded inputs."""
import numpy as np
import torch

import oracle
import speculative_decode_verify_gb300 as va
from speculative_decode_verify_gb300 import synth

DEV = "cuda"


def _bits_np(t):
    return synth.bits(t).numpy()


def cache_state(w: synth.Workload, history_upto: int, placement: str = "all", wrap_offset: int = 0):
    """Device K/V caches holding the history positions [.., history_upto) of w.

    full attention: a [slots,128] cache, row j = position j; rows >= the live extent hold NaN when
    w.poison_tail, else whatever the generated history has there.
    sliding window: a ring filled with finite sentinels (K = 64, V = 1000); placement "all" writes
    the last `slots` history positions, "window" only those row 0's window needs.  Position p lives
    in slot (p + wrap_offset) mod slots when wrap_offset != 0 (a placement-invariance check; the
    positions passed to the kernels are shifted by the same amount then).
    """
    slots = w.slots
    if w.window == 0:
        k = torch.full((slots, 128), 0, dtype=torch.int16)
        v = torch.full((slots, 128), 0, dtype=torch.int16)
        kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
        n = min(w.ctx, slots)
        k[:n] = kb[:n]
        v[:n] = vb[:n]
        lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, 0)
        if w.poison_tail:
            k[hi:] = synth.BF16_NAN
            v[hi:] = synth.BF16_NAN
        else:
            k[n:] = synth.BF16_NAN
            v[n:] = synth.BF16_NAN
        # rows of the live positions are written by the append under test
        for r in range(w.n_live):
            p = int(w.pos[r])
            if p >= history_upto:
                k[p] = synth.BF16_NAN
                v[p] = synth.BF16_NAN
        return k.to(DEV), v.to(DEV)
    k = torch.full((slots, 128), synth.BF16_K_SENTINEL, dtype=torch.int16)
    v = torch.full((slots, 128), synth.BF16_V_SENTINEL, dtype=torch.int16)
    kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
    if placement == "all":
        first = max(0, history_upto - slots)
    else:
        first = max(0, int(w.pos[0]) - w.window + 1)
    p = torch.arange(first, history_upto)
    s = (p + wrap_offset) % slots
    k[s] = kb[first:history_upto]
    v[s] = vb[first:history_upto]
    return k.to(DEV), v.to(DEV)


def run_step(w: synth.Workload, n_splits: int = 0, placement: str = "all", wrap_offset: int = 0,
             append: bool = True, variant: str = ""):
    """append (optional) + split attention + combine through the C ABI.  Returns host numpy dict."""
    pos_dev = (w.pos.to(torch.int64) + wrap_offset).to(torch.int32).to(DEV) if wrap_offset else w.pos.to(DEV)
    history_upto = int(w.pos[0]) if append else int(w.pos[w.n_live - 1]) + 1
    k, v = cache_state(w, history_upto, placement, wrap_offset)
    q = synth.bits(w.q).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if append:
        idx = w.pos[:w.n_live].to(torch.int64)
        k_new = synth.bits(w.k_hist)[idx].contiguous().to(DEV)
        v_new = synth.bits(w.v_hist)[idx].contiguous().to(DEV)
        va.kv_ring_append(k_new, v_new, w.n_live, k, v, pos_dev, dev_status=status)
    if n_splits == 0:
        if w.window > 0:
            n_splits = va.va_auto_splits(w.window + w.n_live - 1, w.window)
        else:
            lo, hi = oracle.read_extent(w.pos.numpy(), w.n_live, 0)
            n_splits = va.va_auto_splits(hi, 0)
    part_o = torch.full((n_splits, w.n_rows, 6, 128), float("nan"), dtype=torch.float32, device=DEV)
    part_lse = torch.full((n_splits, w.n_rows, 6), float("nan"), dtype=torch.float32, device=DEV)
    if w.window > 0:
        used = va.verify_attn_swa(q, w.n_live, k, v, w.window, pos_dev, w.scale, part_o, part_lse, n_splits,
                                  dev_status=status, variant=variant)
    else:
        used = va.verify_attn_full(q, w.n_live, k, v, pos_dev, w.scale, part_o, part_lse, n_splits,
                                   dev_status=status, variant=variant)
    assert used == n_splits
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), dtype=torch.float32, device=DEV)
    sink = w.sink.to(DEV)
    va.attn_split_combine(part_o, part_lse, n_splits, sink, w.n_live, out, out_lse, variant=variant)
    torch.cuda.synchronize()
    return dict(out=oracle.bf16_bits_to_f64(out.cpu().numpy()), out_bits=out.cpu().numpy().view(np.uint16),
                out_lse=out_lse.cpu().numpy().astype(np.float64), part_o=part_o.cpu().numpy().astype(np.float64),
                part_lse=part_lse.cpu().numpy().astype(np.float64), n_splits=n_splits,
                status=int(status.item()), k=k, v=v)


def expected(w: synth.Workload, n_splits: int, n_threads: int = 8):
    """Oracle values for the same seeded inputs (positions unshifted)."""
    res = oracle.verify_attn(_bits_np(w.q), _bits_np(w.k_hist), _bits_np(w.v_hist), w.pos.numpy(), w.n_live,
                             w.sink.numpy(), w.scale, w.window, n_splits=n_splits, n_threads=n_threads)
    res["out_bf16"] = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(res["out"]))
    return res


def run_step_fused(w: synth.Workload, n_splits: int = 0, placement: str = "all", wrap_offset: int = 0,
                   workspace=None, variant: str = ""):
    """The same call as run_step through verify_attn_step (append inside the attention launch, then the
    combine).  The partials are read back from the workspace."""
    pos_dev = (w.pos.to(torch.int64) + wrap_offset).to(torch.int32).to(DEV) if wrap_offset else w.pos.to(DEV)
    k, v = cache_state(w, int(w.pos[0]), placement, wrap_offset)
    q = synth.bits(w.q).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    idx = w.pos[:w.n_live].to(torch.int64)
    k_new = synth.bits(w.k_hist)[idx].contiguous().to(DEV)
    v_new = synth.bits(w.v_hist)[idx].contiguous().to(DEV)
    if n_splits == 0:
        if w.window > 0:
            n_splits = va.va_auto_splits(w.window + w.n_live - 1, w.window)
        else:
            n_splits = va.va_auto_splits(w.slots, 0)
    if workspace is None:
        workspace = torch.full((va.va_workspace_bytes(n_splits) // 4,), float("nan"), dtype=torch.float32,
                               device=DEV)
    out = torch.full((w.n_rows, 6, 128), 0x7FC0, dtype=torch.int16, device=DEV)
    out_lse = torch.full((w.n_rows, 6), float("nan"), dtype=torch.float32, device=DEV)
    used = va.verify_attn_step(q, k_new, v_new, w.n_live, k, v, pos_dev, w.scale, w.sink.to(DEV), workspace, out,
                               out_lse, window=w.window, n_splits=n_splits, dev_status=status, variant=variant)
    assert used == n_splits
    torch.cuda.synchronize()
    n_o = n_splits * 8 * 6 * 128       # part_lse starts after room for 8 rows per split
    part_o = workspace[:n_splits * w.n_rows * 6 * 128].view(n_splits, w.n_rows, 6, 128)
    part_lse = workspace[n_o:n_o + n_splits * w.n_rows * 6].view(n_splits, w.n_rows, 6)
    return dict(out=oracle.bf16_bits_to_f64(out.cpu().numpy()), out_bits=out.cpu().numpy().view(np.uint16),
                out_lse=out_lse.cpu().numpy().astype(np.float64), part_o=part_o.cpu().numpy().astype(np.float64),
                part_lse=part_lse.cpu().numpy().astype(np.float64), n_splits=n_splits,
                status=int(status.item()), k=k, v=v, workspace=workspace)
