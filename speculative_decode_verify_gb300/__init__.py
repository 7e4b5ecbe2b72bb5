"""GB300-native speculative-decoding verify attention.

Thin ctypes binding over the C ABI of ``libverify_attn.so`` (declared in
``include/verify_attn.h``): every function here only marshals torch tensors into pointers and
sizes and calls the entry point of the same name; all the work runs in the library's CUDA
kernels.  There is no CPU fallback: if the compiled library is missing, every call raises.

Source: IQuestRT technical report, sections "Read only the KV tiles needed by the current
positions" and "Expose more parallelism in attention".
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "VerifyAttnError", "lib", "lib_path", "kv_ring_append", "verify_attn_full", "verify_attn_swa",
    "attn_split_combine", "verify_attn_tree", "verify_attn_full_noalloc", "va_sample_workspace_bytes",
    "va_sample_topk_topp", "va_accept_chain", "va_tree_accept_settle", "kv_ring_append_q8", "verify_attn_q8",
    "verify_attn_q8_tree", "verify_attn_q8_step", "verify_attn_step", "va_selftest_bounded_wait", "SAMPLE_MAX_K", "SAMPLE_TILE",
    "SAMPLE_MAX_VOCAB", "NOALLOC_MAX_SPLITS", "va_workspace_bytes", "va_auto_splits", "va_auto_splits_for", "va_status_string",
    "HEAD_DIM", "Q_HEADS", "MAX_ROWS", "TILE", "MAX_SPLITS", "MAX_TREE_NODES", "EXPORTS",
    "VA_OK", "VA_INVALID_ARG", "VA_UNSUPPORTED", "VA_RING_TOO_SMALL", "VA_CUDA_ERROR",
]

HEAD_DIM, Q_HEADS, MAX_ROWS, TILE, MAX_SPLITS, MAX_TREE_NODES = 128, 6, 8, 64, 4096, 16
VA_OK, VA_INVALID_ARG, VA_UNSUPPORTED, VA_RING_TOO_SMALL, VA_CUDA_ERROR = 0, 1, 2, 3, 4
EXPORTS = ("kv_ring_append", "verify_attn_full", "verify_attn_swa", "verify_attn_tree", "attn_split_combine",
           "va_workspace_bytes", "va_auto_splits", "va_auto_splits_for", "va_status_string",
           "verify_attn_full_noalloc", "va_sample_workspace_bytes", "va_sample_topk_topp", "va_accept_chain",
           "va_tree_accept_settle", "kv_ring_append_q8", "verify_attn_q8", "verify_attn_q8_tree", "verify_attn_q8_step",
           "verify_attn_step", "va_selftest_bounded_wait")
NOALLOC_MAX_SPLITS = 160
SAMPLE_MAX_K, SAMPLE_TILE, SAMPLE_MAX_VOCAB = 32, 8192, 262144

_PKG = os.path.dirname(os.path.abspath(__file__))
_lib = {}
_lock = threading.Lock()


class VerifyAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {va_status_string(status)} ({status})")


def lib_path(variant: str = "") -> str:
    return os.path.join(_PKG, "_build", f"libverify_attn{variant}.so")


def lib(variant: str = "") -> ctypes.CDLL:
    """The loaded CUDA library (built by ``speculative_decode_verify_gb300.build``)."""
    with _lock:
        if variant in _lib:
            return _lib[variant]
        path = lib_path(variant)
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path}); run speculative_decode_verify_gb300.build.build()")
        L = ctypes.CDLL(path)
        p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.kv_ring_append.argtypes = [p, p, i, p, p, i, p, p, p]
        L.verify_attn_full.argtypes = [p, i, i, p, p, i, p, f, i, p, p, ctypes.POINTER(i), p, p]
        L.verify_attn_swa.argtypes = [p, i, i, p, p, i, i, p, f, i, p, p, ctypes.POINTER(i), p, p]
        L.verify_attn_tree.argtypes = [p, i, i, p, p, i, i, p, f, i, p, p, ctypes.POINTER(i), p, p]
        L.attn_split_combine.argtypes = [p, p, i, p, i, i, p, p, p]
        L.verify_attn_full_noalloc.argtypes = [p, i, i, p, p, i, p, f, i, p, p, p, ctypes.POINTER(i), p, p]
        for fn in ("kv_ring_append", "verify_attn_full", "verify_attn_swa", "verify_attn_tree",
                   "attn_split_combine", "verify_attn_full_noalloc"):
            getattr(L, fn).restype = i
        L.va_sample_workspace_bytes.argtypes = [i, i, i]
        L.va_sample_workspace_bytes.restype = ctypes.c_size_t
        L.va_sample_topk_topp.argtypes = [p, i, i, i, f, f, p, p, p, p, p, p, ctypes.c_size_t, p]
        L.va_accept_chain.argtypes = [p, p, p, p, p, p, i, p, p, i, p, p, p, p, p, p, p]
        L.va_tree_accept_settle.argtypes = [p, p, i, p, i, p, p, p, p, p, p, p, p]
        L.kv_ring_append_q8.argtypes = [p, p, i, p, p, p, p, i, p, p, p]
        L.verify_attn_q8.argtypes = [p, i, i, p, p, p, p, i, i, p, f, i, p, p, ctypes.POINTER(i), p, p]
        L.verify_attn_q8_tree.argtypes = [p, i, i, p, p, p, p, i, i, p, f, i, p, p, ctypes.POINTER(i), p, p]
        L.verify_attn_q8_step.argtypes = [p, p, p, i, i, p, p, p, p, i, i, p, p, f, i, p, p, p, ctypes.POINTER(i),
                                          p, p]
        for fn in ("va_sample_topk_topp", "va_accept_chain", "va_tree_accept_settle", "kv_ring_append_q8",
                   "verify_attn_q8", "verify_attn_q8_tree", "verify_attn_q8_step"):
            getattr(L, fn).restype = i
        L.verify_attn_step.argtypes = [p, p, p, i, i, p, p, i, i, p, p, f, i, p, p, p, ctypes.POINTER(i), p, p]
        L.verify_attn_step.restype = i
        L.va_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong, p, p, p]
        L.va_selftest_bounded_wait.restype = i
        L.va_workspace_bytes.argtypes = [i]
        L.va_workspace_bytes.restype = ctypes.c_size_t
        L.va_auto_splits.argtypes = [i, i]
        L.va_auto_splits.restype = i
        L.va_auto_splits_for.argtypes = [i, i, i]
        L.va_auto_splits_for.restype = i
        L.va_status_string.argtypes = [i]
        L.va_status_string.restype = ctypes.c_char_p
        _lib[variant] = L
        return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int) -> None:
    if status != VA_OK:
        raise VerifyAttnError(fn, status)


def va_status_string(status: int) -> str:
    return lib().va_status_string(int(status)).decode()


def va_workspace_bytes(n_splits: int) -> int:
    return int(lib().va_workspace_bytes(int(n_splits)))


def verify_attn_step(q, k_new, v_new, n_live: int, k_cache, v_cache, pos, scale: float, sink, workspace, out,
                     out_lse=None, window: int = 0, n_splits: int = 0, dev_status=None, stream=None,
                     variant: str = "") -> int:
    """One whole verify call (append + split attention + combine, two launches); returns the split count.
    workspace: float32 device tensor of at least va_workspace_bytes(n_splits) bytes (the partials)."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_step(_ptr(q), _ptr(k_new), _ptr(v_new), int(q.shape[0]), int(n_live),
                                       _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[0]), int(window), _ptr(pos),
                                       _ptr(sink), float(scale), int(n_splits), _ptr(workspace), _ptr(out),
                                       _ptr(out_lse), ctypes.byref(used), _ptr(dev_status), _stream(stream))
    _check("verify_attn_step", st)
    return used.value


def va_auto_splits(extent_hint: int, window: int = 0) -> int:
    return int(lib().va_auto_splits(int(extent_hint), int(window)))


def va_auto_splits_for(extent_hint: int, window: int, sm_count: int) -> int:
    return int(lib().va_auto_splits_for(int(extent_hint), int(window), int(sm_count)))


def kv_ring_append(k_new, v_new, n_live: int, k_cache, v_cache, pos, dev_status=None, stream=None,
                   variant: str = "") -> None:
    """Write the live rows' K/V ([n_live,128] bf16) to slot pos[r] mod slots of the cache."""
    st = lib(variant).kv_ring_append(_ptr(k_new), _ptr(v_new), int(n_live), _ptr(k_cache), _ptr(v_cache),
                                     int(k_cache.shape[0]), _ptr(pos), _ptr(dev_status), _stream(stream))
    _check("kv_ring_append", st)


def verify_attn_full(q, n_live: int, k_cache, v_cache, pos, scale: float, part_o, part_lse,
                     n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Split-KV attention of a full-attention layer; returns the split count launched."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_full(_ptr(q), int(q.shape[0]), int(n_live), _ptr(k_cache), _ptr(v_cache),
                                       int(k_cache.shape[0]), _ptr(pos), float(scale), int(n_splits),
                                       _ptr(part_o), _ptr(part_lse), ctypes.byref(used), _ptr(dev_status),
                                       _stream(stream))
    _check("verify_attn_full", st)
    return used.value


def verify_attn_swa(q, n_live: int, k_ring, v_ring, window: int, pos, scale: float, part_o, part_lse,
                    n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Split-KV attention of a sliding-window layer read from its ring; returns the split count."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_swa(_ptr(q), int(q.shape[0]), int(n_live), _ptr(k_ring), _ptr(v_ring),
                                      int(k_ring.shape[0]), int(window), _ptr(pos), float(scale), int(n_splits),
                                      _ptr(part_o), _ptr(part_lse), ctypes.byref(used), _ptr(dev_status),
                                      _stream(stream))
    _check("verify_attn_swa", st)
    return used.value


def verify_attn_tree(q, n_nodes: int, k_cache, v_cache, tree, scale: float, part_o, part_lse, window: int = 0,
                     n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Split-KV attention of a draft tree (``tree`` = device int32 [1 + n_nodes]: base, then each node's
    ancestor-or-self mask) over a full cache (window 0) or a ring; returns the split count."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_tree(_ptr(q), int(q.shape[0]), int(n_nodes), _ptr(k_cache), _ptr(v_cache),
                                       int(k_cache.shape[0]), int(window), _ptr(tree), float(scale), int(n_splits),
                                       _ptr(part_o), _ptr(part_lse), ctypes.byref(used), _ptr(dev_status),
                                       _stream(stream))
    _check("verify_attn_tree", st)
    return used.value


def attn_split_combine(part_o, part_lse, n_splits: int, sink, n_live: int, out, out_lse=None, stream=None,
                       variant: str = "") -> None:
    """Log-sum-exp merge of the partials with the sink; writes bf16 ``out`` [n_rows,6,128]."""
    st = lib(variant).attn_split_combine(_ptr(part_o), _ptr(part_lse), int(n_splits), _ptr(sink),
                                         int(out.shape[0]), int(n_live), _ptr(out), _ptr(out_lse),
                                         _stream(stream))
    _check("attn_split_combine", st)


def verify_attn_full_noalloc(q, n_live: int, k_cache, v_cache, pos, scale: float, sink, out, out_lse=None,
                             n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Full-attention verify call plus combine with the partials in the library's own fixed device
    buffer (for callers that cannot allocate); returns the split count launched."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_full_noalloc(_ptr(q), int(q.shape[0]), int(n_live), _ptr(k_cache), _ptr(v_cache),
                                               int(k_cache.shape[0]), _ptr(pos), float(scale), int(n_splits),
                                               _ptr(sink), _ptr(out), _ptr(out_lse), ctypes.byref(used),
                                               _ptr(dev_status), _stream(stream))
    _check("verify_attn_full_noalloc", st)
    return used.value


# ----------------------------------------------------------------------------- after verification
def va_sample_workspace_bytes(n_rows: int, vocab: int, top_k: int) -> int:
    return int(lib().va_sample_workspace_bytes(int(n_rows), int(vocab), int(top_k)))


def va_sample_topk_topp(logits, top_k: int, top_p: float, temperature: float, u, ids, probs, counts, tokens,
                        workspace, stream=None, variant: str = "") -> None:
    """Top-k / temperature / top-p sampling of logits [n_rows, vocab] (float32, device); writes ids/probs
    [n_rows, top_k], counts and tokens [n_rows].  ``workspace``: a device byte tensor of at least
    va_sample_workspace_bytes(n_rows, vocab, top_k) bytes."""
    n_rows, vocab = int(logits.shape[0]), int(logits.shape[1])
    st = lib(variant).va_sample_topk_topp(_ptr(logits), n_rows, vocab, int(top_k), float(top_p), float(temperature),
                                          _ptr(u), _ptr(ids), _ptr(probs), _ptr(counts), _ptr(tokens), _ptr(workspace),
                                          int(workspace.numel() * workspace.element_size()), _stream(stream))
    _check("va_sample_topk_topp", st)


def va_accept_chain(p_ids, p_probs, p_counts, q_ids, q_probs, q_counts, drafts, target_tokens, n_drafts: int,
                    u_accept, u_replace, pos, n_accepted, out_tokens, next_pos=None, stream=None,
                    variant: str = "") -> None:
    """Rejection-sampling acceptance of a chain of n_drafts drafts (all tensors on the device)."""
    st = lib(variant).va_accept_chain(_ptr(p_ids), _ptr(p_probs), _ptr(p_counts), _ptr(q_ids), _ptr(q_probs),
                                      _ptr(q_counts), int(p_ids.shape[1]), _ptr(drafts), _ptr(target_tokens),
                                      int(n_drafts), _ptr(u_accept), _ptr(u_replace), _ptr(pos), _ptr(n_accepted),
                                      _ptr(out_tokens), _ptr(next_pos), _stream(stream))
    _check("va_accept_chain", st)


def va_tree_accept_settle(k_cache, v_cache, tree, n_nodes: int, node_tokens, target_tokens, path, emitted,
                          n_accepted, next_pos=None, dev_status=None, stream=None, variant: str = "") -> None:
    """Accept a draft tree's path and move its K/V to consecutive positions (k/v_cache may be None)."""
    slots = int(k_cache.shape[0]) if k_cache is not None else 0
    st = lib(variant).va_tree_accept_settle(_ptr(k_cache), _ptr(v_cache), slots, _ptr(tree), int(n_nodes),
                                            _ptr(node_tokens), _ptr(target_tokens), _ptr(path), _ptr(emitted),
                                            _ptr(n_accepted), _ptr(next_pos), _ptr(dev_status), _stream(stream))
    _check("va_tree_accept_settle", st)


# ----------------------------------------------------------------------------- quantised K/V cache
def kv_ring_append_q8(k_new, v_new, n_live: int, k_codes, v_codes, k_scale, v_scale, pos, dev_status=None,
                      stream=None, variant: str = "") -> None:
    """Encode the live rows' K/V ([n_live,128] bf16) into the quantised cache at slot pos[r] mod slots."""
    st = lib(variant).kv_ring_append_q8(_ptr(k_new), _ptr(v_new), int(n_live), _ptr(k_codes), _ptr(v_codes),
                                        _ptr(k_scale), _ptr(v_scale), int(k_codes.shape[0]), _ptr(pos),
                                        _ptr(dev_status), _stream(stream))
    _check("kv_ring_append_q8", st)


def verify_attn_q8(q, n_live: int, k_codes, v_codes, k_scale, v_scale, pos, scale: float, part_o, part_lse,
                   window: int = 0, n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Split-KV verify attention over the quantised cache (window 0: full attention); returns the split count."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_q8(_ptr(q), int(q.shape[0]), int(n_live), _ptr(k_codes), _ptr(v_codes),
                                     _ptr(k_scale), _ptr(v_scale), int(k_codes.shape[0]), int(window), _ptr(pos),
                                     float(scale), int(n_splits), _ptr(part_o), _ptr(part_lse), ctypes.byref(used),
                                     _ptr(dev_status), _stream(stream))
    _check("verify_attn_q8", st)
    return used.value


def verify_attn_q8_tree(q, n_nodes: int, k_codes, v_codes, k_scale, v_scale, tree, scale: float, part_o, part_lse,
                        window: int = 0, n_splits: int = 0, dev_status=None, stream=None, variant: str = "") -> int:
    """Tree verify attention over the quantised cache (``tree`` = [base, masks...] int32 on the device, as for
    verify_attn_tree); returns the split count."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_q8_tree(_ptr(q), int(q.shape[0]), int(n_nodes), _ptr(k_codes), _ptr(v_codes),
                                          _ptr(k_scale), _ptr(v_scale), int(k_codes.shape[0]), int(window),
                                          _ptr(tree), float(scale), int(n_splits), _ptr(part_o), _ptr(part_lse),
                                          ctypes.byref(used), _ptr(dev_status), _stream(stream))
    _check("verify_attn_q8_tree", st)
    return used.value


def verify_attn_q8_step(q, k_new, v_new, n_live: int, k_codes, v_codes, k_scale, v_scale, pos, scale: float, sink,
                        workspace, out, out_lse=None, window: int = 0, n_splits: int = 0, dev_status=None,
                        stream=None, variant: str = "") -> int:
    """A whole verify call over the quantised cache (encoding append inside the attention launch, then the
    combine); returns the split count."""
    used = ctypes.c_int(0)
    st = lib(variant).verify_attn_q8_step(_ptr(q), _ptr(k_new), _ptr(v_new), int(q.shape[0]), int(n_live),
                                          _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                          int(k_codes.shape[0]), int(window), _ptr(pos), _ptr(sink), float(scale),
                                          int(n_splits), _ptr(workspace), _ptr(out), _ptr(out_lse),
                                          ctypes.byref(used), _ptr(dev_status), _stream(stream))
    _check("verify_attn_q8_step", st)
    return used.value


# ----------------------------------------------------------------------------- self-test
def va_selftest_bounded_wait(limit_ns: int, abort_after_ns: int = 0, dev_status=None, elapsed_ns=None, stream=None,
                             variant: str = "") -> None:
    """Run the kernels' bounded wait on a barrier nothing completes (see include/verify_attn.h)."""
    st = lib(variant).va_selftest_bounded_wait(int(limit_ns), int(abort_after_ns), _ptr(dev_status),
                                               _ptr(elapsed_ns), _stream(stream))
    _check("va_selftest_bounded_wait", st)
