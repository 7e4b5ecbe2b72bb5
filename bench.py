#!/usr/bin/env python3
"""Throughput of the verify-attention step on GB300.

Workload (one step): a full-attention layer at 196,608 positions (about 100.7 MB of bf16 K/V),
one KV head serving six query heads, head_dim 128, eight verify rows with n_live swept 4..8 - one
call per n_live, each call = kv_ring_append + verify_attn_full (split-KV over every SM) +
attn_split_combine.  Each n_live has its own cache (seeds 8..12), so five distinct 100.7 MB caches
rotate and every call reads K/V that is not in the 126 MB L2.

Reported (one JSON line on rank 0):
  value      algorithmic GB/s of the whole step with inputs resident in HBM, timed with CUDA events
             around K replays of a CUDA graph of the step (15 kernels)
  roofline   the split-attention kernel alone: its algorithmic bytes (K/V extent + Q) over its mean
             CUDA-event duration, against the measured HBM copy bandwidth
  e2e        the same metric through the C ABI with host buffers: per call the H2D copy of q, the new
             K/V rows and the positions from pinned memory and the D2H copy of the output, inside the
             timed region, one wait per step (the host polls the stream)
  cpu_baseline  the FP64 oracle on the host cores (rank 0, N = 1 only)
``--impl reference`` times the oracle itself as the reference arm (bounded sample per step).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-attn µs/call and achieved HBM GB/s vs GB300 peak, 1K–192K ctx, 1 GPU"
CTX = 196608
CAPACITY = 196672
N_LIVES = (4, 5, 6, 7, 8)
Q_BYTES = 8 * 6 * 128 * 2
OUT_BYTES = 8 * 6 * 128 * 2


def call_bytes(hi: int, n_live: int) -> int:
    """Algorithmic bytes of one call: the K/V extent, q, the output, the new rows (read + written)."""
    return 512 * hi + Q_BYTES + OUT_BYTES + 2 * 512 * n_live + 6 * 4


def attn_kernel_bytes(hi: int) -> int:
    """Algorithmic bytes of one split-attention launch: the K/V extent it must read, and q."""
    return 512 * hi + Q_BYTES


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the 1K-192K context sweep")
    ap.add_argument("--no-tree", action="store_true",
                    help="skip the draft-tree, sampling, acceptance and settlement measurements")
    ap.add_argument("--splits", type=int, default=0, help="split count (0 = library policy)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="profiling aid: only the split-attention launches, over --caches rotating caches")
    ap.add_argument("--tree-kernel-only", action="store_true",
                    help="profiling aid: only verify_attn_tree launches (16-node tree, 192K), over 2 caches")
    ap.add_argument("--sample-kernel-only", action="store_true",
                    help="profiling aid: only top-k/top-p sampling launches (8 x 160,000 logits), 2 buffers")
    ap.add_argument("--q8-kernel-only", action="store_true",
                    help="profiling aid: only verify_attn_q8 launches (quantised 192K cache), over 2 caches")
    ap.add_argument("--q8-tree-kernel-only", action="store_true",
                    help="profiling aid: only verify_attn_q8_tree launches (16-node tree, quantised 192K cache), "
                         "over 2 caches")
    ap.add_argument("--caches", type=int, default=5, help="distinct 192K caches to rotate (1..5)")
    ap.add_argument("--variant", default="", help="library build variant to load (A/B tuning aid)")
    ap.add_argument("--ctx", type=int, default=CTX, help="context of the --kernel-only runs")
    ap.add_argument("--ab", nargs=2, metavar=("A", "B"), default=None,
                    help="A/B comparison of two library builds on one GPU, alternated in ABBA BAAB order: each "
                         "argument is a comma-separated list of NAME=VALUE compile definitions ('' = the default "
                         "build); prints one JSON line with each build's per-block times and their spread")
    ap.add_argument("--ab-what", choices=["call", "kernel", "q8call", "q8", "tree", "treecall", "sample"],
                    default="call",
                    help="A/B unit: a whole verify call (verify_attn_step, graph-replayed), the split-attention "
                         "launch alone (verify_attn_full, back to back), or the same two over the quantised cache "
                         "(verify_attn_q8_step / verify_attn_q8), a 16-node tree verify launch (verify_attn_tree) "
                         "or a whole tree call (the nodes' append, verify_attn_tree and the combine, graph-replayed)")
    ap.add_argument("--ab-ctx", type=int, default=CTX, help="A/B workload context (positions)")
    ap.add_argument("--ab-window", type=int, default=0, help="A/B workload window (0 = full attention)")
    ap.add_argument("--ab-blocks", type=int, default=16, help="A/B timed blocks per build (a multiple of 4)")
    ap.add_argument("--ab-reps", type=int, default=40, help="graph replays (or launch rounds) per A/B block")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed control
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(per_rank_units: float, per_rank_seconds: float, dist: Dist):
    """Whole-job throughput: all ranks' units over the slowest rank's time (weak scaling)."""
    t = dist.max(per_rank_seconds)
    return per_rank_units * dist.world / t, t


# ----------------------------------------------------------------------------- clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for r in csv.reader(io.StringIO(open(self.path).read())):
            if len(r) < 9:
                continue
            try:
                rows.append(dict(sm=float(r[1]), max=float(r[2]), power=float(r[3]),
                                 hw=r[5].strip(), hwt=r[6].strip(), swt=r[7].strip(), cap=r[8].strip()))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        busy = [x for x in rows if x["power"] > 0.3 * max(y["power"] for y in rows)] or rows
        reasons = set()
        for x in busy:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("cap", "sw_power_cap")):
                if x[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x["sm"] for x in busy), "sm_max_mhz": max(x["max"] for x in rows),
                "reasons": sorted(reasons), "samples": len(busy)}


KERNEL_SOURCES = ("speculative_decode_verify_gb300/csrc/attn_tc.cu", "speculative_decode_verify_gb300/csrc/tc_ptx.cuh",
                  "speculative_decode_verify_gb300/csrc/va_internal.cuh")


def measured_traffic():
    """DRAM bytes per split-attention launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    import hashlib
    import re
    try:
        txt = open(os.path.join(ROOT, "profiles", "attn_tc_192k.md")).read()
        vals = dict(re.findall(r"^(traffic_bytes_per_launch|kernel_source_sha256)=(\S+)$", txt, re.M))
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        if vals.get("kernel_source_sha256") == h.hexdigest():
            return int(vals["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal (the measured copy bandwidth is the primary denominator)


def cudart():
    """The CUDA toolkit's runtime library (for plain cudaMemcpyAsync / cudaStreamSynchronize calls)."""
    import ctypes
    import glob
    names = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcudart.so")]
    names += sorted(glob.glob("/usr/local/cuda*/lib64/libcudart.so*")) + ["libcudart.so"]
    for n in names:
        try:
            rt = ctypes.CDLL(n)
            break
        except OSError:
            continue
    else:
        raise RuntimeError("libcudart not found")
    rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    rt.cudaMemcpyAsync.restype = ctypes.c_int
    rt.cudaStreamSynchronize.argtypes = [ctypes.c_void_p]
    rt.cudaStreamSynchronize.restype = ctypes.c_int
    rt.cudaStreamQuery.argtypes = [ctypes.c_void_p]
    rt.cudaStreamQuery.restype = ctypes.c_int
    return rt


def stream_poll(rt, stream) -> int:
    """Wait for everything queued on `stream` by polling it (a busy wait, as a latency-bound serving loop
    waits): 0 when done, else the CUDA error."""
    while True:
        r = rt.cudaStreamQuery(stream)
        if r != 600:   # cudaErrorNotReady
            return r


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# ----------------------------------------------------------------------------- oracle timing
def oracle_step_time(w, n_threads: int, min_seconds: float, max_reps: int = 1000):
    import oracle
    from speculative_decode_verify_gb300 import synth
    qb, kb, vb = synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(), synth.bits(w.v_hist).numpy()
    oracle.verify_attn(qb, kb[:64], vb[:64], [0] * w.n_rows, 1, w.sink.numpy(), w.scale, 0, n_threads=1)
    reps, t0 = 0, time.perf_counter()
    while True:
        res = oracle.verify_attn(qb, kb, vb, w.pos.numpy(), w.n_live, w.sink.numpy(), w.scale, 0, n_threads=n_threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            oracle_step_time.last = res
            return el / reps, reps


def cpu_baseline(w_full):
    """The oracle on all host cores (the reported value) and on one thread (for scale)."""
    cores = os.cpu_count() or 1
    per_call, reps = oracle_step_time(w_full, cores, 10.0)
    per_call_1, reps_1 = oracle_step_time(w_full, 1, 4.0, 3)
    hi = int(w_full.pos[w_full.n_live - 1]) + 1
    nbytes = call_bytes(hi, w_full.n_live)
    return {"value": nbytes / per_call / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} full calls of the 196,608-position, n_live={w_full.n_live} workload "
                      f"(all 48 row-head pairs, FP64), {cores} threads, {per_call * 1e3:.1f} ms/call",
            "single_thread": {"value": nbytes / per_call_1 / 1e9, "unit": "GB/s", "calls": reps_1,
                              "ms_per_call": per_call_1 * 1e3}}


def parity_fields(out_bits, out_lse, ref, n_live: int):
    """The GPU call's output against the oracle's for the same inputs: max |out - ref| with ref rounded once
    to bf16, max |out - exact| against the unrounded FP64 result, relative RMS, output LSE error."""
    import numpy as np

    import oracle
    exact = np.asarray(ref["out"], dtype=np.float64)[:n_live]
    got = oracle.bf16_bits_to_f64(np.asarray(out_bits))[:n_live]
    rounded = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(exact))
    a = np.abs(got - exact)
    step = np.exp2(np.floor(np.log2(np.maximum(np.maximum(np.abs(exact), np.abs(got)), 2.0 ** -126))) - 7)
    return {"call": f"196,608 positions, n_live={n_live}", "max_abs": float(np.abs(got - rounded).max()),
            "max_abs_exact": float(a.max()), "exact_bar_ok": bool(np.all(a <= 1e-2 + 0.5 * step)),
            "rel_rms": float(np.linalg.norm(got - rounded) / np.linalg.norm(rounded)),
            "lse_max_abs": float(np.abs(np.asarray(out_lse, dtype=np.float64)[:n_live] -
                                        np.asarray(ref["lse"], dtype=np.float64)[:n_live]).max()),
            "bars": "max_abs <= 1e-2 (one bf16 step where wider), |out - exact| <= 1e-2 + half a step, "
                    "rel_rms <= 2e-3, lse <= 1e-3"}


def workload_config():
    """The workload both arms report (the GPU arm adds how it ran it)."""
    return {"workload": "full-attention verify, 196,608 positions (100.7 MB bf16 K/V), 1 KV head / 6 q heads, d 128, "
                        "8 rows with n_live 4,5,6,7,8 (one call each per step)",
            "calls_per_step": len(N_LIVES), "capacity": CAPACITY}


def reference_arm(args, dist: Dist):
    """The oracle as the reference arm, on the same workload as the GPU arm: per step the five 196,608-position
    calls (n_live 4..8), each the plain FP64 definition over all 48 row-head pairs on every host core."""
    if dist.rank != 0:
        return
    import oracle
    from speculative_decode_verify_gb300 import synth
    cores = os.cpu_count() or 1
    calls = []
    for n in N_LIVES:
        w = synth.full_192k(n)
        calls.append((synth.bits(w.q).numpy(), synth.bits(w.k_hist).numpy(), synth.bits(w.v_hist).numpy(),
                      w.pos.numpy(), n, w.sink.numpy(), w.scale))
    oracle.verify_attn(calls[0][0], calls[0][1][:64], calls[0][2][:64], [0] * 8, 1, calls[0][5], calls[0][6], 0,
                       n_threads=1)

    def step():
        for qb, kb, vb, pos, n, sink, scale in calls:
            oracle.verify_attn(qb, kb, vb, pos, n, sink, scale, 0, n_threads=cores)

    for _ in range(max(args.warmup, 1)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    total = time.perf_counter() - t0
    bytes_step = sum(call_bytes(CTX, n) for n in N_LIVES)
    value = bytes_step * args.steps / total / 1e9
    sample = (f"per step the five verify calls of the GPU arm's workload (196,608 positions, n_live 4..8, 8 rows x 6 "
              f"heads, FP64 oracle), {cores} threads, {total / args.steps / len(N_LIVES) * 1e3:.1f} ms per call")
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
                      "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                      "data": "synthetic",
                      "config": dict(workload_config(), timing="wall clock on the host cores over the same five "
                                                               "calls per step as the GPU arm"),
                      "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle", "cores": cores,
                                       "sample": sample},
                      "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ----------------------------------------------------------------------------- GPU arm
def ours(args, dist: Dist):
    import ctypes

    import torch

    import speculative_decode_verify_gb300 as va
    from speculative_decode_verify_gb300 import build as vbuild
    from speculative_decode_verify_gb300 import synth

    vbuild.build()
    L = va.lib(args.variant)
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    stream = torch.cuda.Stream(dev)
    if args.tree_kernel_only or args.sample_kernel_only:
        return profiling_loop(args, L, dev, stream)
    S = args.splits or va.va_auto_splits(CTX, 0)

    calls = []
    w8 = None
    n_lives = N_LIVES[len(N_LIVES) - max(1, min(args.caches, len(N_LIVES))):]
    ctx = args.ctx if args.kernel_only else CTX
    cap = ctx + 64
    if args.kernel_only and not args.splits:
        S = va.va_auto_splits(ctx, 0)
    # Per-call inputs (q, the live rows' K and V, positions) and outputs (out, out_lse) live in one input
    # and one output block, on the device and in pinned host memory alike, so that the end-to-end loop
    # moves a step's inputs with one host->device copy and its results with one device->host copy.
    in_sizes = [(8 * 6 * 128 * 2, 8 * 128 * 2, 8 * 128 * 2, 8 * 4)] * len(n_lives)
    seg = lambda b: -(-b // 256) * 256
    in_bytes = sum(seg(x) for sz in in_sizes for x in sz)
    out_bytes = len(n_lives) * (seg(8 * 6 * 128 * 2) + seg(8 * 6 * 4))
    in_d = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    in_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    out_d = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    out_h = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    off_in, off_out = 0, 0

    def carve(buf, off, nbytes, dtype, shape):
        return buf[off:off + nbytes].view(dtype).view(shape)

    for n in n_lives:
        w = synth.full_192k(n) if ctx == CTX else synth.make(f"ctx{ctx}", 4 + n, ctx=ctx, n_live=n, slots=cap)
        if n == 8:
            w8 = w
        k = torch.full((cap, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
        v = torch.full((cap, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
        k[:ctx] = synth.bits(w.k_hist).to(dev)
        v[:ctx] = synth.bits(w.v_hist).to(dev)
        idx = w.pos[:n].to(torch.int64)
        c = dict(n=n, k=k, v=v, hi=int(w.pos[n - 1]) + 1)
        for name, nb, dt, shape, val in (("q", 8 * 6 * 128 * 2, torch.int16, (8, 6, 128), synth.bits(w.q)),
                                         ("kn", n * 256, torch.int16, (n, 128), synth.bits(w.k_hist)[idx]),
                                         ("vn", n * 256, torch.int16, (n, 128), synth.bits(w.v_hist)[idx]),
                                         ("pos", 8 * 4, torch.int32, (8,), w.pos)):
            c[name + "_h"] = carve(in_h, off_in, nb, dt, shape)
            c[name + "_h"].copy_(val)
            c[name] = carve(in_d, off_in, nb, dt, shape)
            off_in += seg(nb)
        for name, nb, dt, shape in (("out", 8 * 6 * 128 * 2, torch.int16, (8, 6, 128)),
                                    ("out_lse", 8 * 6 * 4, torch.float32, (8, 6))):
            c[name + "_h"] = carve(out_h, off_out, nb, dt, shape)
            c[name] = carve(out_d, off_out, nb, dt, shape)
            off_out += seg(nb)
        c["sink"] = w.sink.to(dev)
        c["scale"] = w.scale
        calls.append(c)
    in_d.copy_(in_h)
    # one workspace: part_o, then part_lse (the layout verify_attn_step expects)
    ws = torch.empty(va.va_workspace_bytes(S) // 4, dtype=torch.float32, device=dev)
    part_o = ws[:S * 8 * 6 * 128].view(S, 8, 6, 128)
    part_lse = ws[S * 8 * 6 * 128:].view(S, 8, 6)
    del w
    torch.cuda.synchronize(dev)

    sp = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p

    # each call's C-ABI arguments, marshalled once (a caller that repeats a call keeps its pointers)
    for c in calls:
        c["step_args"] = (P(c["q"].data_ptr()), P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), 8, c["n"],
                          P(c["k"].data_ptr()), P(c["v"].data_ptr()), CAPACITY, 0, P(c["pos"].data_ptr()),
                          P(c["sink"].data_ptr()), ctypes.c_float(c["scale"]), S, P(ws.data_ptr()),
                          P(c["out"].data_ptr()), P(c["out_lse"].data_ptr()), None, None, sp)
    step_fn = L.verify_attn_step

    def launch_call(c):
        # one verify call through verify_attn_step: the append inside the attention launch, then the combine
        st = step_fn(*c["step_args"])
        if st:
            raise RuntimeError(f"verify_attn_step failed with status {st}")

    def launch_call_separate(c, ev=None):
        # the same call as the three C-ABI calls (append, attention, combine); ev brackets the attention
        st = L.kv_ring_append(P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), c["n"], P(c["k"].data_ptr()),
                              P(c["v"].data_ptr()), CAPACITY, P(c["pos"].data_ptr()), None, sp)
        if ev is not None:
            ev[0].record(stream)
        st |= L.verify_attn_full(P(c["q"].data_ptr()), 8, c["n"], P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                 CAPACITY, P(c["pos"].data_ptr()), ctypes.c_float(c["scale"]), S,
                                 P(part_o.data_ptr()), P(part_lse.data_ptr()), None, None, sp)
        if ev is not None:
            ev[1].record(stream)
        st |= L.attn_split_combine(P(part_o.data_ptr()), P(part_lse.data_ptr()), S, P(c["sink"].data_ptr()), 8,
                                   c["n"], P(c["out"].data_ptr()), P(c["out_lse"].data_ptr()), sp)
        if st:
            raise RuntimeError(f"verify call failed with status {st}")

    def step():
        for c in calls:
            launch_call(c)

    def sweep_points(ctx, window, reps=100, per_graph=8):
        """us per call and algorithmic GB/s of one verify call (verify_attn_step with the library's split
        choice) at this context for n_live 4..8; two caches alternate so K/V are read cold when they exceed
        L2.  One CUDA graph holds 2 x per_graph calls, as consecutive layers of a decode step would: a graph
        of only two calls adds the device's per-graph launch gap (~3 us) to every other call.  The caches
        hold the whole history, so every n_live uses the same ones (the append rewrites the live rows with
        their own values)."""
        ws = []
        for rep in range(2):
            w = synth.make(f"sweep{ctx}", 900 + rep, ctx=ctx, n_live=8, window=window,
                           slots=(synth.RING_SLOTS if window else ctx + 64))
            slots = w.slots
            k = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
            v = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
            kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
            first = max(0, ctx - slots) if window else 0
            pp = torch.arange(first, ctx)
            k[pp % slots] = kb[first:ctx]
            v[pp % slots] = vb[first:ctx]
            ws.append(dict(w=w, k=k.to(dev), v=v.to(dev), kb=kb, vb=vb, q=synth.bits(w.q).to(dev),
                           sink=w.sink.to(dev), out=torch.empty(8, 6, 128, dtype=torch.int16, device=dev)))
        hbm = (measured_peaks() or {}).get("hbm_gbs", 6800.0)
        points = []
        for n in N_LIVES:
            for c in ws:
                pos = synth.tail_positions(ctx, n)
                idx = pos[:n].to(torch.int64)
                c["pos"] = pos.to(dev)
                c["kn"], c["vn"] = c["kb"][idx].contiguous().to(dev), c["vb"][idx].contiguous().to(dev)
            Ss = va.va_auto_splits(window + n - 1 if window else ctx, window)
            wsp = torch.empty(va.va_workspace_bytes(Ss) // 4, dtype=torch.float32, device=dev)

            def one(c):
                w = c["w"]
                st = L.verify_attn_step(P(c["q"].data_ptr()), P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), 8, n,
                                        P(c["k"].data_ptr()), P(c["v"].data_ptr()), w.slots, window,
                                        P(c["pos"].data_ptr()), P(c["sink"].data_ptr()), ctypes.c_float(w.scale),
                                        Ss, P(wsp.data_ptr()), P(c["out"].data_ptr()), None, None, None, sp)
                if st:
                    raise RuntimeError(f"sweep call failed with status {st}")

            with torch.cuda.stream(stream):
                for _ in range(3):
                    for c in ws:
                        one(c)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for _ in range(per_graph):
                        for c in ws:
                            one(c)
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
                e1.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (reps * 2 * per_graph)
            hi = ctx
            lo = max(0, ctx - n - window + 1) if window else 0
            nbytes = 512 * (hi - lo) + Q_BYTES + OUT_BYTES + 2 * 512 * n + 24
            points.append({"ctx": ctx, "kind": "swa" if window else "full", "n_live": n, "splits": Ss,
                           "us_per_call": us, "gbs": nbytes / us / 1e3, "frac_of_hbm_peak": nbytes / us / 1e3 / hbm})
        return points

    def tree_short_measure(ctx_short=2048, reps=100, per_graph=8):
        """A 16-node best-first tree at a short context (nodes at ctx_short - 16 .. ctx_short - 1): per call
        (kv_ring_append of the nodes + verify_attn_tree + combine), 2 x per_graph calls in one CUDA graph as
        consecutive layers would run, two caches alternating.  Latency-bound; context for the pages'
        single-GPU verify figure, which is quoted at a short median context on other hardware."""
        cap = ctx_short + 64
        ts = []
        for i in range(2):
            w = synth.make_tree(f"bench_tree_short{i}", 540 + i, base=ctx_short - synth.TREE_NODES, slots=cap)
            k = torch.full((cap, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            v = torch.full((cap, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            k[:w.base] = synth.bits(w.k_hist)[:w.base].to(dev)
            v[:w.base] = synth.bits(w.v_hist)[:w.base].to(dev)
            ts.append(dict(w=w, k=k, v=v, q=synth.bits(w.q).to(dev), tree=w.tree.to(dev), pos=w.node_pos.to(dev),
                           kn=synth.bits(w.k_hist)[w.base:].contiguous().to(dev),
                           vn=synth.bits(w.v_hist)[w.base:].contiguous().to(dev), sink=w.sink.to(dev),
                           out=torch.empty(16, 6, 128, dtype=torch.int16, device=dev)))
        St = va.va_auto_splits_for(cap, 0, torch.cuda.get_device_properties(dev).multi_processor_count // 2)
        po = torch.empty(St, 16, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(St, 16, 6, dtype=torch.float32, device=dev)

        def one(c):
            w = c["w"]
            st = L.kv_ring_append(P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), w.n_nodes, P(c["k"].data_ptr()),
                                  P(c["v"].data_ptr()), cap, P(c["pos"].data_ptr()), None, sp)
            st |= L.verify_attn_tree(P(c["q"].data_ptr()), 16, w.n_nodes, P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                     cap, 0, P(c["tree"].data_ptr()), ctypes.c_float(w.scale), St, P(po.data_ptr()),
                                     P(pl.data_ptr()), None, None, sp)
            st |= L.attn_split_combine(P(po.data_ptr()), P(pl.data_ptr()), St, P(c["sink"].data_ptr()), 16, w.n_nodes,
                                       P(c["out"].data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"short tree call failed with status {st}")

        with torch.cuda.stream(stream):
            for _ in range(3):
                for c in ts:
                    one(c)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(per_graph):
                    for c in ts:
                        one(c)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * len(ts) * per_graph)
        return {"workload": f"16-node best-first draft tree, nodes at {ctx_short - 16:,}..{ctx_short - 1:,} of a "
                            f"{ctx_short:,}-position full-attention cache", "n_splits": St, "us_per_call": us}

    def tree_measure(reps=300):
        """A 16-node best-first draft tree at the 192K extent (nodes at 196,592..196,607): per call
        kv_ring_append of the 16 nodes + verify_attn_tree + attn_split_combine, graph-replayed over three
        rotating caches, and the tree kernel alone back to back."""
        ts = []
        for i in range(3):
            w = synth.make_tree(f"bench_tree{i}", 500 + i, base=CTX - synth.TREE_NODES, slots=CAPACITY)
            k = torch.full((CAPACITY, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            v = torch.full((CAPACITY, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            k[:w.base] = synth.bits(w.k_hist)[:w.base].to(dev)
            v[:w.base] = synth.bits(w.v_hist)[:w.base].to(dev)
            ts.append(dict(w=w, k=k, v=v, q=synth.bits(w.q).to(dev), tree=w.tree.to(dev), pos=w.node_pos.to(dev),
                           kn=synth.bits(w.k_hist)[w.base:].contiguous().to(dev),
                           vn=synth.bits(w.v_hist)[w.base:].contiguous().to(dev), sink=w.sink.to(dev),
                           out=torch.empty(16, 6, 128, dtype=torch.int16, device=dev)))
        groups = 2
        St = va.va_auto_splits_for(CAPACITY, 0, torch.cuda.get_device_properties(dev).multi_processor_count // groups)
        po = torch.empty(St, 16, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(St, 16, 6, dtype=torch.float32, device=dev)

        def attn(c):
            w = c["w"]
            return L.verify_attn_tree(P(c["q"].data_ptr()), 16, w.n_nodes, P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                      CAPACITY, 0, P(c["tree"].data_ptr()), ctypes.c_float(w.scale), St,
                                      P(po.data_ptr()), P(pl.data_ptr()), None, None, sp)

        def one(c):
            n = c["w"].n_nodes
            st = L.kv_ring_append(P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), n, P(c["k"].data_ptr()),
                                  P(c["v"].data_ptr()), CAPACITY, P(c["pos"].data_ptr()), None, sp)
            st |= attn(c)
            st |= L.attn_split_combine(P(po.data_ptr()), P(pl.data_ptr()), St, P(c["sink"].data_ptr()), 16, n,
                                       P(c["out"].data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"tree call failed with status {st}")

        with torch.cuda.stream(stream):
            for _ in range(3):
                for c in ts:
                    one(c)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in ts:
                    one(c)
            g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            us_call = e0.elapsed_time(e1) * 1e3 / (reps * len(ts))
            e0.record(stream)
            for _ in range(reps):
                for c in ts:
                    if attn(c):
                        raise RuntimeError("verify_attn_tree failed")
            e1.record(stream)
            e1.synchronize()
            us_attn = e0.elapsed_time(e1) * 1e3 / (reps * len(ts))
        kv = 512 * CTX
        call_b = kv + 2 * 16 * 6 * 128 * 2 + 2 * 512 * 16 + 17 * 4
        attn_b = kv + 16 * 6 * 128 * 2 + 17 * 4
        return {"workload": "16-node best-first draft tree, nodes at 196,592..196,607 of a 196,608-position "
                            "full-attention cache (100.7 MB K/V), 3 rotating caches",
                "n_splits": St, "groups": groups, "us_per_call": us_call, "gbs_call": call_b / us_call / 1e3,
                "attn_us_per_launch": us_attn, "attn_gbs": attn_b / us_attn / 1e3, "short": tree_short_measure()}

    def q8_caches(n_caches):
        """Quantised caches of the 192K workload, encoded on the GPU by kv_ring_append_q8 (one call each)."""
        out = []
        for i in range(n_caches):
            n = 8 - i
            w = synth.full_192k(n)
            kc = torch.full((CAPACITY, 128), 0x7F, dtype=torch.uint8, device=dev)
            vc = torch.zeros(CAPACITY, 128, dtype=torch.int8, device=dev)
            ks = torch.full((CAPACITY,), float("nan"), device=dev)
            vs = torch.full((CAPACITY,), float("nan"), device=dev)
            # the history, encoded by the library (the inputs stay referenced until the copy has run)
            kh, vh = synth.bits(w.k_hist).to(dev), synth.bits(w.v_hist).to(dev)
            hpos = torch.arange(CTX - n, dtype=torch.int32, device=dev)
            st = L.kv_ring_append_q8(P(kh.data_ptr()), P(vh.data_ptr()), CTX - n, P(kc.data_ptr()), P(vc.data_ptr()),
                                     P(ks.data_ptr()), P(vs.data_ptr()), CAPACITY, P(hpos.data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"kv_ring_append_q8 failed with status {st}")
            stream.synchronize()
            del kh, vh, hpos
            idx = w.pos[:n].to(torch.int64)
            out.append(dict(n=n, w=w, kc=kc, vc=vc, ks=ks, vs=vs, q=synth.bits(w.q).to(dev), pos=w.pos.to(dev),
                            kn=synth.bits(w.k_hist)[idx].contiguous().to(dev),
                            vn=synth.bits(w.v_hist)[idx].contiguous().to(dev), sink=w.sink.to(dev),
                            out=torch.empty(8, 6, 128, dtype=torch.int16, device=dev)))
        torch.cuda.synchronize(dev)
        return out

    def q8_measure(reps=300):
        """The quantised-cache verify at the 192K extent (FP8 keys, INT8 values, 264 B per position): the
        attention launch alone back to back, and the whole call (verify_attn_q8_step: the live rows coded by
        the attention launch, then the combine) graph-replayed, five calls per graph over five rotating caches
        with n_live 8..4 (5 x 52 MB > L2), as the bf16 call is measured."""
        qs = q8_caches(5)
        po = torch.empty(S, 8, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(S, 8, 6, dtype=torch.float32, device=dev)
        wsq = torch.empty(va.va_workspace_bytes(S) // 4, dtype=torch.float32, device=dev)

        def attn(c):
            return L.verify_attn_q8(P(c["q"].data_ptr()), 8, c["n"], P(c["kc"].data_ptr()), P(c["vc"].data_ptr()),
                                    P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), CAPACITY, 0, P(c["pos"].data_ptr()),
                                    ctypes.c_float(c["w"].scale), S, P(po.data_ptr()), P(pl.data_ptr()), None, None, sp)

        def one(c):
            st = L.verify_attn_q8_step(P(c["q"].data_ptr()), P(c["kn"].data_ptr()), P(c["vn"].data_ptr()), 8, c["n"],
                                       P(c["kc"].data_ptr()), P(c["vc"].data_ptr()), P(c["ks"].data_ptr()),
                                       P(c["vs"].data_ptr()), CAPACITY, 0, P(c["pos"].data_ptr()),
                                       P(c["sink"].data_ptr()), ctypes.c_float(c["w"].scale), S, P(wsq.data_ptr()),
                                       P(c["out"].data_ptr()), None, None, None, sp)
            if st:
                raise RuntimeError(f"quantised verify call failed with status {st}")

        with torch.cuda.stream(stream):
            for _ in range(3):
                for c in qs:
                    one(c)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                for c in qs:
                    if attn(c):
                        raise RuntimeError("verify_attn_q8 failed")
            e1.record(stream)
            e1.synchronize()
            us_attn = e0.elapsed_time(e1) * 1e3 / (reps * len(qs))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for c in qs:
                    one(c)
            g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            us_call = e0.elapsed_time(e1) * 1e3 / (reps * len(qs))
        hi = statistics.fmean(int(c["pos"][c["n"] - 1]) + 1 for c in qs)
        attn_b = 264 * hi + Q_BYTES
        peak = (measured_peaks() or {}).get("hbm_gbs", 6800.0)
        tree = q8_tree_measure(qs, reps)
        tree["attn_frac_of_hbm_peak"] = tree["attn_gbs"] / peak
        return {"workload": "quantised cache (E4M3 keys after a Hadamard rotation, INT8 values, fp32 row scales: "
                            "264 B per position), 196,608 positions (51.9 MB), 5 rotating caches, n_live 8..4",
                "n_splits": S, "attn_us_per_launch": us_attn, "attn_gbs": attn_b / us_attn / 1e3,
                "attn_frac_of_hbm_peak": attn_b / us_attn / 1e3 / peak, "us_per_call": us_call,
                "bytes_per_position": 264, "tree": tree}

    def q8_tree_measure(qs, reps):
        """A 16-node best-first draft tree over the same quantised caches, nodes at 196,592..196,607: the
        tree attention launch alone back to back, and the whole call (encoding append of the 16 nodes +
        verify_attn_q8_tree + combine) graph-replayed."""
        groups = 2
        St = va.va_auto_splits_for(CAPACITY, 0, torch.cuda.get_device_properties(dev).multi_processor_count // groups)
        po = torch.empty(St, 16, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(St, 16, 6, dtype=torch.float32, device=dev)
        ts = []
        for i, c in enumerate(qs):
            tw = synth.make_tree(f"bench_q8tree{i}", 520 + i, base=0, n_nodes=16)   # q, masks, nodes' K/V
            tree = tw.tree.clone()
            tree[0] = CTX - 16
            ts.append(dict(c=c, tw=tw, tree=tree.to(dev), q=synth.bits(tw.q).to(dev),
                           kn=synth.bits(tw.k_hist).contiguous().to(dev), vn=synth.bits(tw.v_hist).contiguous().to(dev),
                           pos=torch.arange(CTX - 16, CTX, dtype=torch.int32, device=dev), sink=tw.sink.to(dev),
                           out=torch.empty(16, 6, 128, dtype=torch.int16, device=dev)))

        def attn(t):
            c = t["c"]
            return L.verify_attn_q8_tree(P(t["q"].data_ptr()), 16, 16, P(c["kc"].data_ptr()), P(c["vc"].data_ptr()),
                                         P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), CAPACITY, 0,
                                         P(t["tree"].data_ptr()), ctypes.c_float(t["tw"].scale), St, P(po.data_ptr()),
                                         P(pl.data_ptr()), None, None, sp)

        def one(t):
            c = t["c"]
            st = L.kv_ring_append_q8(P(t["kn"].data_ptr()), P(t["vn"].data_ptr()), 16, P(c["kc"].data_ptr()),
                                     P(c["vc"].data_ptr()), P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), CAPACITY,
                                     P(t["pos"].data_ptr()), None, sp)
            st |= attn(t)
            st |= L.attn_split_combine(P(po.data_ptr()), P(pl.data_ptr()), St, P(t["sink"].data_ptr()), 16, 16,
                                       P(t["out"].data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"quantised tree call failed with status {st}")

        with torch.cuda.stream(stream):
            for _ in range(3):
                for t in ts:
                    one(t)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                for t in ts:
                    if attn(t):
                        raise RuntimeError("verify_attn_q8_tree failed")
            e1.record(stream)
            e1.synchronize()
            us_attn = e0.elapsed_time(e1) * 1e3 / (reps * len(ts))
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for t in ts:
                    one(t)
            g.replay()
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            e1.synchronize()
            us_call = e0.elapsed_time(e1) * 1e3 / (reps * len(ts))
        attn_b = 264 * CTX + 16 * 6 * 128 * 2 + 17 * 4
        return {"workload": "16-node best-first draft tree, nodes at 196,592..196,607 of the quantised 196,608-"
                            "position cache", "n_splits": St, "groups": groups, "attn_us_per_launch": us_attn,
                "attn_gbs": attn_b / us_attn / 1e3, "us_per_call": us_call}

    def post_verify_measure(reps=400):
        """The calls after verification, each graph-replayed: top-k 20 / top-p 0.95 sampling of 8 rows of
        160,000 logits (32 rotating logit buffers, 164 MB: read cold), rejection-sampling acceptance of 7
        drafts, and acceptance + settlement of a 16-node tree in the 192K cache."""
        res = {}
        n, vocab = 8, synth.VOCAB
        xs = [synth.logits(700 + i, n).to(dev) for i in range(32)]
        u = synth.uniforms(7, n).to(dev)
        ws = torch.zeros(va.va_sample_workspace_bytes(n, vocab, 20), dtype=torch.uint8, device=dev)
        ids = torch.empty(n, 20, dtype=torch.int32, device=dev)
        prb = torch.empty(n, 20, dtype=torch.float32, device=dev)
        cnt = torch.empty(n, dtype=torch.int32, device=dev)
        tok = torch.empty(n, dtype=torch.int32, device=dev)
        wsb = ws.numel()

        def sample(x):
            st = L.va_sample_topk_topp(P(x.data_ptr()), n, vocab, 20, ctypes.c_float(0.95), ctypes.c_float(1.0),
                                       P(u.data_ptr()), P(ids.data_ptr()), P(prb.data_ptr()), P(cnt.data_ptr()),
                                       P(tok.data_ptr()), P(ws.data_ptr()), wsb, sp)
            if st:
                raise RuntimeError(f"va_sample_topk_topp failed with status {st}")

        c = {k: v.to(dev) for k, v in synth.chain_round(11, 7).items()}
        na = torch.empty(1, dtype=torch.int32, device=dev)
        out = torch.empty(8, dtype=torch.int32, device=dev)
        nxt = torch.empty(1, dtype=torch.int32, device=dev)

        def accept():
            st = L.va_accept_chain(*[P(c[k].data_ptr()) for k in ("p_ids", "p_pr", "p_cnt", "q_ids", "q_pr", "q_cnt")],
                                   20, P(c["drafts"].data_ptr()), P(c["target"].data_ptr()), 7,
                                   P(c["u_accept"].data_ptr()), P(c["u_replace"].data_ptr()), P(c["pos"].data_ptr()),
                                   P(na.data_ptr()), P(out.data_ptr()), P(nxt.data_ptr()), sp)
            if st:
                raise RuntimeError(f"va_accept_chain failed with status {st}")

        parents, ttok, ttgt = synth.tree_round(12)
        tree = torch.cat([torch.tensor([CTX - 16], dtype=torch.int32), synth.ancestor_masks(parents)]).to(dev)
        tk, tt = ttok.to(dev), ttgt.to(dev)
        path = torch.empty(16, dtype=torch.int32, device=dev)
        em = torch.empty(16, dtype=torch.int32, device=dev)
        c0 = calls[0]

        def settle():
            st = L.va_tree_accept_settle(P(c0["k"].data_ptr()), P(c0["v"].data_ptr()), CAPACITY, P(tree.data_ptr()), 16,
                                         P(tk.data_ptr()), P(tt.data_ptr()), P(path.data_ptr()), P(em.data_ptr()),
                                         P(na.data_ptr()), P(nxt.data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"va_tree_accept_settle failed with status {st}")

        def graph_time(fns):
            with torch.cuda.stream(stream):
                for f in fns:
                    f()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for f in fns:
                        f()
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(max(1, reps // len(fns))):
                    g.replay()
                e1.record(stream)
                e1.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (max(1, reps // len(fns)) * len(fns))

        us = graph_time([lambda x=x: sample(x) for x in xs])
        nbytes = n * vocab * 4
        peak = (measured_peaks() or {}).get("hbm_gbs", 6800.0)
        res["sample_topk_topp"] = {"rows": n, "vocab": vocab, "top_k": 20, "top_p": 0.95, "us_per_call": us,
                                   "gbs": nbytes / us / 1e3, "frac_of_hbm_peak": nbytes / us / 1e3 / peak,
                                   "bound": "latency (5.1 MB per call)"}
        res["accept_chain"] = {"drafts": 7, "us_per_call": graph_time([accept] * 16)}
        res["tree_accept_settle"] = {"nodes": 16, "us_per_call": graph_time([settle] * 16)}
        return res

    if args.q8_kernel_only or args.q8_tree_kernel_only:
        # the quantised-cache split kernel alone (chain or 16-node tree), back to back over two caches (for
        # ncu captures)
        qs = q8_caches(2)
        tree_mode = args.q8_tree_kernel_only
        Sq = va.va_auto_splits_for(CAPACITY, 0, torch.cuda.get_device_properties(dev).multi_processor_count // 2) \
            if tree_mode else S
        rows = 16 if tree_mode else 8
        po = torch.empty(Sq, rows, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(Sq, rows, 6, dtype=torch.float32, device=dev)
        for i, c in enumerate(qs):
            tw = synth.make_tree(f"prof_q8tree{i}", 520 + i, base=0, n_nodes=16)
            tree = tw.tree.clone()
            tree[0] = CTX - 16
            c["tree"], c["tq"] = tree.to(dev), synth.bits(tw.q).to(dev)
        with torch.cuda.stream(stream):
            def attn_q8(c):
                if tree_mode:
                    st = L.verify_attn_q8_tree(P(c["tq"].data_ptr()), 16, 16, P(c["kc"].data_ptr()),
                                               P(c["vc"].data_ptr()), P(c["ks"].data_ptr()), P(c["vs"].data_ptr()),
                                               CAPACITY, 0, P(c["tree"].data_ptr()), ctypes.c_float(c["w"].scale), Sq,
                                               P(po.data_ptr()), P(pl.data_ptr()), None, None, sp)
                else:
                    st = L.verify_attn_q8(P(c["q"].data_ptr()), 8, c["n"], P(c["kc"].data_ptr()),
                                          P(c["vc"].data_ptr()), P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), CAPACITY,
                                          0, P(c["pos"].data_ptr()), ctypes.c_float(c["w"].scale), Sq,
                                          P(po.data_ptr()), P(pl.data_ptr()), None, None, sp)
                if st:
                    raise RuntimeError(f"quantised verify failed with status {st}")
            for _ in range(max(args.warmup, 1)):
                for c in qs:
                    attn_q8(c)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                for c in qs:
                    attn_q8(c)
            e1.record(stream)
            e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (args.steps * len(qs))
        print(json.dumps({"kernel_only": "verify_attn_q8_tree" if tree_mode else "verify_attn_q8",
                          "launches": args.steps * len(qs), "us_per_launch": us, "gbs": 264 * CTX / us / 1e3}))
        return

    if args.kernel_only:
        # the split-attention kernel alone, back to back over the rotating caches (for ncu captures)
        with torch.cuda.stream(stream):
            def attn(c):
                st = L.verify_attn_full(P(c["q"].data_ptr()), 8, c["n"], P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                        cap, P(c["pos"].data_ptr()), ctypes.c_float(c["scale"]), S,
                                        P(part_o.data_ptr()), P(part_lse.data_ptr()), None, None, sp)
                if st:
                    raise RuntimeError(f"verify_attn_full failed with status {st}")
            for _ in range(max(args.warmup, 1)):
                for c in calls:
                    attn(c)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                for c in calls:
                    attn(c)
            e1.record(stream)
            e1.synchronize()
        n = args.steps * len(calls)
        us = e0.elapsed_time(e1) * 1e3 / n
        print(json.dumps({"kernel_only": True, "variant": args.variant, "ctx": ctx, "launches": n,
                          "us_per_launch": us, "n_splits": S, "gbs": attn_kernel_bytes(ctx) / us / 1e3}))
        return

    clocks = Clocks(dist.local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
        stream.synchronize()
        # ---- value: K replays of a CUDA graph of the step (inputs resident in HBM)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(3):
            g.replay()
        stream.synchronize()
        dist.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize(dev)
        dist.barrier()
        t_graph = e0.elapsed_time(e1) / 1e3
        # ---- roofline: the split-attention kernel alone, launched back to back over the rotating caches
        # (as consecutive layers run); CUDA events on its stream bracket the region
        def attn_only(c):
            st = L.verify_attn_full(P(c["q"].data_ptr()), 8, c["n"], P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                    CAPACITY, P(c["pos"].data_ptr()), ctypes.c_float(c["scale"]), S,
                                    P(part_o.data_ptr()), P(part_lse.data_ptr()), None, None, sp)
            if st:
                raise RuntimeError(f"verify_attn_full failed with status {st}")
        kr = max(args.steps, 1)
        for c in calls:
            attn_only(c)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(kr):
            for c in calls:
                attn_only(c)
        r1.record(stream)
        r1.synchronize()
        attn_b2b = r0.elapsed_time(r1) / 1e3 / (kr * len(calls))
        # the same kernel timed alone inside the step (events around each launch; no overlap with the
        # previous kernel's tail)
        kb = min(args.steps, 400)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(kb * len(calls))]
        i = 0
        for _ in range(kb):
            for c in calls:
                torch.cuda._sleep(100_000)      # keeps the GPU behind the host: no launch gap in the pair
                launch_call_separate(c, evs[i])
                i += 1
        stream.synchronize()
        attn_s = [a.elapsed_time(b) / 1e3 for a, b in evs]
        # ---- e2e: host buffers, copies inside the timed region, one synchronisation per step: the step's
        # inputs (all five calls' q, live K/V rows and positions) go over in one pinned host->device copy,
        # the five calls run through verify_attn_step, their outputs come back in one device->host copy
        h2d = in_bytes
        d2h = out_bytes
        ke = args.steps
        dist.barrier()
        torch.cuda.synchronize(dev)
        # the copies through the CUDA runtime's cudaMemcpyAsync (as a C caller of the library would issue
        # them), the calls through the C ABI, one wait per step (the host polls the stream)
        rt = cudart()
        memcpy = rt.cudaMemcpyAsync
        def sync(s):
            return stream_poll(rt, s)
        h2d_args = (P(in_d.data_ptr()), P(in_h.data_ptr()), in_bytes, 1, sp)    # cudaMemcpyHostToDevice
        d2h_args = (P(out_h.data_ptr()), P(out_d.data_ptr()), out_bytes, 2, sp)  # cudaMemcpyDeviceToHost
        t0 = time.perf_counter()
        for _ in range(ke):
            if memcpy(*h2d_args):
                raise RuntimeError("cudaMemcpyAsync (inputs) failed")
            for c in calls:
                launch_call(c)
            if memcpy(*d2h_args) or sync(sp):
                raise RuntimeError("cudaMemcpyAsync (outputs) or the stream wait failed")
        t_e2e = time.perf_counter() - t0
        # the same end-to-end step as one CUDA graph (both copies and the five calls), replayed and
        # synchronised once per step: how a serving loop that captures its step would drive the library
        with torch.cuda.stream(stream):
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream):
                in_d.copy_(in_h, non_blocking=True)
                for c in calls:
                    launch_call(c)
                out_h.copy_(out_d, non_blocking=True)
            ge.replay()
            stream.synchronize()
            dist.barrier()
            t0 = time.perf_counter()
            for _ in range(ke):
                ge.replay()
                if sync(sp):
                    raise RuntimeError("end-to-end graph replay failed")
            t_e2e_graph = time.perf_counter() - t0
        dist.barrier()
    clk = clocks.stop()

    tree = None if args.no_tree else tree_measure()
    q8 = None if args.no_tree else q8_measure()
    post = None if args.no_tree else post_verify_measure()
    sweep = []
    if not args.no_sweep:
        for ctx_s in synth.SWEEP_CONTEXTS:
            for window in (0, synth.WINDOW):
                sweep.extend(sweep_points(ctx_s, window))
    step_bytes = sum(call_bytes(c["hi"], c["n"]) for c in calls)
    value, t_max = aggregate(step_bytes * args.steps / 1e9, t_graph, dist)
    e2e_value, _ = aggregate(step_bytes * ke / 1e9, t_e2e, dist)
    e2e_graph_value, _ = aggregate(step_bytes * ke / 1e9, t_e2e_graph, dist)
    mean_attn = attn_b2b
    isolated_attn = statistics.fmean(attn_s)
    attn_bytes = statistics.fmean(attn_kernel_bytes(c["hi"]) for c in calls)
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = attn_bytes / mean_attn / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(), **{"n_splits": S,
                   "l2": "5 distinct 100.7 MB caches rotate: each call reads K/V untouched for ~400 MB of "
                         "traffic, larger than L2 (no flush)",
                   "timing": "CUDA graph of the step replayed K times, CUDA events on its stream",
                   "parallelism": f"replicas x{dist.world} (one KV head per GPU, no collective)"}),
        "us_per_call": t_max / args.steps / len(calls) * 1e6,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": measured_traffic(), "kernel": "verify_attn_full split kernel",
                     "us_per_launch": mean_attn * 1e6, "launches": kr * len(calls),
                     "timing": "CUDA events around back-to-back launches over the 5 rotating caches",
                     "us_per_launch_isolated": isolated_attn * 1e6,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs" if peaks else "fallback 6.8 TB/s"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": t_e2e / ke * 1e6,
                "timing": "host wall clock: per step one H2D cudaMemcpyAsync, five verify_attn_step calls "
                          "through the C ABI, one D2H cudaMemcpyAsync, then the host polls the stream"},
        "e2e_graph": {"value": e2e_graph_value, "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "us_per_step": t_e2e_graph / ke * 1e6,
                      "timing": "host wall clock, one graph replay (copies + five calls) and one wait (stream "
                                "polled) per step"},
        "gpu_launches": 2 * len(calls) * args.steps,
        "sweep": [{k: (round(v, 2) if isinstance(v, float) else v) for k, v in p.items()} for p in sweep],
        "tree": tree,
        "quantised_cache": q8,
        "after_verify": post,
        "clocks": clk,
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w8)
        c8 = next(c for c in calls if c["n"] == 8)
        line["parity"] = parity_fields(c8["out"].cpu().numpy().view("uint16"), c8["out_lse"].cpu().numpy(),
                                       oracle_step_time.last, 8)
    if dist.rank == 0:
        print(json.dumps(line))


def profiling_loop(args, L, dev, stream):
    """Only one kind of launch, back to back (for ncu captures): the 16-node tree verify at 192K over two
    caches, or the top-k / top-p sampling of 8 x 160,000 logits over two buffers."""
    import ctypes

    import torch

    import speculative_decode_verify_gb300 as va
    from speculative_decode_verify_gb300 import synth

    P = ctypes.c_void_p
    sp = ctypes.c_void_p(stream.cuda_stream)
    fns = []
    if args.tree_kernel_only:
        groups = 2
        S = va.va_auto_splits_for(CAPACITY, 0, torch.cuda.get_device_properties(dev).multi_processor_count // groups)
        po = torch.empty(S, 16, 6, 128, dtype=torch.float32, device=dev)
        pl = torch.empty(S, 16, 6, dtype=torch.float32, device=dev)
        for i in range(2):
            w = synth.make_tree(f"prof_tree{i}", 500 + i, base=CTX - synth.TREE_NODES, slots=CAPACITY)
            k = torch.full((CAPACITY, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            v = torch.full((CAPACITY, 128), synth.BF16_NAN, dtype=torch.int16, device=dev)
            k[:w.ctx] = synth.bits(w.k_hist).to(dev)
            v[:w.ctx] = synth.bits(w.v_hist).to(dev)
            c = dict(q=synth.bits(w.q).to(dev), tree=w.tree.to(dev), k=k, v=v, scale=w.scale, n=w.n_nodes)
            fns.append(lambda c=c: L.verify_attn_tree(P(c["q"].data_ptr()), 16, c["n"], P(c["k"].data_ptr()),
                                                      P(c["v"].data_ptr()), CAPACITY, 0, P(c["tree"].data_ptr()),
                                                      ctypes.c_float(c["scale"]), S, P(po.data_ptr()),
                                                      P(pl.data_ptr()), None, None, sp))
        kind, nbytes = "verify_attn_tree", 512 * CTX
    else:
        n, vocab = 8, synth.VOCAB
        ws = torch.zeros(va.va_sample_workspace_bytes(n, vocab, 20), dtype=torch.uint8, device=dev)
        u = synth.uniforms(7, n).to(dev)
        outs = [torch.empty(n, 20, dtype=torch.int32, device=dev), torch.empty(n, 20, dtype=torch.float32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev), torch.empty(n, dtype=torch.int32, device=dev)]
        for i in range(2):
            x = synth.logits(700 + i, n).to(dev)
            fns.append(lambda x=x: L.va_sample_topk_topp(P(x.data_ptr()), n, vocab, 20, ctypes.c_float(0.95),
                                                         ctypes.c_float(1.0), P(u.data_ptr()),
                                                         *[P(t.data_ptr()) for t in outs], P(ws.data_ptr()),
                                                         ws.numel(), sp))
        kind, nbytes = "va_sample_topk_topp", 8 * synth.VOCAB * 4
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            for f in fns:
                if f():
                    raise RuntimeError(f"{kind} failed")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            for f in fns:
                if f():
                    raise RuntimeError(f"{kind} failed")
        e1.record(stream)
        e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (args.steps * len(fns))
    print(json.dumps({"kernel_only": kind, "launches": args.steps * len(fns), "us_per_launch": us,
                      "gbs": nbytes / us / 1e3}))


GRAPHED = ("call", "q8call", "treecall")   # A/B units timed as CUDA graphs of whole calls


def ab_order(n_blocks: int):
    """Drift-cancelling order of two arms ("Qwen3.8-27B on one RTX 4090", "Checking the path that actually
    runs"): ABBA then BAAB, repeated, so a linear drift in clocks or temperature weighs both arms equally."""
    pattern = "ABBABAAB"
    return [pattern[i % len(pattern)] for i in range(2 * n_blocks)]


def ab_compare(args, dist: Dist):
    """Two library builds, the same seeded workload, alternated block by block on one GPU."""
    import ctypes
    import hashlib

    import torch

    import speculative_decode_verify_gb300 as va
    from speculative_decode_verify_gb300 import build as vbuild
    from speculative_decode_verify_gb300 import synth

    if dist.rank != 0:
        return
    arms = {}
    for tag, spec in zip("AB", args.ab):
        defs = tuple(d.strip() for d in spec.split(",") if d.strip())
        name = "_ab" + hashlib.sha1(",".join(defs).encode()).hexdigest()[:10] if defs else ""
        vbuild.build(variant=name, defines=defs)
        arms[tag] = dict(spec=spec or "(default build)", lib=va.lib(name), times=[])
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p
    if args.ab_what == "sample":
        return ab_sample(args, arms, dev, stream, sp)
    ctx, window = args.ab_ctx, args.ab_window
    slots = synth.RING_SLOTS if window else ctx + 64
    n_caches = 5 if 512 * ctx > (32 << 20) else 2
    caches = []
    for i in range(n_caches):
        w = synth.make(f"ab{ctx}_{window}", 950 + i, ctx=ctx, n_live=8, window=window, slots=slots)
        kb, vb = synth.bits(w.k_hist), synth.bits(w.v_hist)
        k = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
        v = torch.full((slots, 128), synth.BF16_NAN, dtype=torch.int16)
        first = max(0, ctx - slots) if window else 0
        pp = torch.arange(first, ctx)
        k[pp % slots], v[pp % slots] = kb[first:ctx], vb[first:ctx]
        caches.append(dict(w=w, kb=kb, vb=vb, k=k.to(dev), v=v.to(dev), q=synth.bits(w.q).to(dev),
                           sink=w.sink.to(dev)))
    calls = []
    for j in range(15):                      # three rounds of n_live 4..8 per graph
        n, c = N_LIVES[j % len(N_LIVES)], caches[j % n_caches]
        pos = synth.tail_positions(ctx, n)
        idx = pos[:n].to(torch.int64)
        calls.append(dict(c=c, n=n, pos=pos.to(dev), kn=c["kb"][idx].contiguous().to(dev),
                          vn=c["vb"][idx].contiguous().to(dev),
                          out=torch.empty(8, 6, 128, dtype=torch.int16, device=dev)))
    # each build picks its own split count (the split policy is one of the things an A/B may change)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for arm in arms.values():
        arm["S"] = arm["lib"].va_auto_splits(window + 7 if window else slots, window)
        if args.ab_what in ("tree", "treecall"):   # two node groups share the SMs
            arm["S"] = arm["lib"].va_auto_splits_for(window + 15 if window else slots, window, sms // 2)
    if args.ab_what in ("tree", "treecall"):
        for i, c in enumerate(caches):
            tw = synth.make_tree(f"abtree{i}", 980 + i, base=ctx - synth.TREE_NODES, n_nodes=synth.TREE_NODES)
            c["tree"], c["tq"] = tw.tree.to(dev), synth.bits(tw.q).to(dev)
            # the nodes' own rows (already in the cache) appended again by every tree call
            c["tkn"] = c["kb"][tw.base:tw.base + tw.n_nodes].contiguous().to(dev)
            c["tvn"] = c["vb"][tw.base:tw.base + tw.n_nodes].contiguous().to(dev)
            c["tpos"] = (torch.arange(tw.n_nodes, dtype=torch.int32) + tw.base).to(dev)
        for x in calls:
            x["tout"] = torch.empty(16, 6, 128, dtype=torch.int16, device=dev)
    S = max(arm["S"] for arm in arms.values())
    ws = torch.zeros(2 * va.va_workspace_bytes(S) // 4, dtype=torch.float32, device=dev)   # room for 16 tree rows
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    quant = args.ab_what in ("q8", "q8call")
    if quant:   # the same histories encoded into quantised caches by the library's encoder (build A's)
        LA = arms["A"]["lib"]
        for c in caches:
            c["kc"] = torch.full((slots, 128), 0x7F, dtype=torch.uint8, device=dev)
            c["vc"] = torch.zeros(slots, 128, dtype=torch.int8, device=dev)
            c["ks"] = torch.full((slots,), float("nan"), device=dev)
            c["vs"] = torch.full((slots,), float("nan"), device=dev)
            first = max(0, ctx - slots) if window else 0
            kh, vh = c["kb"][first:ctx].contiguous().to(dev), c["vb"][first:ctx].contiguous().to(dev)
            hpos = torch.arange(first, ctx, dtype=torch.int32, device=dev)
            st = LA.kv_ring_append_q8(P(kh.data_ptr()), P(vh.data_ptr()), ctx - first, P(c["kc"].data_ptr()),
                                      P(c["vc"].data_ptr()), P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), slots,
                                      P(hpos.data_ptr()), None, sp)
            if st:
                raise RuntimeError(f"kv_ring_append_q8 failed with status {st}")
            torch.cuda.synchronize(dev)
            del kh, vh, hpos

    def launch(arm, x):
        L, S = arm["lib"], arm["S"]
        c = x["c"]
        if args.ab_what == "q8call":
            st = L.verify_attn_q8_step(P(c["q"].data_ptr()), P(x["kn"].data_ptr()), P(x["vn"].data_ptr()), 8, x["n"],
                                       P(c["kc"].data_ptr()), P(c["vc"].data_ptr()), P(c["ks"].data_ptr()),
                                       P(c["vs"].data_ptr()), slots, window, P(x["pos"].data_ptr()),
                                       P(c["sink"].data_ptr()), ctypes.c_float(synth.SCALE), S, P(ws.data_ptr()),
                                       P(x["out"].data_ptr()), None, None, P(status.data_ptr()), sp)
        elif args.ab_what == "q8":
            po = ws.data_ptr()
            pl = po + 4 * S * 8 * 6 * 128
            st = L.verify_attn_q8(P(c["q"].data_ptr()), 8, x["n"], P(c["kc"].data_ptr()), P(c["vc"].data_ptr()),
                                  P(c["ks"].data_ptr()), P(c["vs"].data_ptr()), slots, window, P(x["pos"].data_ptr()),
                                  ctypes.c_float(synth.SCALE), S, P(po), P(pl), None, P(status.data_ptr()), sp)
        elif args.ab_what in ("tree", "treecall"):
            po = ws.data_ptr()
            pl = po + 4 * S * 16 * 6 * 128
            st = 0
            if args.ab_what == "treecall":
                st = L.kv_ring_append(P(c["tkn"].data_ptr()), P(c["tvn"].data_ptr()), 16, P(c["k"].data_ptr()),
                                      P(c["v"].data_ptr()), slots, P(c["tpos"].data_ptr()), P(status.data_ptr()), sp)
            st = st or L.verify_attn_tree(P(c["tq"].data_ptr()), 16, 16, P(c["k"].data_ptr()), P(c["v"].data_ptr()),
                                          slots, window, P(c["tree"].data_ptr()), ctypes.c_float(synth.SCALE), S,
                                          P(po), P(pl), None, P(status.data_ptr()), sp)
            if args.ab_what == "treecall":
                st = st or L.attn_split_combine(P(po), P(pl), S, P(c["sink"].data_ptr()), 16, 16,
                                                P(x["tout"].data_ptr()), None, sp)
        elif args.ab_what == "call":
            st = L.verify_attn_step(P(c["q"].data_ptr()), P(x["kn"].data_ptr()), P(x["vn"].data_ptr()), 8, x["n"],
                                    P(c["k"].data_ptr()), P(c["v"].data_ptr()), slots, window, P(x["pos"].data_ptr()),
                                    P(c["sink"].data_ptr()), ctypes.c_float(synth.SCALE), S, P(ws.data_ptr()),
                                    P(x["out"].data_ptr()), None, None, P(status.data_ptr()), sp)
        else:
            po = ws.data_ptr()
            pl = po + 4 * S * 8 * 6 * 128
            fn = L.verify_attn_swa if window else L.verify_attn_full
            extra = (slots, window) if window else (slots,)
            st = fn(P(c["q"].data_ptr()), 8, x["n"], P(c["k"].data_ptr()), P(c["v"].data_ptr()), *extra,
                    P(x["pos"].data_ptr()), ctypes.c_float(synth.SCALE), S, P(po), P(pl), None,
                    P(status.data_ptr()), sp)
        if st:
            raise RuntimeError(f"A/B launch failed with status {st}")

    with torch.cuda.stream(stream):
        graphs = {}
        for tag, arm in arms.items():
            for _ in range(3):
                for x in calls:
                    launch(arm, x)
            if args.ab_what in GRAPHED:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for x in calls:
                        launch(arm, x)
                graphs[tag] = g
        stream.synchronize()
        outs = {}
        for tag, arm in arms.items():   # both builds must compute the same thing
            if args.ab_what in GRAPHED:
                graphs[tag].replay()
            else:
                for x in calls:
                    launch(arm, x)
            stream.synchronize()
            outs[tag] = torch.stack([x["out"].clone() for x in calls]) if args.ab_what in ("call", "q8call") else \
                torch.stack([x["tout"].clone() for x in calls]) if args.ab_what == "treecall" else ws.clone()
        same = bool(torch.equal(outs["A"], outs["B"]))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for tag in ab_order(max(4, args.ab_blocks)):
            arm = arms[tag]
            if args.ab_what in GRAPHED:
                graphs[tag].replay()            # untimed: the block starts from a warm graph
            e0.record(stream)
            for _ in range(args.ab_reps):
                if args.ab_what in GRAPHED:
                    graphs[tag].replay()
                else:
                    for x in calls:
                        launch(arm, x)
            e1.record(stream)
            e1.synchronize()
            arm["times"].append(e0.elapsed_time(e1) * 1e3 / (args.ab_reps * len(calls)))
    if int(status.item()) != 0:
        raise RuntimeError(f"A/B run: device status {int(status.item()):#x}")
    res = {}
    for tag, arm in arms.items():
        t = arm["times"]
        res[tag] = {"defines": arm["spec"], "us_median": statistics.median(t), "us_min": min(t), "us_max": max(t),
                    "us_stdev": statistics.stdev(t) if len(t) > 1 else 0.0, "blocks": [round(x, 3) for x in t]}
    d = [b - a for a, b in zip(arms["A"]["times"], arms["B"]["times"])]
    print(json.dumps({"ab": args.ab_what, "ctx": ctx, "window": window, "n_splits": [arms["A"]["S"], arms["B"]["S"]],
                      "calls_per_block":
                      args.ab_reps * len(calls), "order": "ABBA BAAB", "A": res["A"], "B": res["B"],
                      "b_minus_a_us_median": statistics.median(d), "b_minus_a_us_min": min(d),
                      "b_minus_a_us_max": max(d), "outputs_identical": same,
                      "unit": "us per verify call" if args.ab_what in GRAPHED else
                      "us per split-attention launch"}))


def ab_sample(args, arms, dev, stream, sp):
    """A/B of va_sample_topk_topp: 8 rows x 160,000 logits, top-k 20 / top-p 0.95, 32 rotating logit
    buffers (read cold), 16 calls per CUDA graph."""
    import ctypes

    import torch

    import speculative_decode_verify_gb300 as va
    from speculative_decode_verify_gb300 import synth

    P = ctypes.c_void_p
    n, vocab, k = 8, synth.VOCAB, 20
    xs = [synth.logits(700 + i, n).to(dev) for i in range(32)]
    u = synth.uniforms(7, n).to(dev)
    wsb = va.va_sample_workspace_bytes(n, vocab, k)
    for arm in arms.values():
        arm["ws"] = torch.zeros(wsb, dtype=torch.uint8, device=dev)
        arm["outs"] = [torch.empty(n * k, dtype=torch.int32, device=dev), torch.empty(n * k, device=dev),
                       torch.empty(n, dtype=torch.int32, device=dev), torch.empty(n, dtype=torch.int32, device=dev)]
    per_graph = 16

    def launch(arm, x):
        o = arm["outs"]
        st = arm["lib"].va_sample_topk_topp(P(x.data_ptr()), n, vocab, k, ctypes.c_float(0.95), ctypes.c_float(1.0),
                                            P(u.data_ptr()), P(o[0].data_ptr()), P(o[1].data_ptr()), P(o[2].data_ptr()),
                                            P(o[3].data_ptr()), P(arm["ws"].data_ptr()), wsb, sp)
        if st:
            raise RuntimeError(f"A/B sample launch failed with status {st}")

    with torch.cuda.stream(stream):
        graphs, outs = {}, {}
        for tag, arm in arms.items():
            for i in range(3):
                launch(arm, xs[i])
            launch(arm, xs[5])
            stream.synchronize()
            outs[tag] = [t.clone() for t in arm["outs"]]
            gs = []
            for g0 in range(2):   # two graphs over different buffers: every call reads logits not in L2
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(per_graph):
                        launch(arm, xs[g0 * per_graph + i])
                gs.append(g)
            graphs[tag] = gs
        stream.synchronize()
        same = all(torch.equal(a, b) for a, b in zip(outs["A"], outs["B"]))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for tag in ab_order(max(4, args.ab_blocks)):
            arm = arms[tag]
            graphs[tag][1].replay()
            e0.record(stream)
            for r in range(args.ab_reps):
                graphs[tag][r & 1].replay()
            e1.record(stream)
            e1.synchronize()
            arm["times"].append(e0.elapsed_time(e1) * 1e3 / (args.ab_reps * per_graph))
    res = {}
    for tag, arm in arms.items():
        t = arm["times"]
        res[tag] = {"defines": arm["spec"], "us_median": statistics.median(t), "us_min": min(t), "us_max": max(t),
                    "us_stdev": statistics.stdev(t) if len(t) > 1 else 0.0, "blocks": [round(x, 3) for x in t]}
    d = [b - a for a, b in zip(arms["A"]["times"], arms["B"]["times"])]
    print(json.dumps({"ab": "sample", "rows": n, "vocab": vocab, "top_k": k, "calls_per_block": args.ab_reps * per_graph,
                      "order": "ABBA BAAB", "A": res["A"], "B": res["B"], "b_minus_a_us_median": statistics.median(d),
                      "b_minus_a_us_min": min(d), "b_minus_a_us_max": max(d), "outputs_identical": same,
                      "unit": "us per sampling call"}))


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            reference_arm(args, dist)
        elif args.ab:
            ab_compare(args, dist)
        else:
            ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
