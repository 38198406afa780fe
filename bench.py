#!/usr/bin/env python3
"""Benchmark of the Top-theta hot path on one GB300 (or N replicas).

Default workload: LLaMA-3-8B-shaped decode attention, batch 16, 32 query /
8 KV heads, d = 128, bf16 KV caches of 8192 tokens, 32 layers (layers 0-1
calibrated for k = 512, the rest for k = 128), post-softmax thresholds with
V-mean compensation.  One step = one generated token for the whole batch:
for each of the 32 layers, the running V mean is updated with the appended
token and topt_decode runs (score pass + select/gather pass).

Printed: one JSON line.  value = tokens/s over all ranks (inputs resident);
e2e = the same metric through the public Python API with the step's inputs
copied from pinned host memory and outputs copied back; roofline = the decode
kernel's algorithmic bytes (whole K cache + union V rows + theta + q, mu,
out) / its average launch duration over calls launched back to back;
cpu_baseline = the float64 oracle on a bounded sample, on the host cores.

The line also carries ``decode_workloads`` (the LLaMA-3-70B-shaped decode with
the k~/k drift over row-length buckets under the nearest-row and the fitted
theta(L), and the LLaMA-2-7B-shaped long-context decode with its dense
timing) and ``prefill``: the LLaMA-3-8B-shaped causal prefill (batch 1, 32
query / 8 KV heads, d = 128, 4096 tokens, k = 64) in both threshold modes, as
dense-equivalent TFLOP/s of the executed tiles against the bf16 tensor peak.
``--workload cfg3`` prints that prefill as the line.

``--impl reference`` times the float64 oracle instead (the method has no
other implementation); it needs no GPU.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes
import datetime as dt
import hashlib
import json
import os
import subprocess
import sys
import time

# The oracle's thread pool gives each thread one BLAS thread.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from calibrated_thresholding_gb300 import synth, topt, workloads  # noqa: E402

METRIC = "decode attn tokens/s & HBM GB/s vs 8 TB/s; prefill kept-elem TFLOP/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch, from one ncu capture
# of each kernel, with the hash of the kernel sources the counters were taken
# on; reported as null once the sources differ.
CSRC = os.path.join(ROOT, "calibrated_thresholding_gb300", "csrc")
DECODE_TRAFFIC = {"sources": ["decode.cu", "common.cuh"],
                  "source_sha256": "7b605ed92726ff074a8ac0386e4db346c6fe918ae09d8bb60643e8ea35294192",
                  "bytes_per_launch": 285353216 + 3473152}   # decode_kernel, one layer call (k = 128)
PREFILL_TRAFFIC = {"sources": ["prefill_tc.cu", "prefill_tc_post.cu", "tc.cuh", "common.cuh"],
                   "source_sha256": "79e668380b2a8edbdd1b903880127feb756a209f111fb2309664c0e76a3fbbbe",
                   # the attention kernel of each threshold mode (pre: prefill_tc_kernel,
                   # post: prefill_post_kernel)
                   "bytes_per_launch": {0: 59804416 + 16286464, 1: 59526912 + 22288384}}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["topt", "reference"], default="topt")
    p.add_argument("--workload", choices=["cfg2", "cfg3", "cfg4", "cfg5", "mkc"], default="cfg2",
                   help="mkc: multi-k cumulative calibration on the cfg3 calibration shape")
    p.add_argument("--no-prefill", action="store_true", help="leave out the prefill object")
    p.add_argument("--no-other-decode", action="store_true",
                   help="leave out the 70B-shaped and long-context decode objects")
    p.add_argument("--dense", action="store_true",
                   help="also time the decode step with theta = -inf (on for cfg5)")
    p.add_argument("--prefill-steps", type=int, default=30)
    p.add_argument("--prefill-mode", choices=["post", "pre"], default="post",
                   help="--workload cfg3: post-softmax + VMC, or pre-softmax + exact SDC + VMC")
    p.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--eager", action="store_true",
                   help="launch every step from the host instead of replaying a CUDA graph")
    return p.parse_args()


WORKLOADS = {"cfg2": workloads.CFG2, "cfg4": workloads.CFG4, "cfg5": workloads.CFG5}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def max_over_ranks(x, world, dev):
    """The largest x over the ranks of the job (the slowest replica's time);
    x itself when the job has one rank."""
    if world <= 1:
        return x
    t = torch.tensor([float(x)], device=dev, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(CSRC, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(rec, key=None):
    """DRAM bytes per launch from an ncu capture, while the kernel's sources
    still hash to the captured ones (else None)."""
    if source_sha(rec["sources"]) != rec["source_sha256"]:
        return None
    return rec["bytes_per_launch"] if key is None else rec["bytes_per_launch"].get(key)


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak():
    """Dense bf16 TFLOP/s: the burst figure (the prefill kernel is timed alone)."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        lo = dt.datetime.fromtimestamp(t0)
        hi = dt.datetime.fromtimestamp(t1)
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            if lo <= ts <= hi:
                rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the decode workload, resident on one GPU
# ---------------------------------------------------------------------------
class DecodeState:
    def __init__(self, wl, layers, rank, dev):
        self.wl, self.layers, self.dev = wl, layers, dev
        B, Hq, Hkv, d, n = wl.B, wl.Hq, wl.Hkv, wl.d, wl.n
        self.ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), Hkv, d)
        self.K, self.V, self.q, self.theta, self.mu, self.out = [], [], [], [], [], []
        self.kept, self.vrows, self.cals = [], [], []
        self.seq_len = torch.full((B,), n, device=dev, dtype=torch.int32)
        self.n_old = torch.full((B,), n - 1, device=dev, dtype=torch.int32)
        zero = torch.zeros((B,), device=dev, dtype=torch.int32)
        for l in range(layers):
            gen = synth.generator(synth.seed_of(wl.name, "eval", rank, l), dev)
            K = synth.keys(gen, B, Hkv, n, d, self.ch, device=dev)
            V = synth.values(gen, B, Hkv, n, d, wl.values, device=dev)
            self.K.append(K)
            self.V.append(V)
            self.q.append(synth.decode_queries(gen, K, Hq, [n] * B))
            self.theta.append(self.calibrate(l, dev))
            mu = torch.zeros((B, Hkv, d), device=dev)
            topt.vmean_update(V, zero, n - 1, mu)          # prompt rows 0..n-2
            self.mu.append(mu)
            self.out.append(torch.empty((B, Hq, d), device=dev))
            self.kept.append(torch.empty((B, Hq), device=dev, dtype=torch.int32))
            self.vrows.append(torch.empty((B, Hkv), device=dev, dtype=torch.int32))
        a0 = self.args(0)
        self.ws = topt.decode_workspace(a0, dev)
        self.dargs = []
        self.vargs = []
        self.new_kv = []
        for l in range(layers):
            a = self.args(l)
            a.workspace = ctypes.c_void_p(self.ws.data_ptr())
            a.workspace_bytes = self.ws.numel()
            self.dargs.append(a)
            # the step's new K, V rows (the current token, row n-1), appended
            # by the vmean launch itself
            self.new_kv.append(torch.stack([self.K[l][:, :, n - 1:], self.V[l][:, :, n - 1:]]).contiguous())
            self.vargs.append(topt.vmean_args(self.V[l], self.n_old, 1, self.mu[l], k_cache=self.K[l],
                                              k_new=self.new_kv[l][0], v_new=self.new_kv[l][1]))
        torch.cuda.synchronize()

    def args(self, l):
        wl = self.wl
        return topt.decode_args(self.q[l], self.K[l], self.V[l], self.seq_len, self.theta[l],
                                mode=wl.mode, sdc=wl.sdc, vmc=wl.vmc, mu=self.mu[l],
                                out=self.out[l], kept=self.kept[l], vrows=self.vrows[l])

    def calibrate(self, layer, dev):
        wl = self.wl
        k = wl.k_of(layer)
        cal = topt.Calibrator(wl.Hq, wl.n, k, wl.mode)
        if wl.cal_len == 0:            # decode rows at L = n
            row_len = torch.tensor([wl.n], device=dev, dtype=torch.int32)
            per = max(1, min(wl.n_cal, (1 << 29) // (wl.Hkv * wl.n * wl.d * 2)))
            for s0 in range(0, wl.n_cal, per):
                cnt = min(per, wl.n_cal - s0)
                gen = synth.generator(synth.seed_of(wl.name, "cal", layer, s0), dev)
                K = synth.keys(gen, cnt, wl.Hkv, wl.n, wl.d, self.ch, device=dev)
                q = synth.decode_queries(gen, K, wl.Hq, [wl.n] * cnt)
                cal.add(q[:, :, None, :].contiguous(), K, row_len, reset=(s0 == 0))
                del K, q
        else:                          # causal prefill rows 1..cal_len
            S = wl.cal_len
            row_len = torch.arange(1, S + 1, device=dev, dtype=torch.int32)
            for s0 in range(wl.n_cal):
                gen = synth.generator(synth.seed_of(wl.name, "cal", layer, s0), dev)
                K = synth.keys(gen, 1, wl.Hkv, S, wl.d, self.ch, device=dev)
                Q = synth.prefill_queries(gen, K, wl.Hq)
                cal.add(Q, K, row_len, reset=(s0 == 0))
                del K, Q
        self.cals.append(cal)
        return cal.finalize().clone()

    def fitted_theta(self, layer):
        """The same calibration finalised as the fitted function of ln L."""
        cal = self.cals[layer]
        cal.fit = True
        try:
            return cal.finalize().clone()
        finally:
            cal.fit = False

    def run_step(self, L, stream, events=None):
        for l in range(self.layers):
            rc = L.topt_vmean_update(ctypes.byref(self.vargs[l]), stream)
            if rc:
                raise topt.ToptError("topt_vmean_update", rc)
            a = self.dargs[l]
            if events is not None:
                a.events[0] = events[l][0]
                a.events[1] = events[l][1]
            rc = L.topt_decode(ctypes.byref(a), stream)
            if rc:
                raise topt.ToptError("topt_decode", rc)

    def clear_events(self):
        for a in self.dargs:
            a.events[0] = None
            a.events[1] = None


def graph_of(dev, fn):
    """``fn(stream_handle)`` captured as one CUDA graph on a side stream, replayed
    three times before it is returned."""
    cur = torch.cuda.current_stream(dev)
    gr = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(cur)
    with torch.cuda.graph(gr, stream=cap):
        fn(ctypes.c_void_p(cap.cuda_stream))
    cur.wait_stream(cap)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize(dev)
    return gr


def time_decode_calls(state, L, stream, dev, reps):
    """Duration of one decode call (ms), measured two ways with CUDA events on
    ``stream``.  Back to back: at least 32 decode calls (every layer's, in
    order) in one graph with no event between them, so each call may start
    while the previous one drains as it does inside a step; events around the
    replay, total / calls.  Isolated: events right before and after every call
    (the call then also pays its launch)."""
    layers = state.layers
    per = max(1, 32 // layers)

    def calls(sh):
        for _ in range(per):
            for l in range(layers):
                rc = L.topt_decode(ctypes.byref(state.dargs[l]), sh)
                if rc:
                    raise topt.ToptError("topt_decode", rc)

    g = graph_of(dev, calls)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b2b = []
    for _ in range(reps):
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        b2b.append(e0.elapsed_time(e1) / (per * layers))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]
    for l_ in evs:                 # a torch event exists once recorded
        for e in l_:
            e.record(stream)
    torch.cuda.synchronize(dev)
    hs = [[ctypes.c_void_p(e.cuda_event) for e in l_] for l_ in evs]

    def calls_ev(sh):
        for l in range(layers):
            a = state.dargs[l]
            a.events[0], a.events[1] = hs[l][0], hs[l][1]
            rc = L.topt_decode(ctypes.byref(a), sh)
            if rc:
                raise topt.ToptError("topt_decode", rc)
        state.clear_events()

    g2 = graph_of(dev, calls_ev)
    iso = []
    for _ in range(reps):
        g2.replay()
        torch.cuda.synchronize(dev)
        iso += [evs[l][0].elapsed_time(evs[l][1]) for l in range(layers)]
    return float(np.median(b2b)), float(np.mean(iso))


def decode_roofline(state, b2b_ms, iso_ms):
    """The decode kernel against the measured copy bandwidth: algorithmic bytes
    of one call (whole K cache + union V rows + theta entries + q, mu, out)
    over its back-to-back duration; the isolated call beside it."""
    peak, peak_kind = hbm_peak()
    _, per_layer = algorithmic_bytes(state)
    alg = float(np.mean(per_layer))
    achieved = alg / (b2b_ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak,
            "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
            "traffic": recorded_traffic(DECODE_TRAFFIC) if state.wl is workloads.CFG2 else None,
            "algorithmic_bytes_per_launch": alg,
            "bytes": "whole K cache + union V rows + theta entries + q, mu, out",
            "avg_launch_ms": b2b_ms,
            "timing": "calls launched back to back in one CUDA graph, CUDA events around the replay",
            "isolated_call_ms": iso_ms,
            "isolated_frac": alg / (iso_ms / 1e3) / 1e9 / peak}


def time_dense(state, L, stream, steps, warmup):
    """The decode step with every threshold at -inf (dense attention: every V row
    read), timed eagerly with CUDA events; the thresholds are put back after."""
    dense = torch.full_like(state.theta[0], float("-inf"))
    saved = [a.theta for a in state.dargs]
    for a in state.dargs:
        a.theta = ctypes.c_void_p(dense.data_ptr())
    sh = ctypes.c_void_p(stream.cuda_stream)
    try:
        for _ in range(warmup):
            state.run_step(L, sh)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(state.dev)
        start.record(stream)
        for _ in range(steps):
            state.run_step(L, sh)
        stop.record(stream)
        torch.cuda.synchronize(state.dev)
        ms = start.elapsed_time(stop) / steps
        vrows = float(np.mean([state.vrows[l].double().mean().item() for l in range(state.layers)]))
    finally:
        for a, t in zip(state.dargs, saved):
            a.theta = t
    wl = state.wl
    return {"ms_per_step": ms, "tokens_per_s": wl.B / (ms / 1e3), "vrows_per_group": vrows,
            "theta": "-inf (every valid key kept)", "launch": "eager host launches"}


def drift_sweep(state, theta=None):
    """k~/k per row-length bucket with the first layer's caches at ~16 lengths
    spread over the buckets, through topt.decode with fresh queries per length.
    ``theta`` defaults to the layer's table (rows longer than the calibrated
    ones take the last calibrated row's threshold)."""
    wl = state.wl
    K, V = state.K[0], state.V[0]
    theta = state.theta[0] if theta is None else theta
    per_bucket = {}
    lengths = list(workloads.DRIFT_LENGTHS)
    for c in range(0, len(lengths), wl.B):
        seq = (lengths[c:c + wl.B] + [lengths[-1]] * wl.B)[:wl.B]
        gen = synth.generator(synth.seed_of(wl.name, "drift", c), state.dev)
        q = synth.decode_queries(gen, K, wl.Hq, seq)
        seq_len = torch.tensor(seq, device=state.dev, dtype=torch.int32)
        mu = torch.stack([V[b, :, :L].float().mean(dim=1) for b, L in enumerate(seq)])
        res = topt.decode(q, K, V, seq_len, theta, mode=wl.mode, sdc=wl.sdc, vmc=wl.vmc, mu=mu,
                          workspace=state.ws)
        kept = res["kept"].double().mean(dim=1).cpu().numpy()
        for b, L in enumerate(seq[:len(lengths[c:c + wl.B])]):
            for (lo, hi) in workloads.BUCKETS:
                if lo <= L <= hi:
                    per_bucket.setdefault(f"{lo}-{hi}", []).append(kept[b] / wl.k_of(0))
    return {k: round(float(np.mean(v)), 4) for k, v in per_bucket.items()}


def algorithmic_bytes(state):
    """Per decode call: whole K cache + union V rows + theta entries (+ q, mu, out)."""
    wl = state.wl
    k_bytes = wl.B * wl.Hkv * wl.n * wl.d * 2
    small = wl.B * wl.Hq * wl.d * 2 + wl.B * wl.Hkv * wl.d * 4 + wl.B * wl.Hq * wl.d * 4
    per_layer = []
    for l in range(state.layers):
        vrows = int(state.vrows[l].sum().item())
        per_layer.append(k_bytes + vrows * wl.d * 2 + wl.B * wl.Hq * 4 + small)
    return k_bytes, per_layer


def kept_ratio_by_bucket(state):
    wl = state.wl
    out = {}
    for (lo, hi) in workloads.BUCKETS:
        if lo <= wl.n <= hi:
            r = [state.kept[l].double().mean().item() / wl.k_of(l) for l in range(state.layers)]
            out[f"{lo}-{hi}"] = round(float(np.mean(r)), 4)
    return out


# ---------------------------------------------------------------------------
# the prefill workload
# ---------------------------------------------------------------------------
PREFILL_MODES = (("post-softmax+VMC", 1, 0), ("pre-softmax+exact SDC+VMC", 0, 1))
PREFILL_KERNEL = {0: "prefill_tc_kernel", 1: "prefill_post_kernel"}  # the attention kernel per mode


def prefill_mode(args):
    """The (name, mode, sdc) of the cfg3 line's threshold mode."""
    return PREFILL_MODES[0] if args.prefill_mode == "post" else PREFILL_MODES[1]
L2_FLUSH_BYTES = 256 << 20     # written between timed prefill calls (L2 is 129 MB)


class PrefillState:
    """One causal prefill of `wl` resident on the GPU, theta calibrated on the GPU."""

    def __init__(self, wl, dev, mode, sdc):
        self.wl, self.dev, self.mode, self.sdc = wl, dev, mode, sdc
        B, Hq, Hkv, d, S = wl.B, wl.Hq, wl.Hkv, wl.d, wl.S
        self.ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), Hkv, d)
        cal = topt.Calibrator(Hq, S, wl.k, mode)
        row_len = torch.arange(1, S + 1, device=dev, dtype=torch.int32)
        for s_ in range(wl.n_cal):
            Q, K, _ = self.inputs(synth.seed_of(wl.name, "cal", s_), 1)
            cal.add(Q, K, row_len, reset=(s_ == 0))
        self.theta = cal.finalize().clone()
        self.Q, self.K, self.V = self.inputs(synth.seed_of(wl.name, "eval"), B)
        self.out = torch.empty((B, Hq, S, d), device=dev)
        self.kept = torch.empty((B, Hq, S), device=dev, dtype=torch.int32)
        self.tiles = torch.zeros(2, device=dev, dtype=torch.int64)
        self.args = topt.prefill_args(self.Q, self.K, self.V, self.theta, mode=mode, sdc=sdc,
                                      vmc=True, out=self.out, kept=self.kept, tiles=self.tiles)
        self.ws = torch.empty(max(1, topt.prefill_workspace_bytes(self.args)), device=dev,
                              dtype=torch.uint8)
        self.args.workspace = ctypes.c_void_p(self.ws.data_ptr())
        self.args.workspace_bytes = self.ws.numel()
        self.tile_rows, self.tile_keys = topt.prefill_tile_shape(self.args)

    def inputs(self, seed, B):
        wl = self.wl
        gen = synth.generator(seed & 0xffffffff, self.dev)
        K = synth.keys(gen, B, wl.Hkv, wl.S, wl.d, self.ch, device=self.dev)
        V = synth.values(gen, B, wl.Hkv, wl.S, wl.d, device=self.dev)
        Q = synth.prefill_queries(gen, K, wl.Hq)
        return Q, K, V

    def call(self, L, stream, events=(None, None)):
        self.args.events[0], self.args.events[1] = events
        rc = L.topt_prefill(ctypes.byref(self.args), stream)
        self.args.events[0] = self.args.events[1] = None
        if rc:
            raise topt.ToptError("topt_prefill", rc)


def time_prefill(L, st, stream, steps, warmup):
    """CUDA-event times (s) of whole calls and of the attention kernel, L2 flushed
    between calls.  Whole calls are timed without the inner events (an event
    between the preparation grids and the attention kernel would serialise
    their programmatic overlap); the kernel alone in a second run with them."""
    sh = ctypes.c_void_p(stream.cuda_stream)
    flush = torch.empty(L2_FLUSH_BYTES, device=st.dev, dtype=torch.uint8)
    for _ in range(warmup):
        st.call(L, sh)
    torch.cuda.synchronize(st.dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in ev:            # a torch event exists once recorded: create them all first
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(st.dev)
    st.tiles.zero_()
    for e in ev:
        flush.fill_(1)
        e[0].record(stream)
        st.call(L, sh)
        e[3].record(stream)
    torch.cuda.synchronize(st.dev)
    call_s = [e[0].elapsed_time(e[3]) / 1e3 for e in ev]
    tiles = [int(x) // steps for x in st.tiles.tolist()]
    for e in ev:
        flush.fill_(1)
        st.call(L, sh, (ctypes.c_void_p(e[1].cuda_event), ctypes.c_void_p(e[2].cuda_event)))
    torch.cuda.synchronize(st.dev)
    kern_s = [e[1].elapsed_time(e[2]) / 1e3 for e in ev]
    return call_s, kern_s, tiles


def prefill_flops(st, tiles):
    """Dense-equivalent flops of one call: QK^T over every causal tile plus P.V
    over the executed tiles (the pass-1 recomputation of QK^T not counted)."""
    per_tile = 2.0 * st.wl.d * st.tile_rows * st.tile_keys
    executed, causal = tiles
    return per_tile * (causal + executed), per_tile * (2 * causal + executed)


def prefill_report(L, wl, dev, stream, steps, warmup):
    peak, kind = tensor_peak()
    out = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "S": wl.S,
           "k": wl.k, "modes": []}
    for name, mode, sdc in PREFILL_MODES:
        st = PrefillState(wl, dev, mode, sdc)
        call_s, kern_s, tiles = time_prefill(L, st, stream, steps, warmup)
        useful, issued = prefill_flops(st, tiles)
        kern = float(np.mean(kern_s))
        call = float(np.mean(call_s))
        achieved = useful / kern / 1e12
        kept = st.kept.double()
        kept_total = float(st.kept.double().sum().item())
        out["modes"].append({
            "mode": name, "tflops_call": useful / call / 1e12, "ms_per_call": call * 1e3,
            "kept_elem_tflops_call": kept_elem_flops(wl, kept_total) / call / 1e12,
            "tokens_per_s": wl.B * wl.S / call,
            "roofline": {"bound": "tensor", "kernel": PREFILL_KERNEL[mode], "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_source": f"{kind} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                         if kind == "measured" else "fallback 1.9 PFLOP/s",
                         "traffic": recorded_traffic(PREFILL_TRAFFIC, mode),
                         "avg_launch_ms": kern * 1e3,
                         "flops_per_launch": useful,
                         "flops": "dense-equivalent: QK^T on every causal tile + P.V on executed tiles",
                         "issued_tflops": issued / kern / 1e12},
            "tiles_executed": tiles[0], "tiles_causal": tiles[1],
            "tiles_skipped_frac": 1.0 - tiles[0] / max(1, tiles[1]),
            "tile": [st.tile_rows, st.tile_keys],
            "kept_over_k": round(kept[..., wl.k:].mean().item() / wl.k, 4)})
        del st
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def oracle_rows_per_second(q, K, V, seq_len, theta, mu, wl, rows, seconds, cores):
    """Wall-clock rate of oracle.decode_ref over (b, h) rows on `cores` threads."""
    import oracle.topt_ref as ref
    done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        it = 0
        while True:
            batch = [rows[(it + j) % len(rows)] for j in range(cores * 4)]
            it += len(batch)
            list(ex.map(lambda bh: ref.decode_ref(q, K, V, seq_len, theta, wl.mode, wl.sdc,
                                                   wl.vmc, mu, heads=[bh]), batch))
            done += len(batch)
            if time.perf_counter() - t0 >= seconds:
                break
    return done / (time.perf_counter() - t0), done


SAMPLE_SEQS = 2   # sequences of the batch the host sample holds


def host_decode_sample(wl, layer_ids, n_cal=8, dev="cpu"):
    """Host copies of a few layers (generated on the CPU) for the oracle runs.

    Holds SAMPLE_SEQS sequences of the batch; the oracle's cost per (batch,
    head) row does not depend on which sequence the row belongs to."""
    import oracle.topt_ref as ref
    out = []
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
    B = min(wl.B, SAMPLE_SEQS)
    for l in layer_ids:
        gen = synth.generator(synth.seed_of(wl.name, "host", l), dev)
        K = synth.keys(gen, B, wl.Hkv, wl.n, wl.d, ch)
        V = synth.values(gen, B, wl.Hkv, wl.n, wl.d, wl.values)
        q = synth.decode_queries(gen, K, wl.Hq, [wl.n] * B)
        Kc = synth.keys(gen, n_cal, wl.Hkv, wl.n, wl.d, ch)
        qc = synth.decode_queries(gen, Kc, wl.Hq, [wl.n] * n_cal)
        th, _ = ref.calibrate_ref(synth.as_f64(qc)[:, :, None, :], synth.as_f64(Kc), [wl.n],
                                  wl.k_of(l), wl.mode, 0.0, wl.n)
        Vn = synth.as_f64(V)
        mu = Vn[:, :, :wl.n].mean(axis=2)
        out.append((synth.as_f64(q), synth.as_f64(K), Vn, np.full(B, wl.n), th, mu))
    return out


def cpu_baseline(wl, seconds, layers_total):
    cores = host_cores()
    sample = host_decode_sample(wl, [0, 2])
    rows = [(b, h) for b in range(min(wl.B, SAMPLE_SEQS)) for h in range(wl.Hq)]
    rates = []
    done = 0
    for (q, K, V, sl, th, mu) in sample:
        r, n = oracle_rows_per_second(q, K, V, sl, th, mu, wl, rows, seconds / len(sample), cores)
        rates.append(r)
        done += n
    rate = float(np.mean(rates))                       # (b, h) rows per second
    rows_per_step = wl.B * wl.Hq * layers_total
    return {"value": rate / rows_per_step * wl.B, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{done} (batch, head) decode rows of layers 0 (k={wl.k_of(0)}) and 2 "
                      f"(k={wl.k_of(2)}), float64 numpy, {cores} threads x 1 BLAS thread; "
                      f"scaled to {rows_per_step} rows per step"}


def causal_flops(wl):
    """Dense-equivalent flops of one prefill call over the causal triangle:
    QK^T and P.V on every (i, j <= i) element, 2 d flops each."""
    return 4.0 * wl.d * wl.B * wl.Hq * (wl.S * (wl.S + 1) / 2)


def kept_elem_flops(wl, kept_total):
    """The metric's "kept-element" flops of one prefill call: QK^T on every causal
    element plus P.V on every kept element, 2 d flops each."""
    return 2.0 * wl.d * (wl.B * wl.Hq * (wl.S * (wl.S + 1) / 2) + kept_total)


def host_prefill_sample(wl, n_cal=2, heads=4):
    """One KV group of the prefill workload on the host, theta from the oracle's
    calibration over n_cal sequences (all rows)."""
    import oracle.topt_ref as ref
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)[:1]
    samples = {}
    for mode in (0, 1):
        gen = synth.generator(synth.seed_of(wl.name, "host", mode), "cpu")
        Kc = synth.keys(gen, n_cal, 1, wl.S, wl.d, ch)
        Qc = synth.prefill_queries(gen, Kc, heads)
        th, _ = ref.calibrate_ref(synth.as_f64(Qc), synth.as_f64(Kc), list(range(1, wl.S + 1)),
                                  wl.k, mode, 0.0, wl.S)
        K = synth.keys(gen, 1, 1, wl.S, wl.d, ch)
        V = synth.values(gen, 1, 1, wl.S, wl.d)
        Q = synth.prefill_queries(gen, K, heads)
        samples[mode] = (synth.as_f64(Q), synth.as_f64(K), synth.as_f64(V), th)
    return samples


def oracle_prefill_row_seconds(sample, mode, sdc, rows, cores):
    """Wall-clock seconds per prefill row of the oracle on `cores` threads, and the
    mean kept count of those rows."""
    import oracle.topt_ref as ref
    Q, K, V, th = sample
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        res = list(ex.map(lambda r: ref.prefill_ref(Q, K, V, th, mode, sdc, True, rows=[r]), rows))
    dt = (time.perf_counter() - t0) / len(rows)
    kept = float(np.mean([next(iter(d.values()))["kept"] for d in res]))
    return dt, kept


def prefill_rows_sample(wl, n, heads=4, seed=0):
    rng = np.random.default_rng(seed)
    return [(0, int(rng.integers(heads)), int(i)) for i in rng.integers(0, wl.S, n)]


def prefill_cpu_baseline(wl, seconds, pmode=PREFILL_MODES[0]):
    name, mode, sdc = pmode
    cores = host_cores()
    sample = host_prefill_sample(wl)
    done, spent, kept_sum = 0, 0.0, 0.0
    while spent < seconds:
        rows = prefill_rows_sample(wl, 8 * cores, seed=done)
        dt, kept = oracle_prefill_row_seconds(sample[mode], mode, sdc, rows, cores)
        spent += dt * len(rows)
        kept_sum += kept * len(rows)
        done += len(rows)
    t_row = spent / done
    rows_per_call = wl.B * wl.Hq * wl.S
    kept_total = kept_sum / done * rows_per_call
    return {"value": kept_elem_flops(wl, kept_total) / (t_row * rows_per_call) / 1e12, "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": f"{done} prefill rows (uniform row index, {name}, k={wl.k}), "
                      f"float64 numpy, {cores} threads; scaled to {rows_per_call} rows per call"}


def prefill_config(wl, mode_name, world):
    """The ``config`` of a prefill line (both arms print the same one)."""
    return {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
            "S": wl.S, "k": wl.k, "mode": mode_name,
            "flops": "kept-element: 2 d per causal element (QK^T) + 2 d per kept element (P.V)",
            "l2": f"{L2_FLUSH_BYTES >> 20} MiB written between timed calls",
            "parallelism": f"replicas x{world} (independent prefills per GPU)"}


def run_reference_prefill(args, wl):
    cores = host_cores()
    sample = host_prefill_sample(wl)
    per_step = 4 * cores

    _, mode, sdc = prefill_mode(args)

    def one_step(i):
        rows = prefill_rows_sample(wl, per_step, seed=i)
        return oracle_prefill_row_seconds(sample[mode], mode, sdc, rows, cores)

    for i in range(args.warmup):
        one_step(i)
    runs = [one_step(args.warmup + i) for i in range(args.steps)]
    t_row = sum(r[0] for r in runs) / args.steps
    rows_per_call = wl.B * wl.Hq * wl.S
    kept_total = float(np.mean([r[1] for r in runs])) * rows_per_call
    ms = t_row * rows_per_call * 1e3               # the whole call's rows at the sampled rate
    value = kept_elem_flops(wl, kept_total) / (ms / 1e3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_row * per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(wl, prefill_mode(args)[0], args.gpus),
            "extrapolated": True, "sample_rows_per_step": per_step, "rows_per_step": rows_per_call,
            "note": "ms_per_step is the measured time of the sampled rows of a step; value "
                    "scales their rate to the call's rows",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} prefill rows per step of {rows_per_call}, "
                                       "float64 numpy oracle"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args):
    """--impl reference: the float64 oracle, timed per step on a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if args.workload == "cfg3":
        run_reference_prefill(args, workloads.CFG3)
        return
    if args.workload == "mkc":
        run_reference_mkc(args, workloads.CFG3)
        return
    wl = WORKLOADS[args.workload]
    layers_total = args.layers or wl.layers
    cores = host_cores()
    sample = host_decode_sample(wl, [0, 2])
    rows = [(b, h) for b in range(min(wl.B, SAMPLE_SEQS)) for h in range(wl.Hq)]
    per_step_rows = min(len(rows), 4 * cores)
    import oracle.topt_ref as ref

    def one_step(i):
        q, K, V, sl, th, mu = sample[i % len(sample)]
        chosen = [rows[(i * per_step_rows + j) % len(rows)] for j in range(per_step_rows)]
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(lambda bh: ref.decode_ref(q, K, V, sl, th, wl.mode, wl.sdc, wl.vmc, mu,
                                                   heads=[bh]), chosen))
        return time.perf_counter() - t0

    for i in range(args.warmup):
        one_step(i)
    total = sum(one_step(i) for i in range(args.steps))
    rows_per_step = wl.B * wl.Hq * layers_total
    t_row = total / (args.steps * per_step_rows)
    value = wl.B / (t_row * rows_per_step)      # the whole step's rows at the sampled rate
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(wl, layers_total, args.gpus),
            "extrapolated": True,
            "sample_rows_per_step": per_step_rows, "rows_per_step": rows_per_step,
            "note": "ms_per_step is the measured time of the sampled rows of a step; value "
                    "scales their rate to the step's rows",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step_rows} (batch, head) rows per step of "
                                       f"{rows_per_step}, float64 numpy oracle"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# main (GPU) arm
# ---------------------------------------------------------------------------
def decode_config(wl, layers, world, eager=False):
    """The ``config`` of a decode line (both arms print the same one)."""
    return {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
            "n": wl.n, "layers": layers, "k": wl.k,
            "k_layers_0_1": wl.k_first_layers or wl.k,
            "mode": "post-softmax+VMC" if wl.mode == 1 else "pre-softmax",
            "l2": "inputs larger than L2: each layer call streams a distinct "
                  f"{wl.B * wl.Hkv * wl.n * wl.d * 2 / 1e6:.0f} MB K cache",
            "parallelism": f"replicas x{world} (independent sequences per GPU)",
            "launch": "eager host launches" if eager else "one step replayed as a CUDA graph"}


def decode_step_graph(state, L, dev):
    """One decode step (vmean update + decode per layer) as a CUDA graph."""
    return graph_of(dev, lambda sh: state.run_step(L, sh))


def other_decode_report(wl, L, dev, stream, steps, warmup):
    """A decode workload besides the main line: tokens/s of its step (graph
    replays, CUDA events), the decode kernel's roofline, V rows per group, and
    k~/k -- per row-length bucket for the 70B-shaped workload (nearest-row and
    fitted theta(L)), with dense (theta = -inf) timing for the long-context one."""
    state = DecodeState(wl, wl.layers, 0, dev)
    g = decode_step_graph(state, L, dev)
    for _ in range(warmup):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    step_ms = e0.elapsed_time(e1) / steps
    b2b, iso = time_decode_calls(state, L, stream, dev, max(5, steps // 2))
    out = {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d, "n": wl.n,
           "k": wl.k, "layers": wl.layers,
           "mode": "post-softmax+VMC" if wl.mode == 1 else "pre-softmax",
           "tokens_per_s": wl.B / (step_ms / 1e3), "ms_per_step": step_ms,
           "roofline": decode_roofline(state, b2b, iso),
           "vrows_per_group": float(np.mean([state.vrows[l].double().mean().item()
                                             for l in range(state.layers)])),
           "kept_over_k": kept_ratio_by_bucket(state),
           "gpu_launches_per_step": 2 * wl.layers}
    if wl.cal_len:
        out["kept_over_k_by_bucket"] = {
            "nearest_row": drift_sweep(state),
            "fitted_ln_L": drift_sweep(state, state.fitted_theta(0)),
            "theta": f"calibrated on rows 1..{wl.cal_len} of {wl.n_cal} sequences"}
    if wl is workloads.CFG5:
        dense = time_dense(state, L, stream, max(10, steps), warmup)
        dense["topt_over_dense_speedup"] = dense["ms_per_step"] / step_ms
        out["dense"] = dense
    del state
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.workload == "cfg3":
        main_prefill(args, dev, rank, local, world)
        return
    if args.workload == "mkc":
        main_mkc(args, dev, rank, local, world)
        return
    wl = WORKLOADS[args.workload]
    layers = args.layers or wl.layers

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds, layers)

    from calibrated_thresholding_gb300 import build
    build.build()
    L = topt.lib()
    state = DecodeState(wl, layers, rank, dev)
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        state.run_step(L, sh)
    torch.cuda.synchronize(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the timed step: one CUDA graph (no event inside, so each kernel may start
    # while the previous one drains), or eager host launches
    graph = None if args.eager else decode_step_graph(state, L, dev)
    barrier()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    t0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        if graph is None:
            state.run_step(L, sh)
        else:
            graph.replay()
    stop.record(stream)
    barrier()
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    ms_per_step = ms / args.steps
    tokens = wl.B * args.steps * world
    value = tokens / (ms / 1e3)
    b2b_ms, iso_ms = time_decode_calls(state, L, stream, dev, max(5, args.steps // 4))
    vrows_per_group = float(np.mean([state.vrows[l].double().mean().item() for l in range(layers)]))

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(state, args, dev, world)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": decode_config(wl, layers, world, args.eager),
        "roofline": decode_roofline(state, b2b_ms, iso_ms),
        "vrows_per_group": vrows_per_group,
        "kept_over_k": kept_ratio_by_bucket(state),
        "gpu_launches": args.steps * layers * 2,   # vmean + decode per layer
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if args.workload == "cfg4":
        line["kept_over_k_by_bucket"] = {"nearest_row": drift_sweep(state),
                                         "fitted_ln_L": drift_sweep(state, state.fitted_theta(0))}
    if args.dense or args.workload == "cfg5":
        # after every thresholded figure above: it overwrites kept and vrows
        line["dense"] = time_dense(state, L, stream, max(10, args.steps // 4), args.warmup)
    if cpu is not None:
        line["cpu_baseline"] = cpu
    del state
    torch.cuda.empty_cache()
    if args.workload == "cfg2" and not args.no_other_decode:
        line["decode_workloads"] = [other_decode_report(w, L, dev, stream, 10, 3)
                                    for w in (workloads.CFG4, workloads.CFG5)]
    if not args.no_prefill:
        line["prefill"] = prefill_report(L, workloads.CFG3, dev, stream, args.prefill_steps, 3)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main_prefill(args, dev, rank, local, world):
    """--workload cfg3: the causal prefill as the bench line (post-softmax + VMC)."""
    wl = workloads.CFG3
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = prefill_cpu_baseline(wl, args.cpu_seconds, prefill_mode(args))
    from calibrated_thresholding_gb300 import build
    build.build()
    L = topt.lib()
    name, mode, sdc = prefill_mode(args)
    st = PrefillState(wl, dev, mode, sdc)
    stream = torch.cuda.current_stream(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    t0 = time.time()
    call_s, kern_s, tiles = time_prefill(L, st, stream, args.steps, args.warmup)
    t1 = time.time()
    clk = clocks.stop(t0, t1)
    ms = max_over_ranks(float(np.sum(call_s)) * 1e3, world, dev)
    call = ms / 1e3 / args.steps
    kept_total = float(st.kept.double().sum().item())
    value = kept_elem_flops(wl, kept_total) * world / call / 1e12
    useful, issued = prefill_flops(st, tiles)
    kern = float(np.mean(kern_s))
    peak, kind = tensor_peak()
    achieved = useful / kern / 1e12
    e2e = None if args.no_e2e else prefill_e2e(st, args, dev, world)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": call * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": prefill_config(wl, name, world),
        "roofline": {"bound": "tensor", "kernel": PREFILL_KERNEL[mode], "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"{kind} dense bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
                     if kind == "measured" else "fallback 1.9 PFLOP/s",
                     "traffic": recorded_traffic(PREFILL_TRAFFIC, mode), "avg_launch_ms": kern * 1e3,
                     "flops_per_launch": useful,
                     "flops": "dense-equivalent: QK^T on every causal tile + P.V on executed tiles",
                     "issued_tflops": issued / kern / 1e12},
        "dense_equiv_tflops_call": causal_flops(wl) * world / call / 1e12,
        "tiles_executed": tiles[0], "tiles_causal": tiles[1],
        "tiles_skipped_frac": 1.0 - tiles[0] / max(1, tiles[1]),
        "kept_over_k": round(st.kept.double()[..., wl.k:].mean().item() / wl.k, 4),
        "gpu_launches": args.steps * 3,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


MKC_KS = (16, 32, 64, 128, 256, 512)
MKC_WORKSPACE = 4 << 30     # scores of 8 heads per pass (512 MiB per head)


class _CalInputs:
    """The calibration sequences of a prefill workload, as PrefillState draws them."""

    def __init__(self, wl, dev):
        self.wl, self.dev = wl, dev
        self.ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)

    inputs = PrefillState.inputs


def host_mkc_sample(wl, heads=2):
    """One KV group of the calibration sequences of `wl` on the host, float64."""
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)[:1]
    gen = synth.generator(synth.seed_of(wl.name, "host", 7), "cpu")
    Kc = synth.keys(gen, wl.n_cal, 1, wl.S, wl.d, ch)
    Qc = synth.prefill_queries(gen, Kc, heads)
    return synth.as_f64(Qc), synth.as_f64(Kc)


def oracle_mkc_seconds(sample, groups, mode, cores):
    """Wall-clock seconds of the oracle's Algorithm 2 on (head, row length)
    groups: scores of the group's rows, interval sequences, MergeIntervals and
    the inverse for every k of MKC_KS; returns (seconds, pooled scores)."""
    import oracle.topt_ref as ref
    Q, K = sample

    def one(group):
        h, L = group
        rows = []
        for n in range(Q.shape[0]):
            a = ref.row_scores(Q[n, h, L - 1], K[n, 0], L)
            rows.append(a if mode == 0 else ref.row_softmax(a))
        pieces = ref.merge_intervals([ref.mkc_interval_sequence(r) for r in rows])
        return [ref.mkc_theta(pieces, k) for k in MKC_KS if L > k]

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(one, groups))
    return time.perf_counter() - t0, sum(Q.shape[0] * L for _, L in groups)


def mkc_groups_sample(wl, n, heads=2, seed=0):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(heads)), int(L)) for L in rng.integers(1, wl.S + 1, n)]


def mkc_cpu_baseline(wl, seconds):
    cores = host_cores()
    sample = host_mkc_sample(wl)
    done, spent, pooled = 0, 0.0, 0
    while spent < seconds:
        groups = mkc_groups_sample(wl, 2 * cores, seed=done)
        dt, n = oracle_mkc_seconds(sample, groups, 0, cores)
        spent += dt
        pooled += n
        done += len(groups)
    return {"value": pooled / spent, "unit": "scores/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} (head, row length) groups, length uniform in 1..{wl.S}, "
                      f"{wl.n_cal} rows each, pre-softmax, all {len(MKC_KS)} k; float64 numpy, "
                      f"{cores} threads"}


def mkc_config(wl, world):
    """The ``config`` of a multi-k calibration line (both arms print the same one)."""
    return {"workload": wl.name + " calibration (MKC)", "N": wl.n_cal, "Hq": wl.Hq,
            "Hkv": wl.Hkv, "d": wl.d, "S": wl.S, "ks": list(MKC_KS),
            "l2": "scores workspace of 4 GiB, larger than L2, rewritten every call",
            "parallelism": f"replicas x{world} (independent calibrations per GPU)"}


def run_reference_mkc(args, wl):
    cores = host_cores()
    sample = host_mkc_sample(wl)
    per_step = 2 * cores
    for i in range(args.warmup):
        oracle_mkc_seconds(sample, mkc_groups_sample(wl, per_step, seed=i), 0, cores)
    runs = [oracle_mkc_seconds(sample, mkc_groups_sample(wl, per_step, seed=args.warmup + i), 0, cores)
            for i in range(args.steps)]
    value = sum(r[1] for r in runs) / sum(r[0] for r in runs)
    pooled = wl.n_cal * wl.Hq * wl.S * (wl.S + 1) // 2
    line = {"impl": "reference",
            "metric": "multi-k cumulative calibration: pooled calibration scores per second",
            "value": value, "unit": "scores/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sum(r[0] for r in runs) / args.steps * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": mkc_config(wl, args.gpus),
            "extrapolated": True, "sample_scores_per_step": sum(r[1] for r in runs) // args.steps,
            "scores_per_call": pooled,
            "note": "ms_per_step is the measured time of the sampled groups of a step; value is "
                    "their pooled-score rate",
            "cpu_baseline": {"value": value, "unit": "scores/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} (head, row length) groups per step, "
                                       "float64 numpy oracle, pre-softmax"},
            "e2e": {"value": value, "unit": "scores/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main_mkc(args, dev, rank, local, world):
    """--workload mkc: one layer of multi-k cumulative calibration (App. D,
    Algorithm 2) on the calibration shape of the LLaMA-3-8B prefill workload:
    8 causal sequences of 4096 rows, 32/8 heads, d = 128, bf16; the tables of
    every k in MKC_KS come from one call.  value = pooled calibration scores
    (sequences x heads x causal elements) per second, pre-softmax."""
    wl = workloads.CFG3
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = mkc_cpu_baseline(wl, args.cpu_seconds)
    from calibrated_thresholding_gb300 import build
    build.build()
    topt.lib()
    src = _CalInputs(wl, dev)
    Qs, Ks = zip(*[src.inputs(synth.seed_of(wl.name, "cal", s_), 1)[:2] for s_ in range(wl.n_cal)])
    Q, K = torch.cat(Qs).contiguous(), torch.cat(Ks).contiguous()
    del Qs, Ks
    row_len = torch.arange(1, wl.S + 1, device=dev, dtype=torch.int32)
    ks = torch.tensor(MKC_KS, device=dev, dtype=torch.int32)
    theta = torch.empty((len(MKC_KS), wl.Hq, wl.S), device=dev, dtype=torch.float32)
    status = torch.zeros(1, device=dev, dtype=torch.int32)
    ws = torch.empty(MKC_WORKSPACE + (64 << 20), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    pooled = wl.n_cal * wl.Hq * wl.S * (wl.S + 1) // 2
    per_head = wl.n_cal * wl.S * wl.S * 4
    heads_per_pass = min(wl.Hq, (ws.numel() - (16 << 20)) // per_head)
    passes = -(-wl.Hq // heads_per_pass)
    res = {}
    clocks = ClockSampler(local)
    time.sleep(0.3)
    t0 = time.time()
    for name, mode in (("pre", 0), ("post", 1)):
        for _ in range(args.warmup):
            topt.calibrate_multik(Q, K, row_len, ks, mode, wl.S, theta=theta, status=status, workspace=ws)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            ev[2 * i].record(stream)
            topt.calibrate_multik(Q, K, row_len, ks, mode, wl.S, theta=theta, status=status, workspace=ws)
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize(dev)
        ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]
        if int(status.item()) != 0:
            raise RuntimeError(f"topt_calibrate_multik status {int(status.item())}")
        res[name] = max_over_ranks(float(np.mean(ms)), world, dev)
    # offline SDC estimate E~ beside the k = 64 pre-softmax table, same rows
    ki64 = MKC_KS.index(64)
    topt.calibrate_multik(Q, K, row_len, ks, 0, wl.S, theta=theta, status=status, workspace=ws)
    th64 = theta[ki64].clone()
    sdc_cal = topt.SdcCalibrator(th64, device=dev)
    sdc_ws = ws[:1 << 30]
    for _ in range(args.warmup):
        sdc_cal.add(Q, K, row_len, reset=True, workspace=sdc_ws)
        sdc_cal.finalize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        ev[2 * i].record(stream)
        sdc_cal.add(Q, K, row_len, reset=True, workspace=sdc_ws)
        sdc_cal.finalize()
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    sdc_ms = float(np.mean([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)]))
    clk = clocks.stop(t0, time.time())
    launches_pre = 1 + passes * 2 + 1
    launches_post = launches_pre + passes
    rows_total = wl.n_cal * wl.Hq * wl.S
    sdc_passes = -(-rows_total // min((1 << 30) // (wl.S * 4) // 8 * 8, 65535 * 8))
    line = {
        "metric": "multi-k cumulative calibration: pooled calibration scores per second",
        "value": pooled * world / (res["pre"] / 1e3), "unit": "scores/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["pre"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": mkc_config(wl, world),
        "heads_per_pass": int(heads_per_pass),
        "ms_per_call": res, "pooled_scores": pooled,
        "post_scores_per_s": pooled * world / (res["post"] / 1e3),
        "sdc_offline_calibration": {"ms_per_call": sdc_ms, "table": "k = 64 pre-softmax theta",
                                    "rows": rows_total, "scores_per_s": pooled / (sdc_ms / 1e3)},
        "gpu_launches": args.steps * (launches_pre + launches_post + 2 * sdc_passes + 2),
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def prefill_e2e(st, args, dev, world):
    """The prefill through topt.prefill with Q, K, V copied in from pinned host
    memory and the output copied back, every step."""
    wl = st.wl
    host = [x.cpu().pin_memory() for x in (st.Q, st.K, st.V)]
    out_host = torch.empty_like(st.out, device="cpu").pin_memory()

    def step():
        for d_, h_ in zip((st.Q, st.K, st.V), host):
            d_.copy_(h_, non_blocking=True)
        topt.prefill(st.Q, st.K, st.V, st.theta, mode=st.mode, sdc=st.sdc, vmc=True, out=st.out,
                     kept=st.kept, workspace=st.ws)
        out_host.copy_(st.out, non_blocking=True)

    for _ in range(3):
        step()
    steps = max(5, args.steps // 2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    dt_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = sum(h_.numel() * h_.element_size() for h_ in host)
    kept_total = float(st.kept.double().sum().item())
    return {"value": kept_elem_flops(wl, kept_total) * steps * world / dt_s / 1e12, "unit": "TFLOP/s",
            "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": out_host.numel() * 4}


def run_e2e(state, args, dev, world):
    """The same step through the public API with host inputs and outputs: the
    per-layer calls are prepared once (topt.decode_args / topt.vmean_args, as a
    serving loop would).  Every step copies all layers' q and new K/V rows in
    from pinned host memory (one copy, into the other of two device buffers
    while the previous step computes) and every layer's outputs back (one copy
    per group of eight layers, as soon as the group is done); each layer's
    topt_vmean_update appends its new K/V rows and updates mu, then
    topt_decode runs."""
    wl = state.wl
    layers = state.layers
    B, Hq, Hkv, d = wl.B, wl.Hq, wl.Hkv, wl.d
    group = 8 if layers % 8 == 0 else 1
    # host inputs of a step: per layer q [B][Hq][d] and the new K, V rows [2][B][Hkv][1][d]
    per_in = B * Hq * d + 2 * B * Hkv * d
    in_host = torch.empty(layers * per_in, dtype=torch.bfloat16).pin_memory()
    for l in range(layers):
        o = l * per_in
        in_host[o:o + B * Hq * d].copy_(state.q[l].reshape(-1).cpu())
        in_host[o + B * Hq * d:o + per_in].copy_(state.new_kv[l].reshape(-1).cpu())
    in_dev = [torch.empty_like(in_host, device=dev) for _ in range(2)]
    out_dev = torch.empty((layers, B, Hq, d), device=dev, dtype=torch.float32)
    out_host = torch.empty_like(out_dev, device="cpu").pin_memory()
    L = topt.lib()
    comp = torch.cuda.current_stream(dev)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sh = ctypes.c_void_p(comp.cuda_stream)
    dargs, vargs = [[], []], [[], []]
    for buf in range(2):
        for l in range(layers):
            o = l * per_in
            q_in = in_dev[buf][o:o + B * Hq * d].view(B, Hq, d)
            kv_in = in_dev[buf][o + B * Hq * d:o + per_in].view(2, B, Hkv, 1, d)
            a = topt.decode_args(q_in, state.K[l], state.V[l], state.seq_len, state.theta[l],
                                 mode=wl.mode, sdc=wl.sdc, vmc=wl.vmc, mu=state.mu[l], out=out_dev[l],
                                 kept=state.kept[l], vrows=state.vrows[l])
            a.workspace = ctypes.c_void_p(state.ws.data_ptr())
            a.workspace_bytes = state.ws.numel()
            dargs[buf].append(a)
            vargs[buf].append(topt.vmean_args(state.V[l], state.n_old, 1, state.mu[l], k_cache=state.K[l],
                                              k_new=kv_in[0], v_new=kv_in[1]))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_grp = [torch.cuda.Event() for _ in range(layers // group)]
    ev_out = torch.cuda.Event()
    count = [0]

    def h2d(buf):
        with torch.cuda.stream(cin):
            cin.wait_event(ev_used[buf])           # the step that read this buffer is done with it
            in_dev[buf].copy_(in_host, non_blocking=True)
            ev_in[buf].record(cin)

    def step():
        buf = count[0] & 1
        h2d(buf ^ 1)                               # the next step's inputs travel during this step
        comp.wait_event(ev_in[buf])
        comp.wait_event(ev_out)                    # the previous step's outputs have been read back
        for l in range(layers):
            rc = L.topt_vmean_update(ctypes.byref(vargs[buf][l]), sh)
            rc = rc or L.topt_decode(ctypes.byref(dargs[buf][l]), sh)
            if rc:
                raise topt.ToptError("e2e step", rc)
            if (l + 1) % group == 0:
                g = l // group
                ev_grp[g].record(comp)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_grp[g])
                    out_host[g * group:(g + 1) * group].copy_(out_dev[g * group:(g + 1) * group],
                                                              non_blocking=True)
        ev_used[buf].record(comp)
        ev_out.record(cout)
        count[0] += 1

    h2d(0)
    for _ in range(max(3, args.warmup)):
        step()
    steps = max(10, args.steps // 4)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    dt_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    return {"value": wl.B * steps * world / dt_s, "unit": "tokens/s", "steps": steps,
            "h2d_bytes_per_step": in_host.numel() * 2, "d2h_bytes_per_step": out_host.numel() * 4,
            "calls": "topt_vmean_update (appends the new K/V rows, updates mu) + topt_decode per layer, "
                     "prepared once (topt.vmean_args, topt.decode_args); next step's inputs copied in "
                     "while this step computes, outputs copied back per group of 8 layers"}


if __name__ == "__main__":
    main()
