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
copied from pinned host memory and outputs copied back; roofline = the score
kernel's algorithmic bytes / its CUDA-event duration; cpu_baseline = the
float64 oracle on a bounded sample, on the host cores.

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

# dram__bytes_read.sum + dram__bytes_write.sum per launch of decode_scores_kernel
# (one layer call of the default workload), with the hash of the kernel source
# those counters were taken on.  Reported as null when the source differs.
DECODE_TRAFFIC = {"source_sha256": None, "bytes_per_launch": None}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["topt", "reference"], default="topt")
    p.add_argument("--workload", choices=["cfg2", "cfg4", "cfg5"], default="cfg2")
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


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


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
        self.kept, self.vrows = [], []
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
        for l in range(layers):
            a = self.args(l)
            a.workspace = ctypes.c_void_p(self.ws.data_ptr())
            a.workspace_bytes = self.ws.numel()
            self.dargs.append(a)
            v = topt.VmeanArgs()
            v.batch, v.n_kv_heads, v.head_dim, v.cache_len = B, Hkv, d, n
            v.dtype, v.n_new = topt.BF16, 1
            v.v_cache = ctypes.c_void_p(self.V[l].data_ptr())
            v.n_old = ctypes.c_void_p(self.n_old.data_ptr())
            v.mu = ctypes.c_void_p(self.mu[l].data_ptr())
            self.vargs.append(v)
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
        return cal.finalize().clone()

    def run_step(self, L, stream, events=None):
        for l in range(self.layers):
            rc = L.topt_vmean_update(ctypes.byref(self.vargs[l]), stream)
            if rc:
                raise topt.ToptError("topt_vmean_update", rc)
            a = self.dargs[l]
            if events is not None:
                a.events[0] = events[l][0]
                a.events[1] = events[l][1]
                a.events[2] = events[l][2]
            rc = L.topt_decode(ctypes.byref(a), stream)
            if rc:
                raise topt.ToptError("topt_decode", rc)

    def clear_events(self):
        for a in self.dargs:
            a.events[0] = None
            a.events[1] = None
            a.events[2] = None


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


def run_reference(args):
    """--impl reference: the float64 oracle, timed per step on a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
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
    value = wl.B / (t_row * rows_per_step)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_row * rows_per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                       "n": wl.n, "layers": layers_total},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{per_step_rows} (batch, head) rows per step of "
                                       f"{rows_per_step}, float64 numpy oracle"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# main (GPU) arm
# ---------------------------------------------------------------------------
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
    if args.eager:
        # events around the two decode kernels of every layer call of every step
        ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(layers)]
              for _ in range(args.steps)]
        for s_ in ev:
            for l_ in s_:
                for e in l_:
                    e.record(stream)
        handles = [[[ctypes.c_void_p(e.cuda_event) for e in l_] for l_ in s_] for s_ in ev]
    else:
        # One step captured as a CUDA graph, twice: `graph` times the whole
        # decode call of every layer (events before the score kernel and after
        # the select kernel, which leave the two kernels' overlap intact);
        # `graph_split` adds an event between them to time the score kernel.
        def capture(with_split):
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(layers)]
            for l_ in evs:
                for e in l_:
                    e.record(stream)
            torch.cuda.synchronize(dev)
            hs = [[ctypes.c_void_p(e.cuda_event) for e in l_] for l_ in evs]
            if not with_split:
                for l_ in hs:
                    l_[1] = None
            gr = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(gr, stream=cap):
                state.run_step(L, ctypes.c_void_p(cap.cuda_stream), hs)
            state.clear_events()
            stream.wait_stream(cap)
            for _ in range(3):
                gr.replay()
            torch.cuda.synchronize(dev)
            return gr, evs
        graph, ev1 = capture(False)
        graph_split, ev_split = capture(True)
    barrier()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    t0 = time.time()
    start.record(stream)
    if args.eager:
        for s_ in range(args.steps):
            state.run_step(L, sh, handles[s_])
    else:
        for _ in range(args.steps):
            graph.replay()
    stop.record(stream)
    barrier()
    t1 = time.time()
    state.clear_events()
    clk = clocks.stop(t0, t1)
    ms = start.elapsed_time(stop)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    if args.eager:
        score_ms = [ev[s_][l_][0].elapsed_time(ev[s_][l_][1]) for s_ in range(args.steps) for l_ in range(layers)]
        kern_ms = [ev[s_][l_][0].elapsed_time(ev[s_][l_][2]) for s_ in range(args.steps) for l_ in range(layers)]
    else:
        # whole calls: the last replay of the timed region; score kernel: a
        # short run of the split graph right after it
        kern_ms = [ev1[l_][0].elapsed_time(ev1[l_][2]) for l_ in range(layers)]
        score_ms = []
        for _ in range(max(5, args.steps // 20)):
            graph_split.replay()
            torch.cuda.synchronize(dev)
            score_ms += [ev_split[l_][0].elapsed_time(ev_split[l_][1]) for l_ in range(layers)]
    ms_per_step = ms / args.steps
    tokens = wl.B * args.steps * world
    value = tokens / (ms / 1e3)

    k_bytes, per_layer = algorithmic_bytes(state)
    kern_avg = float(np.mean(kern_ms)) / 1e3
    score_avg = float(np.mean(score_ms)) / 1e3
    peak, peak_kind = hbm_peak()
    alg_bytes = float(np.mean(per_layer))
    q_bytes = wl.B * wl.Hq * wl.d * 2
    achieved = (k_bytes + q_bytes) / score_avg / 1e9
    call_gbs = alg_bytes / kern_avg / 1e9
    traffic = None
    src = os.path.join(ROOT, "calibrated_thresholding_gb300", "csrc", "decode.cu")
    if DECODE_TRAFFIC["source_sha256"] == source_sha(src):
        traffic = DECODE_TRAFFIC["bytes_per_launch"]
    vrows_per_group = float(np.mean([state.vrows[l].double().mean().item() for l in range(layers)]))

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(state, args, dev, world)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "n": wl.n, "layers": layers, "k": wl.k,
                   "k_layers_0_1": wl.k_first_layers or wl.k,
                   "mode": "post-softmax+VMC" if wl.mode == 1 else "pre-softmax",
                   "l2": "inputs larger than L2: each layer call streams a distinct "
                         f"{k_bytes / 1e6:.0f} MB K cache",
                   "parallelism": f"replicas x{world} (independent sequences per GPU)",
                   "launch": "eager host launches" if args.eager else "one step replayed as a CUDA graph"},
        "roofline": {"bound": "hbm", "kernel": "decode_scores_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": k_bytes + q_bytes,
                     "bytes": "whole K cache + q",
                     "avg_launch_ms": score_avg * 1e3},
        "decode_call": {"gbs": call_gbs, "frac_of_measured": call_gbs / peak,
                        "frac_of_8tbs": call_gbs / NOMINAL_HBM_GBS, "avg_ms": kern_avg * 1e3,
                        "select_avg_ms": (kern_avg - score_avg) * 1e3,
                        "bytes_per_call": alg_bytes,
                        "bytes": "whole K cache + union V rows + theta entries + q, mu, out"},
        "vrows_per_group": vrows_per_group,
        "kept_over_k": kept_ratio_by_bucket(state),
        "gpu_launches": args.steps * layers * 2,
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


def run_e2e(state, args, dev, world):
    """Same step through topt.decode with host inputs copied in and outputs copied out."""
    wl = state.wl
    layers = state.layers
    q_host = [state.q[l].cpu().pin_memory() for l in range(layers)]
    kv_host = [torch.stack([state.K[l][:, :, wl.n - 1], state.V[l][:, :, wl.n - 1]]).cpu().pin_memory()
               for l in range(layers)]
    out_host = [torch.empty_like(state.out[l], device="cpu").pin_memory() for l in range(layers)]
    kv_dev = torch.empty_like(kv_host[0], device=dev)

    def step():
        for l in range(layers):
            state.q[l].copy_(q_host[l], non_blocking=True)
            kv_dev.copy_(kv_host[l], non_blocking=True)
            state.K[l][:, :, wl.n - 1].copy_(kv_dev[0])
            state.V[l][:, :, wl.n - 1].copy_(kv_dev[1])
            topt.vmean_update(state.V[l], state.n_old, 1, state.mu[l])
            topt.decode(state.q[l], state.K[l], state.V[l], state.seq_len, state.theta[l],
                        mode=wl.mode, sdc=wl.sdc, vmc=wl.vmc, mu=state.mu[l], out=state.out[l],
                        kept=state.kept[l], vrows=state.vrows[l], workspace=state.ws)
            out_host[l].copy_(state.out[l], non_blocking=True)

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
    dt_s = time.perf_counter() - t0
    if world > 1:
        t = torch.tensor([dt_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        dt_s = float(t.item())
    h2d = sum(q_host[l].numel() * 2 + kv_host[l].numel() * 2 for l in range(layers))
    d2h = sum(out_host[l].numel() * 4 for l in range(layers))
    return {"value": wl.B * steps * world / dt_s, "unit": "tokens/s", "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


if __name__ == "__main__":
    main()
