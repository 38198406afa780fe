"""GPU parity at the five workloads' full sizes.

Decode: every (batch, head) row is checked against the oracle.  Prefill at
S = 4096: the masks and kept counts of every row of every head against the
oracle's whole-matrix decisions, and the outputs of one row in 16 per head
(every 128-row block).  The single-head fp32 workload runs every combination
of threshold mode, SDC and VMC.  The theta tables come from the GPU
calibration and are checked against the oracle's Algorithm 1 on the cells the
oracle can afford.  Masks must agree outside the 1e-3 band around theta
(at most 1e-4 of the elements compared, recorded per case), outputs within
2e-3.
"""
import numpy as np
import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt, workloads

from gpu_cases import mask_words, prefill_case
import parity
from parity import check_decode, check_prefill, check_prefill_all_masks, record_band, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_cuda()
    build.build()
    topt.lib()


def decode_calibration(wl, layer, ch, seqs):
    """GPU calibration of one layer (the bench recipe) + the raw calibration rows."""
    k = wl.k_of(layer)
    cal = topt.Calibrator(wl.Hq, wl.n, k, wl.mode)
    kept_rows = []
    if wl.cal_len == 0:
        row_len = torch.tensor([wl.n], device="cuda", dtype=torch.int32)
        for s in range(wl.n_cal):
            gen = synth.generator(synth.seed_of(wl.name, "test-cal", layer, s), "cuda")
            K = synth.keys(gen, 1, wl.Hkv, wl.n, wl.d, ch, device="cuda")
            q = synth.decode_queries(gen, K, wl.Hq, [wl.n])
            cal.add(q[:, :, None, :].contiguous(), K, row_len, reset=(s == 0))
            if s < seqs:
                kept_rows.append((q, K))
    else:
        S = wl.cal_len
        row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
        for s in range(wl.n_cal):
            gen = synth.generator(synth.seed_of(wl.name, "test-cal", layer, s), "cuda")
            K = synth.keys(gen, 1, wl.Hkv, S, wl.d, ch, device="cuda")
            Q = synth.prefill_queries(gen, K, wl.Hq)
            cal.add(Q, K, row_len, reset=(s == 0))
            if s < seqs:
                kept_rows.append((Q, K))
    return cal.finalize().clone(), cal, kept_rows


def check_decode_calibration(wl, theta, cal, layer, ch, heads):
    """Oracle Algorithm 1 over all calibration sequences for a few heads."""
    k = wl.k_of(layer)
    got = theta.cpu().double().numpy()
    for h in heads:
        sets = {}
        for s in range(wl.n_cal):
            gen = synth.generator(synth.seed_of(wl.name, "test-cal", layer, s), "cuda")
            K = synth.keys(gen, 1, wl.Hkv, wl.n, wl.d, ch, device="cuda")
            q = synth.decode_queries(gen, K, wl.Hq, [wl.n])
            kv = h // (wl.Hq // wl.Hkv)
            a = ref.row_scores(synth.as_f64(q[0, h]), synth.as_f64(K[0, kv]), wl.n)
            sets.setdefault((0, wl.n), []).append(ref.calibration_sample(a, k, wl.mode))
        want = ref.finalize_thresholds(sets, 1, wl.n, k, 0.0)[0]
        assert int(cal.count[h, wl.n - 1]) == wl.n_cal
        w = want[wl.n - 1]
        assert abs(got[h, wl.n - 1] - w) <= 1e-4 * (abs(w) + 1e-6), (h, got[h, wl.n - 1], w)
        assert np.all(got[h, : k] == -np.inf)
        assert np.all(got[h, k:] == got[h, wl.n - 1])   # one calibrated row: nearest-row rule


def decode_full(wl, layer, seq, seed_tag, vmc_mu=True):
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
    gen = synth.generator(synth.seed_of(wl.name, seed_tag, layer), "cuda")
    K = synth.keys(gen, wl.B, wl.Hkv, wl.n, wl.d, ch, device="cuda")
    V = synth.values(gen, wl.B, wl.Hkv, wl.n, wl.d, wl.values, device="cuda")
    q = synth.decode_queries(gen, K, wl.Hq, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = torch.zeros((wl.B, wl.Hkv, wl.d), device="cuda")
    topt.vmean_update(V, torch.zeros_like(seq_len), min(seq), mu)
    for b, L in enumerate(seq):                 # per-sequence lengths: finish on the host side
        if L > min(seq):
            mu[b] = V[b, :, :L].float().mean(dim=1)
    return ch, K, V, q, seq_len, mu


def run_and_check(wl, q, K, V, seq_len, theta, mu, mode=None, sdc=None):
    mode = wl.mode if mode is None else mode
    sdc = wl.sdc if sdc is None else sdc
    mask = torch.full((wl.B, wl.Hq, mask_words(wl.n)), -1, device="cuda", dtype=torch.int32)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    res = topt.decode(q, K, V, seq_len, theta, mode=mode, sdc=sdc, vmc=wl.vmc, mu=mu, mask=mask,
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n, n_band, worst = check_decode(q, K, V, seq_len, theta, mode, sdc, wl.vmc, mu, res)
    return res, n_band, worst


def test_cfg2_llama3_8b_decode():
    wl = workloads.CFG2
    for layer in (0, 2):                              # k = 512 and k = 128
        ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
        theta, cal, _ = decode_calibration(wl, layer, ch, 0)
        check_decode_calibration(wl, theta, cal, layer, ch, heads=(0, 13, 31))
        ch, K, V, q, seq_len, mu = decode_full(wl, layer, [wl.n] * wl.B, "test-eval")
        res, n_band, worst = run_and_check(wl, q, K, V, seq_len, theta, mu)
        record_band(wl.name, f"layer {layer} (k = {wl.k_of(layer)})")
        ratio = res["kept"].double().mean().item() / wl.k_of(layer)
        print(f"cfg2 layer {layer}: k~/k {ratio:.3f}, V rows/group "
              f"{res['vrows'].double().mean().item():.1f}, band elements {n_band}, max err {worst:.2e}")


def test_cfg4_llama3_70b_decode_and_drift():
    wl = workloads.CFG4
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
    theta, cal, _ = decode_calibration(wl, 0, ch, 0)
    got = theta.cpu().numpy()
    assert np.all(got[:, : wl.k] == -np.inf)
    assert np.all(np.isfinite(got[:, wl.k: wl.cal_len]))
    assert np.all(got[:, wl.cal_len:] == got[:, wl.cal_len - 1: wl.cal_len])   # nearest row
    # full length
    ch, K, V, q, seq_len, mu = decode_full(wl, 0, [wl.n] * wl.B, "test-eval")
    _, n_band, _ = run_and_check(wl, q, K, V, seq_len, theta, mu)
    record_band(wl.name, "full length")
    # drift sweep over the row-length buckets, same caches
    lengths = list(workloads.DRIFT_LENGTHS)
    per_bucket = {}
    tally = {"elements": 0, "band": 0, "band_disagree": 0}
    for c in range(0, len(lengths), wl.B):
        seq = lengths[c:c + wl.B]
        ch, K, V, q, seq_len, mu = decode_full(wl, 0, seq, "test-eval")
        res, _, _ = run_and_check(wl, q, K, V, seq_len, theta, mu)
        for key in tally:
            tally[key] += parity.LAST[key]
        kept = res["kept"].cpu().numpy()
        for b, L in enumerate(seq):
            for (lo, hi) in workloads.BUCKETS:
                if lo <= L <= hi:
                    per_bucket.setdefault(f"{lo}-{hi}", []).append(kept[b].mean() / wl.k)
    record_band(wl.name, "drift sweep lengths", tally)
    print("cfg4 k~/k per bucket:", {k: round(float(np.mean(v)), 3) for k, v in per_bucket.items()})


def test_cfg5_llama2_mhsa_long_decode_and_dense():
    wl = workloads.CFG5
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
    theta, cal, _ = decode_calibration(wl, 0, ch, 0)
    check_decode_calibration(wl, theta, cal, 0, ch, heads=(0, 31))
    ch, K, V, q, seq_len, mu = decode_full(wl, 0, [wl.n] * wl.B, "test-eval")
    _, n_band, _ = run_and_check(wl, q, K, V, seq_len, theta, mu)
    record_band(wl.name, "full length")
    dense = torch.full_like(theta, float("-inf"))
    res, _, _ = run_and_check(wl, q, K, V, seq_len, dense, mu)
    assert int(res["vrows"].min()) == wl.n


CFG1_CASES = [(mode, sdc, vmc) for mode in (ref.PRE, ref.POST) for sdc in (ref.SDC_NONE, ref.SDC_EXACT)
              for vmc in (False, True)] + [(ref.PRE, ref.SDC_EXPTH, False), (ref.PRE, ref.SDC_EXPTH, True)]


@pytest.mark.parametrize("mode,sdc,vmc", CFG1_CASES)
def test_cfg1_single_head_fp32(mode, sdc, vmc):
    wl = workloads.CFG1
    Qs, Ks = [], []
    cal = topt.Calibrator(wl.Hq, wl.S, wl.k, mode)
    row_len = torch.arange(1, wl.S + 1, device="cuda", dtype=torch.int32)
    for s in range(wl.n_cal):
        Q, K, _ = prefill_case(synth.seed_of(wl.name, "cal", s) & 0xffffffff, 1, 1, 1, wl.d, wl.S,
                               torch.float32, iid=True)
        cal.add(Q, K, row_len, reset=(s == 0))
        Qs.append(synth.as_f64(Q)[0])
        Ks.append(synth.as_f64(K)[0])
    theta = cal.finalize().clone()
    want, _ = ref.calibrate_ref(np.stack(Qs), np.stack(Ks), np.arange(1, wl.S + 1), wl.k, mode, 0.0, wl.S)
    got = theta.cpu().double().numpy()
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    fin = np.isfinite(want)
    assert np.all(np.abs(got[fin] - want[fin]) <= 1e-4 * (np.abs(want[fin]) + 1e-6))
    Q, K, V = prefill_case(synth.seed_of(wl.name, "eval") & 0xffffffff, 1, 1, 1, wl.d, wl.S,
                           torch.float32, iid=True)
    mask = torch.full((1, 1, wl.S, mask_words(wl.S)), -1, device="cuda", dtype=torch.int32)
    res = topt.prefill(Q, K, V, theta, mode=mode, sdc=sdc, vmc=vmc, mask=mask)
    torch.cuda.synchronize()
    n, n_band, worst, _ = check_prefill(Q, K, V, theta, mode, sdc, vmc, res)
    record_band(wl.name, f"mode {mode} sdc {sdc} vmc {int(vmc)}")


@pytest.mark.parametrize("mode,sdc", [(ref.PRE, ref.SDC_EXACT), (ref.POST, ref.SDC_NONE)])
def test_cfg3_llama3_8b_prefill(mode, sdc):
    wl = workloads.CFG3
    ch = synth.outlier_channels(synth.seed_of(wl.name, "channels"), wl.Hkv, wl.d)
    cal = topt.Calibrator(wl.Hq, wl.S, wl.k, mode)
    row_len = torch.arange(1, wl.S + 1, device="cuda", dtype=torch.int32)
    for s in range(wl.n_cal):
        Q, K, _ = prefill_case(synth.seed_of(wl.name, "cal", s) & 0xffffffff, 1, wl.Hq, wl.Hkv, wl.d,
                               wl.S, channels=ch)
        cal.add(Q, K, row_len, reset=(s == 0))
    theta = cal.finalize().clone()
    # theta of a few cells against Algorithm 1 over the same 8 sequences
    cells = [(0, 100), (7, 4096), (31, 2049)]
    got = theta.cpu().double().numpy()
    for (h, L) in cells:
        obs = []
        for s in range(wl.n_cal):
            Q, K, _ = prefill_case(synth.seed_of(wl.name, "cal", s) & 0xffffffff, 1, wl.Hq, wl.Hkv,
                                   wl.d, wl.S, channels=ch)
            a = ref.row_scores(synth.as_f64(Q[0, h, L - 1]), synth.as_f64(K[0, h // 4]), L)
            obs.append(ref.calibration_sample(a, wl.k, mode))
        w = float(np.mean(obs))
        assert abs(got[h, L - 1] - w) <= 1e-4 * (abs(w) + 1e-6), (h, L, got[h, L - 1], w)
    Q, K, V = prefill_case(synth.seed_of(wl.name, "eval") & 0xffffffff, 1, wl.Hq, wl.Hkv, wl.d, wl.S,
                           channels=ch)
    mask = torch.full((1, wl.Hq, wl.S, mask_words(wl.S)), -1, device="cuda", dtype=torch.int32)
    tiles = torch.zeros(2, device="cuda", dtype=torch.int64)
    res = topt.prefill(Q, K, V, theta, mode=mode, sdc=sdc, vmc=True, mask=mask, tiles=tiles)
    torch.cuda.synchronize()
    stats = check_prefill_all_masks(Q, K, theta, mode, res)
    record_band(wl.name, f"mode {mode} sdc {sdc} vmc 1 (every row of every head)", stats)
    n_band = stats["band"]
    rows = [(0, h, i) for h in range(wl.Hq) for i in range(h % 16, wl.S, 16)]   # every 128-row block
    n, _, worst, _ = check_prefill(Q, K, V, theta, mode, sdc, True, res, rows=rows)
    kept = res["kept"].double()
    rows_long = kept[0, :, wl.k:]
    print(f"cfg3 mode {mode}: k~/k {rows_long.mean().item() / wl.k:.3f}, tiles executed "
          f"{tiles[0].item()}/{tiles[1].item()}, band {n_band}, max err {worst:.2e}")
