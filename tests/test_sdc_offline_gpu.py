"""GPU parity of the offline-calibrated SDC estimate (Top-Theta §3.2.1,
estimator 1): topt_calibrate_sdc against the float64 oracle, and decode and
prefill with TOPT_SDC_OFFLINE.

Thresholds and E~ tables come from the oracle's own calibration on seeded
calibration sequences (rounded to fp32, the form the library takes), so both
sides see identical tables.
"""
import numpy as np
import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt

from gpu_cases import decode_case, mask_words, prefill_case
from parity import check_decode, check_prefill, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_cuda()
    build.build()
    topt.lib()


def _oracle_tables(seed, N, Hq, Hkv, d, S, k, Lmax, dtype):
    """theta (pre-softmax, Algorithm 1) and E~ from N causal calibration
    sequences of length S, by the oracle; returned as fp32 tables and the
    calibration inputs."""
    Qs, Ks = [], []
    for n in range(N):
        Q, K, _ = prefill_case(seed * 1000 + n, 1, Hq, Hkv, d, S, dtype)
        Qs.append(Q)
        Ks.append(K)
    Q, K = torch.cat(Qs).contiguous(), torch.cat(Ks).contiguous()
    Qn, Kn = synth.as_f64(Q), synth.as_f64(K)
    rows = np.arange(1, S + 1)
    th, _ = ref.calibrate_ref(Qn, Kn, rows, k, ref.PRE, 0.0, Lmax)
    th32 = th.astype(np.float32).astype(np.float64)
    et, _ = ref.calibrate_discarded_ref(Qn, Kn, rows, th32)
    return th32, et.astype(np.float32).astype(np.float64), Q, K


def _band_slack(Qn, Kn, rows, theta):
    """Per table cell, the mean exponent mass of calibration elements within
    the decision band of theta: a decision there may go either way in fp32."""
    N, Hq, R, _ = Qn.shape
    g = Hq // Kn.shape[1]
    Lmax = theta.shape[1]
    sets = {}
    for n in range(N):
        for h in range(Hq):
            for i in range(R):
                L = int(rows[i])
                t = ref.theta_for_row(theta[h], L)
                if not np.isfinite(t):
                    continue
                a = ref.row_scores(Qn[n, h, i], Kn[n, h // g], L)
                band = np.abs(a - t) <= ref.BAND_REL * abs(t)
                sets.setdefault((h, L), []).append(float(np.exp(a[band] - a.max()).sum()))
    out = np.zeros((Hq, Lmax))
    for h in range(Hq):
        value = {L: float(np.mean(v)) for (hh, L), v in sets.items() if hh == h}
        row = ref.fill_row_ids(value, Lmax, 0)
        row[~np.isfinite(row)] = 0.0
        out[h] = row
    return out


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_sdc_calibration_matches_oracle(d, dtype):
    N, Hq, Hkv, S, k, Lmax = 3, 4, 2, 64, 6, 80
    th32, _, _, _ = _oracle_tables(81, 2, Hq, Hkv, d, S, k, Lmax, dtype)
    Qs, Ks = zip(*[prefill_case(82 * 1000 + n, 1, Hq, Hkv, d, S, dtype)[:2] for n in range(N)])
    theta = torch.tensor(th32, dtype=torch.float32, device="cuda")
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    cal = topt.SdcCalibrator(theta)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    cal.add(Qs[0], Ks[0], row_len, reset=True, status=status)
    cal.add(torch.cat(Qs[1:]).contiguous(), torch.cat(Ks[1:]).contiguous(), row_len, status=status)
    got = cal.finalize(status=status).cpu().double().numpy()
    assert int(status.item()) == 0
    Qn = synth.as_f64(torch.cat(Qs))
    Kn = synth.as_f64(torch.cat(Ks))
    want, sets = ref.calibrate_discarded_ref(Qn, Kn, np.arange(1, S + 1), th32)
    cnt = cal.count.cpu().numpy()
    for (h, L), v in sets.items():
        assert cnt[h, L - 1] == len(v), (h, L)
    assert np.all(got[~np.isfinite(th32)] == 0.0)
    slack = _band_slack(Qn, Kn, np.arange(1, S + 1), th32)
    err = np.abs(got - want)
    tol = 1e-4 * np.abs(want) + 1e-6 + slack
    assert np.all(err <= tol), float(np.max(err - tol))


@pytest.mark.parametrize("vmc", [True, False])
def test_decode_offline_sdc_matches_oracle(vmc):
    B, Hq, Hkv, d, Nmax, k = 3, 8, 2, 128, 600, 12
    seq = [600, 1, 333]
    th32, et32, _, _ = _oracle_tables(83, 2, Hq, Hkv, d, 96, k, Nmax, torch.bfloat16)
    assert np.any(et32 > 0)
    q, K, V, _ = decode_case(84, B, Hq, Hkv, d, Nmax, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = torch.stack([V[b, :, :int(L)].float().mean(dim=1) for b, L in enumerate(seq)])
    theta = torch.tensor(th32, dtype=torch.float32, device="cuda")
    et = torch.tensor(et32, dtype=torch.float32, device="cuda")
    mask = torch.zeros((B, Hq, mask_words(Nmax)), device="cuda", dtype=torch.int32) - 1
    res = topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_OFFLINE, vmc=vmc, mu=mu,
                      mask=mask, e_tilde=et)
    torch.cuda.synchronize()
    check_decode(q, K, V, seq_len, theta, ref.PRE, ref.SDC_OFFLINE, vmc, mu if vmc else None, res,
                 e_tilde=et)
    # without its table the offline mode is refused on the host
    with pytest.raises(topt.ToptError):
        topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_OFFLINE, vmc=vmc, mu=mu)


@pytest.mark.parametrize("d,dtype,S", [(128, torch.bfloat16, 300), (64, torch.float32, 129)])
def test_prefill_offline_sdc_matches_oracle(d, dtype, S):
    B, Hq, Hkv, k = 1, 4, 2, 8
    th32, et32, _, _ = _oracle_tables(85, 2, Hq, Hkv, d, 64, k, 80, dtype)
    Q, K, V = prefill_case(86, B, Hq, Hkv, d, S, dtype)
    theta = torch.tensor(th32, dtype=torch.float32, device="cuda")
    et = torch.tensor(et32, dtype=torch.float32, device="cuda")
    for vmc in (True, False):
        mask = torch.full((B, Hq, S, mask_words(S)), -1, device="cuda", dtype=torch.int32)
        res = topt.prefill(Q, K, V, theta, mode=ref.PRE, sdc=ref.SDC_OFFLINE, vmc=vmc, mask=mask,
                           e_tilde=et)
        torch.cuda.synchronize()
        check_prefill(Q, K, V, theta, ref.PRE, ref.SDC_OFFLINE, vmc, res, e_tilde=et)
