"""GPU parity of calibration with a fitted function of ln L (topt_calibrate
with TOPT_CALIB_FIT) against the float64 oracle: prefill calibration rows,
pre and post softmax, alpha 0 and 0.5, a table longer than the calibrated
rows (extrapolation), and decode rows at three and at one length.
"""
import numpy as np
import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt

from gpu_cases import prefill_case
from parity import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_cuda()
    build.build()
    topt.lib()


def _compare(got, want, tol_rel):
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    fin = np.isfinite(want)
    err = np.abs(got[fin] - want[fin])
    # relative, with a floor of 5 % of the table's median magnitude so that a
    # fitted value passing near zero keeps a meaningful bound
    tol = tol_rel * (np.abs(want[fin]) + 0.05 * np.median(np.abs(want[fin])))
    assert np.all(err <= tol), float(np.max(err / tol))


@pytest.mark.parametrize("mode", [ref.PRE, ref.POST])
@pytest.mark.parametrize("alpha", [0.0, 0.5])
def test_fitted_calibration_matches_oracle(mode, alpha):
    N, Hq, Hkv, d, S, k, Lmax = 3, 4, 2, 128, 64, 5, 160
    Qs, Ks = zip(*[prefill_case(101 * 1000 + n, 1, Hq, Hkv, d, S)[:2] for n in range(N)])
    Q, K = torch.cat(Qs).contiguous(), torch.cat(Ks).contiguous()
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    cal = topt.Calibrator(Hq, Lmax, k, mode, alpha, fit=True)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    cal.add(Q, K, row_len, reset=True, status=status)
    got = cal.finalize(status=status).cpu().double().numpy()
    assert int(status.item()) == 0
    want, _ = ref.calibrate_ref(synth.as_f64(Q), synth.as_f64(K), np.arange(1, S + 1), k, mode, alpha,
                                Lmax, fit=True)
    # calibrated values agree to ~1e-5 (fp32 scores); the fit and its
    # extrapolation to 2.5x the calibrated length amplify that a few times
    _compare(got, want, 5e-4 if alpha == 0.0 else 2e-3)


@pytest.mark.parametrize("lens", [[20, 50, 90], [40]])
def test_fitted_calibration_decode_rows(lens):
    N, Hq, Hkv, d, Lmax, k = 4, 2, 1, 64, 128, 8
    gen = synth.generator(103, "cuda")
    K = synth.iid_normal(gen, (N, Hkv, max(lens), d), "cuda", torch.float32)
    Q = synth.iid_normal(gen, (N, Hq, len(lens), d), "cuda", torch.float32)
    row_len = torch.tensor(lens, device="cuda", dtype=torch.int32)
    for mode in (ref.PRE, ref.POST):
        cal = topt.Calibrator(Hq, Lmax, k, mode, 0.0, fit=True)
        cal.add(Q, K, row_len, reset=True)
        got = cal.finalize().cpu().double().numpy()
        want, _ = ref.calibrate_ref(synth.as_f64(Q), synth.as_f64(K), lens, k, mode, 0.0, Lmax, fit=True)
        _compare(got, want, 5e-4)
