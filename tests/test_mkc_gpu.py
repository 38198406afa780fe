"""GPU parity of multi-k cumulative calibration (topt_calibrate_multik) against
the float64 oracle of App. D, Algorithm 2 and Eq. 8.

Small shapes are compared whole; the prefill-calibration shape of the
LLaMA-3-8B workload (32/8 heads, d = 128, 8 sequences of 4096 rows) on sampled
(head, row length) groups the oracle merges one by one.  Edge cases: repeated
and missing row lengths, targets k at and above the row length, one sequence
(Algorithm 1 with alpha = 0), bad device-side lengths and oversized groups.
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


def _seqs(seed, N, Hq, Hkv, d, S, dtype):
    Qs, Ks = [], []
    for n in range(N):
        Q, K, _ = prefill_case(seed * 1000 + n, 1, Hq, Hkv, d, S, dtype)
        Qs.append(Q)
        Ks.append(K)
    return torch.cat(Qs).contiguous(), torch.cat(Ks).contiguous()


TOL = 1e-4   # relative: theta is one calibration score, an fp32 dot product of d terms


def _tol(want, mode):
    # the same bound as the Algorithm 1 calibration parity; softmax values add
    # one expf and one division
    return TOL * (np.abs(want) + (1e-6 if mode == ref.PRE else 0.0))


def _compare(got, want, mode, what):
    assert np.array_equal(np.isneginf(got), np.isneginf(want)), what
    fin = np.isfinite(want)
    err = np.abs(got[fin] - want[fin])
    tol = _tol(want[fin], mode)
    bad = np.flatnonzero(err > tol)
    assert bad.size == 0, (what, bad.size, float(np.max(err / tol)))


@pytest.mark.parametrize("mode", [ref.PRE, ref.POST])
@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16)])
def test_mkc_prefill_rows_match_oracle(mode, d, dtype):
    N, Hq, Hkv, S, Lmax = 3, 4, 2, 96, 112
    ks = [1, 2, 5, 17, 95, 96, 200]
    Q, K = _seqs(21, N, Hq, Hkv, d, S, dtype)
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    theta = topt.calibrate_multik(Q, K, row_len, torch.tensor(ks, dtype=torch.int32, device="cuda"),
                                  mode, Lmax, status=status)
    assert int(status.item()) == 0
    want, _ = ref.mkc_ref(synth.as_f64(Q), synth.as_f64(K), np.arange(1, S + 1), mode, ks, (Hq, Lmax))
    _compare(theta.cpu().double().numpy(), want, mode, "prefill rows")


@pytest.mark.parametrize("mode", [ref.PRE, ref.POST])
def test_mkc_repeated_and_missing_lengths(mode):
    """Decode-style rows: several rows share a length, most lengths are absent,
    the table runs past the longest row; an explicit small workspace forces one
    head per pass."""
    N, Hq, Hkv, d, Nk, Lmax = 3, 4, 1, 64, 40, 48
    lens = [5, 9, 9, 33, 33, 33, 40, 2]
    ks = [1, 3, 8, 9, 32, 39, 4]
    gen = synth.generator(77, "cuda")
    K = synth.iid_normal(gen, (N, Hkv, Nk, d), "cuda", torch.bfloat16)
    Q = synth.iid_normal(gen, (N, Hq, len(lens), d), "cuda", torch.bfloat16)
    row_len = torch.tensor(lens, device="cuda", dtype=torch.int32)
    kt = torch.tensor(ks, dtype=torch.int32, device="cuda")
    fixed = 3 * 256 + 256 + ((len(ks) * Hq * Lmax * 4 + 255) // 256) * 256
    per_head = ((N * len(lens) * Nk * 4 + 255) // 256) * 256
    ws = torch.empty(fixed + per_head + 100, device="cuda", dtype=torch.uint8)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    theta = topt.calibrate_multik(Q, K, row_len, kt, mode, Lmax, status=status, workspace=ws)
    assert int(status.item()) == 0
    want, _ = ref.mkc_ref(synth.as_f64(Q), synth.as_f64(K), lens, mode, ks, (Hq, Lmax))
    _compare(theta.cpu().double().numpy(), want, mode, "decode rows")
    # the same call with room for every head at once gives the same tables
    again = topt.calibrate_multik(Q, K, row_len, kt, mode, Lmax)
    assert torch.equal(again, theta)


def test_mkc_one_sequence_equals_algorithm1():
    """N = 1: theta(k) is the k-th largest score of each row, bit for bit what
    topt_calibrate gives with alpha = 0 on the same scores."""
    Hq, Hkv, d, S, Lmax = 4, 2, 128, 200, 200
    Q, K = _seqs(31, 1, Hq, Hkv, d, S, torch.bfloat16)
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    ks = [1, 4, 64, 150]
    theta = topt.calibrate_multik(Q, K, row_len, torch.tensor(ks, dtype=torch.int32, device="cuda"),
                                  ref.PRE, Lmax)
    for ki, k in enumerate(ks):
        cal = topt.Calibrator(Hq, Lmax, k, ref.PRE, 0.0)
        cal.add(Q, K, row_len, reset=True)
        a1 = cal.finalize()
        assert torch.equal(theta[ki], a1), k


def test_mkc_bad_lengths_and_oversized_groups_set_status():
    Hq, Hkv, d, Nk, Lmax = 2, 1, 64, 16, 16
    gen = synth.generator(5, "cuda")
    K = synth.iid_normal(gen, (1, Hkv, Nk, d), "cuda", torch.float32)
    Q = synth.iid_normal(gen, (1, Hq, 3, d), "cuda", torch.float32)
    ks = torch.tensor([2], dtype=torch.int32, device="cuda")
    for bad in ([4, 0, 7], [4, 17, 7], [4, 5, -1]):
        status = torch.zeros(1, device="cuda", dtype=torch.int32)
        topt.calibrate_multik(Q, K, torch.tensor(bad, device="cuda", dtype=torch.int32), ks,
                              ref.PRE, Lmax, status=status)
        assert int(status.item()) == 1, bad                      # TOPT_EINVAL
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    topt.calibrate_multik(Q, K, torch.tensor([4, 5, 7], device="cuda", dtype=torch.int32),
                          torch.tensor([2, 0], dtype=torch.int32, device="cuda"), ref.PRE, Lmax,
                          status=status)
    assert int(status.item()) == 1                               # k = 0
    # 4097 rows of one length in one head: more than one CTA's event arrays
    R = 4097
    Q2 = synth.iid_normal(gen, (1, 1, R, d), "cuda", torch.float32)
    K2 = synth.iid_normal(gen, (1, 1, 4, d), "cuda", torch.float32)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    topt.calibrate_multik(Q2, K2, torch.full((R,), 4, device="cuda", dtype=torch.int32), ks,
                          ref.PRE, 4, status=status)
    assert int(status.item()) == 1
    # 4096 rows is the limit and works
    status.zero_()
    th = topt.calibrate_multik(Q2[:, :, :4096].contiguous(), K2,
                               torch.full((4096,), 4, device="cuda", dtype=torch.int32), ks,
                               ref.PRE, 4, status=status)
    assert int(status.item()) == 0
    rows = synth.as_f64(Q2)[0, 0, :4096] @ synth.as_f64(K2)[0, 0].T / np.sqrt(d)
    pieces = ref.merge_intervals([ref.mkc_interval_sequence(r) for r in rows])
    want = ref.mkc_theta(pieces, 2)
    got = float(th[0, 0, 3])
    assert abs(got - want) <= TOL * (abs(want) + 1e-6), (got, want)


def test_mkc_llama3_8b_calibration_shape_sampled():
    """32/8 heads, d = 128, 8 causal sequences of 4096 rows, bf16, five targets;
    sampled (head, length) groups merged by the oracle one by one."""
    N, Hq, Hkv, d, S = 8, 32, 8, 128, 4096
    ks = [16, 64, 128, 512, 4095]
    Q, K = _seqs(41, N, Hq, Hkv, d, S, torch.bfloat16)
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    for mode in (ref.PRE, ref.POST):
        theta = topt.calibrate_multik(Q, K, row_len, torch.tensor(ks, dtype=torch.int32, device="cuda"),
                                      mode, S, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        th = theta.cpu().double().numpy()
        # dense rows, every longer row calibrated, non-increasing in k
        for ki, k in enumerate(ks):
            assert np.all(np.isneginf(th[ki, :, :k]))
            assert np.all(np.isfinite(th[ki, :, k:]))
            if ki:
                assert np.all(th[ki, :, k:] <= th[ki - 1, :, k:])
        for h, L in ((0, 65), (13, 1000), (31, 4096), (7, 129), (22, 2048)):
            g = h // (Hq // Hkv)
            rows = []
            for n in range(N):
                a = ref.row_scores(synth.as_f64(Q[n, h, L - 1]), synth.as_f64(K[n, g]), L)
                rows.append(a if mode == ref.PRE else ref.row_softmax(a))
            pieces = ref.merge_intervals([ref.mkc_interval_sequence(r) for r in rows])
            for ki, k in enumerate(ks):
                want = ref.mkc_theta(pieces, k) if L > k else -np.inf
                got = th[ki, h, L - 1]
                if np.isneginf(want):
                    assert np.isneginf(got), (mode, h, L, k)
                    continue
                assert abs(got - want) <= TOL * (abs(want) + (1e-6 if mode == ref.PRE else 0)), \
                    (mode, h, L, k, got, want)
