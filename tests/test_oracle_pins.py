"""Pins of the float64 oracle to facts the pages and the mathematics fix.

Each check compares the oracle with something other than itself: hand-derived
closed forms (tests/golden), a library attention routine, brute force on tiny
rows, and identities of the method (Eq. 4, Eq. 5-7).  The last test plants
mistakes in the oracle and checks that these pins catch each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.topt_ref as ref

MODES = {"pre": ref.PRE, "post": ref.POST}
SDCS = {"none": ref.SDC_NONE, "exact": ref.SDC_EXACT, "expth": ref.SDC_EXPTH}


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Dense limit: theta = -inf is ordinary softmax attention (Eq. 1-3).
# ---------------------------------------------------------------------------
def _sdpa(q, k, v, mask=None, causal=False):
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.as_tensor(q), torch.as_tensor(k), torch.as_tensor(v),
        attn_mask=None if mask is None else torch.as_tensor(mask), is_causal=causal)
    return out.numpy()


def check_dense_decode(seed=0):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, d, Nmax = 2, 4, 2, 16, 23
    seq_len = np.array([23, 9])
    q = rng.standard_normal((B, Hq, d))
    Kc = rng.standard_normal((B, Hkv, Nmax, d)) * 2
    Vc = rng.standard_normal((B, Hkv, Nmax, d))
    theta = np.full((Hq, Nmax), -np.inf)
    for mode in (ref.PRE, ref.POST):
        res, vrows = ref.decode_ref(q, Kc, Vc, seq_len, theta, mode)
        g = Hq // Hkv
        Kr = np.repeat(Kc, g, axis=1)
        Vr = np.repeat(Vc, g, axis=1)
        mask = np.zeros((B, 1, 1, Nmax), dtype=bool)
        for b in range(B):
            mask[b, 0, 0, :seq_len[b]] = True
        want = _sdpa(q[:, :, None, :], Kr, Vr, mask)[:, :, 0, :]
        for (b, h), r in res.items():
            assert r["kept"] == seq_len[b]
            np.testing.assert_allclose(r["out"], want[b, h], rtol=1e-12, atol=1e-12)
        for (b, kv), n in vrows.items():
            assert n == seq_len[b]


def test_dense_decode_matches_library_sdpa():
    check_dense_decode()


def check_dense_prefill(seed=1):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, S, d = 1, 2, 1, 19, 8
    Q = rng.standard_normal((B, Hq, S, d))
    K = rng.standard_normal((B, Hkv, S, d))
    V = rng.standard_normal((B, Hkv, S, d))
    theta = np.full((Hq, S), -np.inf)
    want = _sdpa(Q, np.repeat(K, 2, axis=1), np.repeat(V, 2, axis=1), causal=True)
    for mode, sdc, vmc in [(ref.PRE, ref.SDC_NONE, False), (ref.POST, ref.SDC_NONE, True),
                           (ref.PRE, ref.SDC_EXACT, True), (ref.PRE, ref.SDC_EXPTH, True)]:
        res = ref.prefill_ref(Q, K, V, theta, mode, sdc, vmc)
        for (b, h, i), r in res.items():
            assert r["kept"] == i + 1
            assert abs(r["beta"]) < 1e-12          # full mask: nothing discarded
            np.testing.assert_allclose(r["out"], want[b, h, i], rtol=1e-12, atol=1e-12)


def test_dense_prefill_matches_library_causal_sdpa():
    check_dense_prefill()


# ---------------------------------------------------------------------------
# Hand-derived closed forms of Eq. 4-7 (tests/golden/sdc_vmc_five_keys.json).
# ---------------------------------------------------------------------------
def check_golden_sdc_vmc(golden_dir):
    g = _load(golden_dir, "sdc_vmc_five_keys.json")
    a = np.array(g["a"])
    V = np.eye(5)
    mu = ref.vmean_ref(V)
    np.testing.assert_allclose(mu, 0.2, rtol=1e-15)
    for c in g["cases"]:
        r = ref.attend_row(a, V, c["theta"], MODES[c["mode"]], SDCS[c["sdc"]], c["vmc"], mu)
        assert r["kept"] == c["kept"], c
        assert abs(r["beta"] - c["beta"]) < 1e-14, c
        np.testing.assert_allclose(r["out"], c["out"], rtol=1e-13, atol=1e-15, err_msg=str(c))


def test_golden_sdc_vmc_closed_forms(golden_dir):
    check_golden_sdc_vmc(golden_dir)


# ---------------------------------------------------------------------------
# Algorithm 1 by hand (tests/golden/calibration_two_samples.json).
# ---------------------------------------------------------------------------
def check_golden_calibration(golden_dir):
    g = _load(golden_dir, "calibration_two_samples.json")
    d, k, L, Lmax = g["d"], g["k"], g["L"], g["Lmax"]
    S = g["sample_scores"]
    N = len(S)
    Qc = np.zeros((N, 1, 1, d))
    Kc = np.zeros((N, 1, L, d))
    for n in range(N):
        Qc[n, 0, 0] = g["q"]
        Kc[n, 0, :, 0] = S[n]
    for e in g["expect"]:
        theta, sets = ref.calibrate_ref(Qc, Kc, [L], k, MODES[e["mode"]], e["alpha"], Lmax)
        assert len(sets[(0, L)]) == N
        assert abs(theta[0, L - 1] - e["theta"]) < 1e-14, e
        for LL in range(1, Lmax + 1):
            want = -np.inf if LL <= k else e["theta"]
            assert theta[0, LL - 1] == pytest.approx(want, abs=1e-14), (e, LL)


def test_golden_two_sample_calibration(golden_dir):
    check_golden_calibration(golden_dir)


def check_golden_nearest_row(golden_dir):
    g = _load(golden_dir, "nearest_row.json")
    d, k, Lmax = g["d"], g["k"], g["Lmax"]
    Nk = len(g["K_col0"])
    Qc = np.zeros((1, 1, 2, d))
    Qc[0, 0, 0] = g["q"][0]
    Qc[0, 0, 1] = g["q"][1]
    Kc = np.zeros((1, 1, Nk, d))
    Kc[0, 0, :, 0] = g["K_col0"]
    Kc[0, 0, :, 1] = g["K_col1"]
    theta, _ = ref.calibrate_ref(Qc, Kc, g["row_len"], k, ref.PRE, 0.0, Lmax)
    want = np.array([float(x) for x in g["theta"]])
    np.testing.assert_array_equal(np.isinf(theta[0]), np.isinf(want))
    fin = np.isfinite(want)
    np.testing.assert_allclose(theta[0][fin], want[fin], rtol=0, atol=1e-15)
    # beyond the table: the last entry is used
    assert ref.theta_for_row(theta[0], 10 * Lmax) == want[-1]


def test_golden_nearest_calibrated_row(golden_dir):
    check_golden_nearest_row(golden_dir)


# ---------------------------------------------------------------------------
# Brute force on rows of 4-16 elements: a threshold calibrated on one row and
# applied to the same row keeps exactly that row's top-k.
# ---------------------------------------------------------------------------
def check_bruteforce_topk(seed=2, trials=300):
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        L = int(rng.integers(4, 17))
        k = int(rng.integers(1, L))
        d = 4
        vals = rng.permutation(L).astype(np.float64) * 0.37 - 1.1   # distinct
        Qc = np.zeros((1, 1, 1, d))
        Qc[0, 0, 0, 0] = 2.0                                        # a_j = K[j][0]
        Kc = np.zeros((1, 1, L, d))
        Kc[0, 0, :, 0] = vals
        want = set(sorted(range(L), key=lambda j: -vals[j])[:k])
        for mode in (ref.PRE, ref.POST):
            theta, _ = ref.calibrate_ref(Qc, Kc, [L], k, mode, 0.0, L)
            th = ref.theta_for_row(theta[0], L)
            a = ref.row_scores(Qc[0, 0, 0], Kc[0, 0], L)
            np.testing.assert_allclose(a, vals, rtol=0, atol=0)
            r = ref.attend_row(a, np.eye(L), th, mode)
            assert set(np.flatnonzero(r["keep"])) == want, (L, k, mode)
            assert r["kept"] == k


def test_bruteforce_calibrated_row_selects_topk():
    check_bruteforce_topk()


def test_bruteforce_kth_largest_all_orders():
    # every permutation of a 5-element row with a repeated value
    base = [3.0, -1.0, 2.0, 2.0, 0.5]
    for perm in itertools.permutations(base):
        srt = sorted(perm, reverse=True)
        for k in range(1, 6):
            assert ref.kth_largest(np.array(perm), k) == srt[k - 1]


def test_ties_are_all_kept():
    a = np.array([1.0, 3.0, 2.0, 2.0, 2.0, 0.0])
    k = 2
    th = ref.kth_largest(a, k)                 # = 2.0, shared by three keys
    r = ref.attend_row(a, np.eye(6), th, ref.PRE)
    assert r["kept"] == 4 and r["kept"] >= k
    assert list(np.flatnonzero(r["keep"])) == [1, 2, 3, 4]


def test_short_rows_are_dense():
    rng = np.random.default_rng(3)
    d, k, S = 8, 6, 12
    Qc = rng.standard_normal((3, 1, S, d))
    Kc = rng.standard_normal((3, 1, S, d))
    theta, sets = ref.calibrate_ref(Qc, Kc, np.arange(1, S + 1), k, ref.PRE, 0.0, S)
    assert all(L > k for (_, L) in sets)
    assert np.all(np.isneginf(theta[0, :k])) and np.all(np.isfinite(theta[0, k:]))


# ---------------------------------------------------------------------------
# Identities of the method.
# ---------------------------------------------------------------------------
def check_sdc_exact_equals_post(seed=4, trials=50):
    """Eq. 4: for one kept set, pre-softmax + exact SDC equals post-softmax."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        L = int(rng.integers(2, 40))
        d = 6
        a = rng.standard_normal(L) * 3
        V = rng.standard_normal((L, d))
        mu = ref.vmean_ref(V)
        k = int(rng.integers(1, L + 1))
        th_pre = ref.kth_largest(a, k)
        th_post = ref.kth_largest(ref.row_softmax(a), k)
        for vmc in (False, True):
            p = ref.attend_row(a, V, th_pre, ref.PRE, ref.SDC_EXACT, vmc, mu)
            q = ref.attend_row(a, V, th_post, ref.POST, ref.SDC_NONE, vmc, mu)
            assert np.array_equal(p["keep"], q["keep"])
            np.testing.assert_allclose(p["out"], q["out"], rtol=1e-12, atol=1e-13)
            assert abs(p["beta"] - q["beta"]) < 1e-13
            # the discarded mass of post-softmax is E/Z
            assert abs(q["beta"] - q["E"] / q["Z"]) < 1e-13


def test_sdc_exact_pre_equals_post_softmax():
    check_sdc_exact_equals_post()


def check_vmc_constant_values(seed=5, trials=40):
    """Eq. 5-7: if every V row equals v, the compensated output is v for any mask."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        L = int(rng.integers(1, 30))
        v = rng.standard_normal(5)
        V = np.tile(v, (L, 1))
        a = rng.standard_normal(L) * 2
        mu = ref.vmean_ref(V)
        th_pre = float(rng.normal(0, 2))
        th_post = float(rng.uniform(0, 0.6))
        cases = [(ref.POST, ref.SDC_NONE, th_post), (ref.PRE, ref.SDC_EXACT, th_pre),
                 (ref.PRE, ref.SDC_EXPTH, th_pre)]
        for mode, sdc, th in cases:
            r = ref.attend_row(a, V, th, mode, sdc, True, mu)
            np.testing.assert_allclose(r["out"], v, rtol=1e-12, atol=1e-12)
        r = ref.attend_row(a, V, th_pre, ref.PRE, ref.SDC_NONE, True, mu)
        want = v if r["kept"] else np.zeros(5)
        np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)


def test_vmc_constant_value_rows_give_that_row():
    check_vmc_constant_values()


def test_exp_threshold_is_zero_on_a_dense_row():
    a = np.array([0.3, -0.2, 1.5])
    V = np.arange(9.0).reshape(3, 3)
    d = ref.attend_row(a, V, -np.inf, ref.PRE, ref.SDC_NONE)
    e = ref.attend_row(a, V, -np.inf, ref.PRE, ref.SDC_EXPTH, True, ref.vmean_ref(V))
    np.testing.assert_allclose(e["out"], d["out"], rtol=1e-14)
    assert abs(e["beta"]) < 1e-15


def test_running_mean_equals_batch_mean():
    rng = np.random.default_rng(6)
    V = rng.standard_normal((257, 7))
    mu = np.zeros(7)
    n = 0
    for i in range(40):                         # one row at a time (decode)
        mu = ref.vmean_update_ref(mu, n, V[i:i + 1])
        n += 1
    for lo, hi in [(40, 41), (41, 100), (100, 257)]:   # chunks (prefill)
        mu = ref.vmean_update_ref(mu, n, V[lo:hi])
        n = hi
    np.testing.assert_allclose(mu, V.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_tile_counts_match_bruteforce():
    rng = np.random.default_rng(7)
    for S, tm, tn in [(10, 4, 3), (17, 8, 8), (33, 16, 8)]:
        keep = {i: rng.random(i + 1) < 0.1 for i in range(S)}
        hit, total = ref.tile_counts_ref(keep, S, tm, tn)
        tiles = {}
        for i in range(S):
            for j in range(i + 1):
                key = (i // tm, j // tn)
                tiles[key] = tiles.get(key, False) or bool(keep[i][j])
        assert total == len(tiles)
        assert hit == sum(tiles.values())


def test_output_error_metric():
    assert ref.output_rel_error([1.0, 2.0], [1.0, 2.0]) == 0.0
    assert ref.output_rel_error([1.0, 2.002], [1.0, 2.0]) == pytest.approx(1e-3)


# ---------------------------------------------------------------------------
# Offline-calibrated SDC (§3.2.1 estimator 1) by hand and by identities.
# ---------------------------------------------------------------------------
def check_golden_offline_sdc(golden_dir):
    g = _load(golden_dir, "sdc_offline_two_samples.json")
    d, k, L, Lmax = g["d"], g["k"], g["L"], g["Lmax"]
    S = g["sample_scores"]
    Qc = np.zeros((len(S), 1, 1, d))
    Kc = np.zeros((len(S), 1, L, d))
    for n in range(len(S)):
        Qc[n, 0, 0] = g["q"]
        Kc[n, 0, :, 0] = S[n]
    theta, _ = ref.calibrate_ref(Qc, Kc, [L], k, ref.PRE, 0.0, Lmax)
    et, sets = ref.calibrate_discarded_ref(Qc, Kc, [L], theta)
    assert len(sets[(0, L)]) == len(S)
    np.testing.assert_allclose(et[0], g["e_tilde"], rtol=1e-14, atol=1e-15)
    a = ref.row_scores(Qc[0, 0, 0], Kc[0, 0], L)
    r = ref.attend_row(a, np.eye(L), ref.theta_for_row(theta[0], L), ref.PRE, ref.SDC_OFFLINE,
                       e_tilde=ref.theta_for_row(et[0], L))
    np.testing.assert_allclose(r["out"], g["row1_out"], rtol=1e-14, atol=1e-15)
    assert abs(r["beta"] - g["row1_beta"]) < 1e-14


def test_golden_offline_sdc(golden_dir):
    check_golden_offline_sdc(golden_dir)


def test_offline_sdc_identities():
    """E~ = the row's own E is exact SDC; E~ = 0 is plain pre-softmax."""
    rng = np.random.default_rng(8)
    for _ in range(200):
        L = int(rng.integers(2, 20))
        a = rng.normal(size=L) * 2
        V = rng.normal(size=(L, 5))
        mu = V.mean(axis=0)
        th = float(np.sort(a)[rng.integers(0, L)])
        ex = ref.attend_row(a, V, th, ref.PRE, ref.SDC_EXACT, True, mu)
        off = ref.attend_row(a, V, th, ref.PRE, ref.SDC_OFFLINE, True, mu, e_tilde=ex["E"])
        np.testing.assert_allclose(off["out"], ex["out"], rtol=1e-13, atol=1e-15)
        assert abs(off["beta"] - ex["beta"]) < 1e-13
        none = ref.attend_row(a, V, th, ref.PRE, ref.SDC_NONE, True, mu)
        zero = ref.attend_row(a, V, th, ref.PRE, ref.SDC_OFFLINE, True, mu, e_tilde=0.0)
        np.testing.assert_allclose(zero["out"], none["out"], rtol=1e-13, atol=1e-15)
        assert none["beta"] == 0.0 and abs(zero["beta"]) < 1e-13


def test_offline_sdc_one_row_calibration_is_exact_on_that_row():
    """E~ calibrated on one decode row, applied to the same row, reproduces
    exact SDC: the only sample is that row's own E."""
    rng = np.random.default_rng(9)
    for _ in range(50):
        L, d = int(rng.integers(4, 30)), 8
        k = int(rng.integers(1, L))
        Kc = rng.normal(size=(1, 1, L, d))
        q = rng.normal(size=(1, 1, d)) * 2
        V = rng.normal(size=(1, 1, L, d))
        theta, _ = ref.calibrate_ref(q[:, :, None, :], Kc, [L], k, ref.PRE, 0.0, L)
        et, _ = ref.calibrate_discarded_ref(q[:, :, None, :], Kc, [L], theta)
        ex, _ = ref.decode_ref(q, Kc, V, [L], theta, ref.PRE, ref.SDC_EXACT, True, V.mean(axis=2))
        off, _ = ref.decode_ref(q, Kc, V, [L], theta, ref.PRE, ref.SDC_OFFLINE, True, V.mean(axis=2),
                                e_tilde=et)
        np.testing.assert_allclose(off[(0, 0)]["out"], ex[(0, 0)]["out"], rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Fitted theta(L) (reading c22): exact recovery of lines in ln L.
# ---------------------------------------------------------------------------
def check_fitted_theta():
    k, Lmax = 3, 200
    c = (0.7, 0.45)
    f = lambda L: c[0] + c[1] * math.log(L)
    # one calibration row per length, its k-th largest score set to f(L)
    for L in (5, 9, 17, 33, 64, 90):
        row = np.concatenate([f(L) + 1.0 + np.arange(k - 1), [f(L)], f(L) - 1.0 - np.arange(L - k)])
        Qc, Kc = _mkc_inputs([row])
        th, _ = ref.calibrate_ref(Qc, Kc, [L], k, ref.PRE, 0.0, Lmax, fit=False)
        assert th[0, L - 1] == f(L)
    sets = {(0, L): [f(L)] for L in (5, 9, 17, 33, 64, 90)}
    theta = ref.finalize_fitted(sets, 1, Lmax, k, 0.0, ref.PRE)
    want = np.array([f(L) for L in range(1, Lmax + 1)])
    assert np.all(np.isneginf(theta[0, :k]))
    np.testing.assert_allclose(theta[0, k:], want[k:], rtol=0, atol=1e-12)
    # end to end through Algorithm 1 on the rows built above
    Ls = (5, 9, 17, 33)
    rows = [np.concatenate([f(L) + 1.0 + np.arange(k - 1), [f(L)], f(L) - 1.0 - np.arange(L - k)])
            for L in Ls]
    Nk = max(Ls)
    # each row sees its own keys: put row i at keys 0..L_i-1 of its own sequence
    Qs = np.zeros((len(Ls), 1, 1, 4))
    Ks = np.zeros((len(Ls), 1, Nk, 4))
    for i, (L, r) in enumerate(zip(Ls, rows)):
        Qs[i, 0, 0, 0] = 2.0
        Ks[i, 0, :L, 0] = r
    sets = {}
    for i, L in enumerate(Ls):
        ref.collect_thresholds(Qs[i:i + 1], Ks[i:i + 1], [L], k, ref.PRE, sets)
    th = ref.finalize_fitted(sets, 1, 120, k, 0.0, ref.PRE)
    np.testing.assert_allclose(th[0, k:], want[k:120], rtol=0, atol=1e-12)
    # post-softmax: a power law in L is a line in ln L after the log; rows
    # shorter than the shortest calibrated one would extrapolate above every
    # calibrated value and stay at the largest one instead
    sets = {(0, L): [0.3 * L ** -1.2] for L in (6, 20, 70)}
    th = ref.finalize_fitted(sets, 1, Lmax, k, 0.0, ref.POST)
    Lr = np.arange(6, Lmax + 1)
    np.testing.assert_allclose(th[0, 5:], 0.3 * Lr ** -1.2, rtol=1e-12, atol=0)
    assert np.all(th[0, k:5] == 0.3 * 6 ** -1.2)
    # an extrapolated probability threshold never reaches 1 (the row would keep
    # nothing) nor falls to 0 (it would keep everything)
    th = ref.finalize_fitted({(0, 10): [0.9], (0, 40): [0.5]}, 1, 60, k, 0.0, ref.POST)
    assert th[0, 3] == 0.9 and 0.5 < th[0, 19] < 0.9      # L = 4 extrapolates to 1.33
    th = ref.finalize_fitted({(0, 10): [1e-30], (0, 20): [1e-36]}, 1, 400, k, 0.0, ref.POST)
    assert th[0, 399] == 2.0 ** -126 and abs(th[0, 9] - 1e-30) < 1e-12 * 1e-30
    # two calibrated lengths: the line through both points in ln L
    th = ref.finalize_fitted({(0, 10): [1.0], (0, 40): [2.0]}, 1, 80, k, 0.0, ref.PRE)
    assert abs(th[0, 9] - 1.0) < 1e-13 and abs(th[0, 39] - 2.0) < 1e-13
    assert abs(th[0, 19] - 1.5) < 1e-13              # ln 20 is halfway between ln 10 and ln 40
    # one length: a constant; none: dense
    th = ref.finalize_fitted({(0, 10): [1.5]}, 1, 30, k, 0.0, ref.PRE)
    assert np.all(th[0, k:] == 1.5)
    assert np.all(np.isneginf(ref.finalize_fitted({}, 1, 30, k, 0.0, ref.PRE)))


def test_fitted_theta_recovers_lines_in_log_length():
    check_fitted_theta()


# ---------------------------------------------------------------------------
# GQA group policies (§4.6): set invariants against the heads' own decisions.
# ---------------------------------------------------------------------------
def _gqa_case(seed, same_q=False):
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, d, Nmax = 2, 8, 2, 16, 40
    K = rng.normal(size=(B, Hkv, Nmax, d))
    V = rng.normal(size=(B, Hkv, Nmax, d))
    q = rng.normal(size=(B, Hq, d)) * 2
    if same_q:
        q[:, 1:4] = q[:, :1]
        q[:, 5:8] = q[:, 4:5]
    seq = [40, 23]
    theta = rng.normal(size=(Hq, Nmax)) * 0.5 + 0.8
    if same_q:                    # identical heads: same query and same thresholds
        theta[1:4] = theta[:1]
        theta[5:8] = theta[4:5]
    mu = V.mean(axis=2)
    return q, K, V, seq, theta, mu


def check_gqa_policies(seed=10):
    g = 4
    for same_q in (False, True):
        q, K, V, seq, theta, mu = _gqa_case(seed, same_q)
        for mode, sdc in ((ref.PRE, ref.SDC_NONE), (ref.PRE, ref.SDC_EXACT), (ref.POST, ref.SDC_NONE)):
            own, v_own = ref.decode_ref(q, K, V, seq, theta, mode, sdc, True, mu)
            uni, v_uni = ref.decode_ref(q, K, V, seq, theta, mode, sdc, True, mu, gqa=ref.GQA_UNION)
            assert v_uni == v_own                       # the union reads the same V rows
            for (b, h), r in own.items():
                grp = np.any([own[(b, (h // g) * g + i)]["keep"] for i in range(g)], axis=0)
                assert np.array_equal(uni[(b, h)]["keep"], grp)
                assert np.all(uni[(b, h)]["keep"] >= r["keep"])
                if same_q:                              # identical heads: the union is each own set
                    np.testing.assert_allclose(uni[(b, h)]["out"], r["out"], rtol=1e-13, atol=1e-15)
            one, v_one = ref.decode_ref(q, K, V, seq, theta, mode, sdc, True, mu, gqa=ref.GQA_VOTE,
                                        gqa_min_heads=1)
            assert v_one == v_own
            for key in own:
                np.testing.assert_allclose(one[key]["out"], own[key]["out"], rtol=1e-13, atol=1e-15)
            prev = one
            for t in range(2, g + 2):
                vt, v_vt = ref.decode_ref(q, K, V, seq, theta, mode, sdc, True, mu, gqa=ref.GQA_VOTE,
                                          gqa_min_heads=t)
                for (b, kv), n in v_vt.items():
                    votes = np.zeros(seq[b], dtype=int)
                    for i in range(g):
                        votes += own[(b, kv * g + i)]["keep"]
                    assert n == int((votes >= t).sum())  # brute-force vote count
                for key, r in vt.items():
                    assert np.all(r["keep"] <= prev[key]["keep"])
                    assert np.all(r["keep"] <= own[key]["keep"])
                    if t > g:
                        assert r["kept"] == 0
                prev = vt


def test_gqa_policies_invariants():
    check_gqa_policies()


# ---------------------------------------------------------------------------
# Multi-k cumulative calibration (App. D, Algorithm 2, Eq. 8).
# ---------------------------------------------------------------------------
def _mkc_inputs(rows, d=4):
    """Calibration tensors whose scores are exactly ``rows`` (a_j = K[j][0])."""
    N, L = len(rows), len(rows[0])
    Qc = np.zeros((N, 1, 1, d))
    Qc[:, 0, 0, 0] = 2.0
    Kc = np.zeros((N, 1, L, d))
    for n in range(N):
        Kc[n, 0, :, 0] = rows[n]
    return Qc, Kc


def check_golden_mkc(golden_dir):
    g = _load(golden_dir, "mkc_two_rows.json")
    L, Lmax, ks = g["L"], g["Lmax"], g["ks"]
    Qc, Kc = _mkc_inputs(g["sample_scores"], g["d"])
    sets = ref.mkc_collect(Qc, Kc, [L], ref.PRE)
    pieces = ref.merge_intervals(sets[(0, L)])
    assert [list(p) for p in pieces] == g["pieces_pre"]
    for mode, key in ((ref.PRE, "theta_pre"), (ref.POST, "theta_post")):
        theta, _ = ref.mkc_ref(Qc, Kc, [L], mode, ks, (1, Lmax))
        for ki, k in enumerate(ks):
            t = float(g[key][ki])
            want = [-np.inf if (LL <= k or not np.isfinite(t)) else t for LL in range(1, Lmax + 1)]
            np.testing.assert_allclose(theta[ki, 0], want, rtol=1e-14, atol=0, err_msg=f"{key} k={k}")


def test_golden_mkc_two_rows(golden_dir):
    check_golden_mkc(golden_dir)


def check_mkc_single_row(seed=5, trials=200):
    """One calibration row: theta(k) is its k-th largest element, which is also
    what Algorithm 1 gives with alpha = 0 (one sample, no spread)."""
    rng = np.random.default_rng(seed)
    for t in range(trials):
        L = int(rng.integers(2, 14))
        if t % 2:
            row = rng.integers(0, 4, L).astype(np.float64)        # ties
        else:
            row = rng.normal(size=L)
        srt = sorted(row, reverse=True)
        pieces = ref.merge_intervals([ref.mkc_interval_sequence(row)])
        for k in range(1, L + 1):
            # no interval starts below the row minimum, so a k-th largest that
            # equals the minimum (ties at the bottom, or k = L) gives no theta
            want = srt[k - 1] if srt[k - 1] > srt[-1] else -np.inf
            assert ref.mkc_theta(pieces, k) == want, (row, k)
        Qc, Kc = _mkc_inputs([row])
        ks = list(range(1, L))
        th, _ = ref.mkc_ref(Qc, Kc, [L], ref.POST, ks, (1, L + 2))
        for ki, k in enumerate(ks):
            if srt[k - 1] == srt[-1]:
                continue
            a1, _ = ref.calibrate_ref(Qc, Kc, [L], k, ref.POST, 0.0, L + 2)
            np.testing.assert_allclose(th[ki], a1, rtol=1e-15, atol=0)


def test_mkc_single_row_is_kth_largest():
    check_mkc_single_row()


def _kbar_direct(rows, theta):
    """Eq. 8 by counting: mean over the rows whose [min, max) holds theta of the
    number of their elements above theta; None where no row holds theta."""
    cnt = [int(np.sum(r > theta)) for r in rows if r.min() <= theta < r.max()]
    return None if not cnt else sum(cnt) / len(cnt)


def check_mkc_bruteforce(seed=6, trials=300):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        N, L = int(rng.integers(1, 6)), int(rng.integers(2, 9))
        if t % 3 == 0:
            rows = [rng.integers(0, 5, L).astype(np.float64) for _ in range(N)]
        else:
            rows = [rng.normal(size=L) * rng.uniform(0.2, 3) + rng.normal() for _ in range(N)]
        pooled = np.unique(np.concatenate(rows))
        pieces = ref.merge_intervals([ref.mkc_interval_sequence(r) for r in rows])
        for k in range(1, L + 1):
            th = ref.mkc_theta(pieces, k)
            for y in pooled[pooled >= th]:
                kb = _kbar_direct(rows, y)
                assert kb is None or kb < k, (rows, k, th, y)
            if np.isfinite(th):
                assert th in pooled
                below = pooled[pooled < th]
                kb = _kbar_direct(rows, below[-1])
                assert kb is not None and kb >= k, (rows, k, th)
            else:
                for y in pooled:
                    kb = _kbar_direct(rows, y)
                    assert kb is None or kb < k
        ths = [ref.mkc_theta(pieces, k) for k in range(1, L + 1)]
        assert all(a >= b for a, b in zip(ths, ths[1:]))          # non-increasing in k


def test_mkc_bruteforce_sup_of_kbar():
    check_mkc_bruteforce()


def test_mkc_rows_spanning_theta_give_pooled_order_statistic():
    """When every row holds theta in its [min, max), Eq. 8 is the pooled count
    over N rows, so theta(k) is the (k N)-th largest pooled element."""
    rng = np.random.default_rng(7)
    for _ in range(100):
        N, L = int(rng.integers(1, 7)), int(rng.integers(4, 12))
        rows = [np.concatenate([[50.0 + n], rng.normal(size=L - 2), [-50.0 - n]]) for n in range(N)]
        pooled = np.sort(np.concatenate(rows))[::-1]
        pieces = ref.merge_intervals([ref.mkc_interval_sequence(r) for r in rows])
        for k in range(2, L - 1):
            assert ref.mkc_theta(pieces, k) == pooled[k * N - 1], (N, L, k)


# ---------------------------------------------------------------------------
# The pins above catch plausible mistakes in the oracle.
# ---------------------------------------------------------------------------
def _planted(monkeypatch, name, fn, check):
    with monkeypatch.context() as m:
        m.setattr(ref, name, fn)
        with pytest.raises(AssertionError):
            check()


def test_pins_catch_planted_mistakes(monkeypatch, golden_dir):
    orig_scores, orig_kth = ref.row_scores, ref.kth_largest
    orig_sample, orig_attend = ref.calibration_sample, ref.attend_row

    # 1/sqrt(d) dropped from Eq. 1
    _planted(monkeypatch, "row_scores",
             lambda q, K, L: np.asarray(K, float)[:L] @ np.asarray(q, float),
             check_dense_decode)
    # off-by-one order statistic
    _planted(monkeypatch, "kth_largest",
             lambda x, k: orig_kth(x, min(k + 1, len(x))), check_bruteforce_topk)
    # post-softmax quantile taken on a instead of s
    _planted(monkeypatch, "calibration_sample",
             lambda a, k, mode: orig_kth(a, k), lambda: check_golden_calibration(golden_dir))

    # wrong sign of the VMC term, wrong gamma, wrong max in the exp-threshold term
    def flip_beta(*args, **kw):
        r = orig_attend(*args, **kw)
        if len(args) > 5 and args[5]:
            mu = np.asarray(args[6], float)
            r["out"] = r["out"] - 2 * r["beta"] * mu
        return r
    _planted(monkeypatch, "attend_row", flip_beta, lambda: check_golden_sdc_vmc(golden_dir))

    def gamma_doubled(*args, **kw):
        kw = dict(kw)
        if len(args) > 7:
            args = args[:7] + (2 * ref.GAMMA,) + args[8:]
        else:
            kw["gamma"] = 2 * ref.GAMMA
        return orig_attend(*args, **kw)
    _planted(monkeypatch, "attend_row", gamma_doubled, lambda: check_golden_sdc_vmc(golden_dir))

    # nearest-row rule replaced by "always the first calibrated row"
    orig_fin = ref.finalize_thresholds

    def first_row(sets, Hq, Lmax, k, alpha):
        th = orig_fin(sets, Hq, Lmax, k, alpha)
        for h in range(Hq):
            fin = np.flatnonzero(np.isfinite(th[h]))
            if fin.size:
                th[h, fin] = th[h, fin[0]]
        return th
    _planted(monkeypatch, "finalize_thresholds", first_row,
             lambda: check_golden_nearest_row(golden_dir))

    # fitted theta(L) taken in L instead of ln L
    orig_fit = ref.fit_row_ids

    def fit_in_L(value, Lmax, k, mode):
        pts = [(L, v) for L, v in sorted(value.items()) if L > k]
        row = np.full(Lmax, -np.inf)
        if not pts:
            return row
        x = np.array([L for L, _ in pts], float)
        coef = np.polynomial.polynomial.polyfit(x, [v for _, v in pts], min(2, len(pts) - 1))
        row[k:] = np.polynomial.polynomial.polyval(np.arange(k + 1, Lmax + 1, dtype=float), coef)
        return row
    _planted(monkeypatch, "fit_row_ids", fit_in_L, check_fitted_theta)
    assert ref.fit_row_ids is orig_fit

    # GQA: intersection instead of union, and votes compared with > instead of >=
    orig_pol = ref.group_policy

    def wrong_union(keeps, policy, min_heads=1):
        if policy == ref.GQA_UNION:
            K = np.asarray(keeps, dtype=bool)
            return np.repeat(K.all(axis=0)[None, :], K.shape[0], axis=0)
        return orig_pol(keeps, policy, min_heads)
    _planted(monkeypatch, "group_policy", wrong_union, check_gqa_policies)

    def strict_vote(keeps, policy, min_heads=1):
        if policy == ref.GQA_VOTE:
            K = np.asarray(keeps, dtype=bool)
            return K & (K.sum(axis=0) > min_heads)[None, :]
        return orig_pol(keeps, policy, min_heads)
    _planted(monkeypatch, "group_policy", strict_vote, check_gqa_policies)

    # offline E~ summed without subtracting the row maximum
    _planted(monkeypatch, "discarded_sum",
             lambda a, th: float(np.exp(np.asarray(a, float)[np.asarray(a, float) < th]).sum()),
             lambda: check_golden_offline_sdc(golden_dir))

    # MKC: Eq. 8 averaged over all rows instead of the rows holding theta
    def merge_all_rows(seqs):
        out = []
        for lo, hi, tot, cnt in orig_merge(seqs):
            tot = sum(next((t0 for t0, a, b in sq if a <= lo < b), len(sq) + 1 if sq and lo < sq[0][1] else 0)
                      for sq in seqs)
            out.append((lo, hi, tot, len(seqs)))
        return out
    orig_merge, orig_seq, orig_inv = ref.merge_intervals, ref.mkc_interval_sequence, ref.mkc_theta
    _planted(monkeypatch, "merge_intervals", merge_all_rows, lambda: check_golden_mkc(golden_dir))
    # effective k off by one (elements at or above the threshold)
    _planted(monkeypatch, "mkc_interval_sequence",
             lambda x: [(t0 + 1, a, b) for t0, a, b in orig_seq(x)], check_mkc_single_row)
    # inverse taken at the lower end of the piece
    _planted(monkeypatch, "mkc_theta",
             lambda pieces, k: max([lo for lo, hi, t, c in pieces if t >= k * c], default=-np.inf),
             check_mkc_bruteforce)
    assert ref.row_scores is orig_scores and ref.calibration_sample is orig_sample


# ---------------------------------------------------------------------------
# The whole-matrix prefill decisions equal attend_row's, row by row.
# ---------------------------------------------------------------------------
def test_prefill_decisions_match_rows():
    rng = np.random.default_rng(5)
    S, d = 40, 8
    Q = rng.standard_normal((S, d))
    K = rng.standard_normal((S, d))
    V = rng.standard_normal((S, d))
    for mode in (ref.PRE, ref.POST):
        theta = np.full(S, -np.inf)
        for L in range(4, S + 1):
            a = ref.row_scores(Q[L - 1], K, L)
            x = a if mode == ref.PRE else ref.row_softmax(a)
            xs = np.sort(x)
            theta[L - 1] = 0.5 * (xs[-3] + xs[-4])         # between the 3rd and 4th largest
        xs = np.sort(ref.row_scores(Q[20], K, 21) if mode == ref.PRE
                     else ref.row_softmax(ref.row_scores(Q[20], K, 21)))
        theta[20] = xs[-3] * (1 + 5e-4 * np.sign(xs[-3]))  # a row with an element inside the band
        keep, band = ref.prefill_decisions(Q, K, theta, mode)
        assert not np.triu(keep, 1).any() and not np.triu(band, 1).any()
        for i in range(S):
            a = ref.row_scores(Q[i], K, i + 1)
            r = ref.attend_row(a, V[:i + 1], ref.theta_for_row(theta, i + 1), mode)
            assert np.array_equal(keep[i, :i + 1], r["keep"]), (mode, i)
            assert np.array_equal(band[i, :i + 1], r["band"]), (mode, i)
        assert band.any()                                  # the band case is exercised
        assert keep[10].sum() == 3 and keep[2].sum() == 3  # 3rd largest keeps 3; a dense row keeps all
