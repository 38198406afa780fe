"""GPU parity of every entry point against the float64 oracle, small shapes.

Shapes span several tiles and chunks with ragged tails; edge cases: rows
shorter than k, a single key, dense (theta = -inf) and empty selections,
bad device-side lengths.
"""
import numpy as np
import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt

from gpu_cases import (calibrate_decode_rows, calibrate_prefill_rows, decode_case, mask_words,
                       prefill_case)
from parity import check_decode, check_prefill, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_cuda()
    build.build()
    topt.lib()


# ---------------------------------------------------------------------------
# radix select: bit-exact
# ---------------------------------------------------------------------------
def test_select_kth_is_exact():
    rng = np.random.default_rng(0)
    rows, stride = 37, 3000
    x = rng.standard_normal((rows, stride)).astype(np.float32) * 5
    x[3, :50] = 1.5                                   # ties
    x[4, :] = np.round(x[4, :])                       # many ties, zeros
    x[5, ::2] = -0.0
    x[6, :] = -np.abs(x[6, :])                        # all negative
    x[7, :10] = np.inf
    x[8, :] = np.float32(1e-40)                       # denormals
    lens = rng.integers(1, stride + 1, rows).astype(np.int32)
    lens[:10] = [1, 2, 3000, 2999, 400, 1000, 777, 64, 3000, 17]
    xd = torch.from_numpy(x).cuda()
    ld = torch.from_numpy(lens).cuda()
    for k in (1, 2, 7, 128, 512):
        got = topt.select_kth(xd, ld, k).cpu().numpy()
        for r in range(rows):
            L = lens[r]
            if L < k:
                assert got[r] == -np.inf
                continue
            want = np.partition(x[r, :L], L - k)[L - k]
            assert got[r] == want, (k, r, got[r], want)
            if want != 0:
                assert got[r].view(np.uint32) == np.float32(want).view(np.uint32)


# ---------------------------------------------------------------------------
# calibration table vs Algorithm 1 in float64
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [ref.PRE, ref.POST])
@pytest.mark.parametrize("alpha", [0.0, 0.5])
@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (128, torch.bfloat16)])
def test_calibration_matches_oracle(mode, alpha, d, dtype):
    Hq, Hkv, S, k, Lmax, N = 4, 2, 48, 5, 64, 3
    theta, cal = calibrate_prefill_rows(11, N, Hq, Hkv, d, S, k, mode, Lmax, alpha, dtype)
    Qs, Ks = [], []
    for n in range(N):
        Q, K, _ = prefill_case(11 * 1000 + n, 1, Hq, Hkv, d, S, dtype)
        Qs.append(synth.as_f64(Q)[0])
        Ks.append(synth.as_f64(K)[0])
    want, sets = ref.calibrate_ref(np.stack(Qs), np.stack(Ks), np.arange(1, S + 1), k, mode, alpha, Lmax)
    got = theta.cpu().double().numpy()
    cnt = cal.count.cpu().numpy()
    for h in range(Hq):
        for L in range(1, Lmax + 1):
            assert cnt[h, L - 1] == len(sets.get((h, L), [])), (h, L)
    assert np.array_equal(np.isneginf(got), np.isneginf(want))
    fin = np.isfinite(want)
    tol = 1e-4 * (np.abs(want[fin]) + 1e-6) if mode == ref.PRE else 1e-4 * np.abs(want[fin])
    if alpha:
        # std of three samples amplifies score rounding; bound it by the sample spread
        tol = tol + 2e-5 * (np.abs(want[fin]) + 1.0)
    assert np.all(np.abs(got[fin] - want[fin]) <= tol), np.max(np.abs(got[fin] - want[fin]) / tol)


def test_calibration_accumulates_across_calls():
    Hq, Hkv, d, S, k, Lmax = 2, 1, 64, 40, 4, 40
    whole, _ = calibrate_prefill_rows(5, 4, Hq, Hkv, d, S, k, ref.PRE, Lmax)
    cal = topt.Calibrator(Hq, Lmax, k, ref.PRE)
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    Qs, Ks = zip(*[prefill_case(5 * 1000 + n, 1, Hq, Hkv, d, S)[:2] for n in range(4)])
    cal.add(torch.cat(Qs[:1]), torch.cat(Ks[:1]), row_len, reset=True)
    cal.add(torch.cat(Qs[1:]), torch.cat(Ks[1:]), row_len)
    got = cal.finalize()
    fin = torch.isfinite(whole)
    assert torch.equal(torch.isfinite(got), fin)
    torch.testing.assert_close(got[fin], whole[fin], rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
DECODE_MODES = [
    (ref.POST, ref.SDC_NONE, True), (ref.POST, ref.SDC_NONE, False),
    (ref.PRE, ref.SDC_NONE, False), (ref.PRE, ref.SDC_EXACT, True),
    (ref.PRE, ref.SDC_EXPTH, True), (ref.PRE, ref.SDC_EXPTH, False),
]


def run_decode(q, K, V, seq_len, theta, mode, sdc, vmc, mu=None, status=None):
    B, Hq, _ = q.shape
    mask = torch.zeros((B, Hq, mask_words(K.shape[2])), device="cuda", dtype=torch.int32) - 1
    res = topt.decode(q, K, V, seq_len, theta, mode=mode, sdc=sdc, vmc=vmc, mu=mu, mask=mask,
                      status=status)
    torch.cuda.synchronize()
    return res


def mean_rows(V, seq_len):
    return torch.stack([V[b, :, :int(L)].float().mean(dim=1) for b, L in enumerate(seq_len.tolist())])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (16, 2), (6, 2), (4, 2), (10, 2), (14, 2)])
def test_decode_matches_oracle(d, Hq, Hkv):
    """Group sizes 1, 4, 8, 3, 2, 5, 7: every score-column layout (G, G padded
    to even) the kernel is built for, at both head sizes."""
    B, Nmax, k = 3, 1100, 16
    seq = [1100, 1, 601]
    q, K, V, ch = decode_case(21, B, Hq, Hkv, d, Nmax, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = mean_rows(V, seq_len)
    for mode, sdc, vmc in DECODE_MODES:
        theta, _ = calibrate_prefill_rows(22, 2, Hq, Hkv, d, 1024, k, mode, Nmax)
        res = run_decode(q, K, V, seq_len, theta, mode, sdc, vmc, mu)
        check_decode(q, K, V, seq_len, theta, mode, sdc, vmc, mu, res)


def test_decode_dense_and_empty():
    B, Hq, Hkv, d, Nmax = 2, 8, 2, 128, 777
    seq = [777, 40]
    q, K, V, _ = decode_case(31, B, Hq, Hkv, d, Nmax, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = mean_rows(V, seq_len)
    dense = torch.full((Hq, Nmax), float("-inf"), device="cuda")
    for mode, sdc, vmc in DECODE_MODES:
        res = run_decode(q, K, V, seq_len, dense, mode, sdc, vmc, mu)
        assert torch.equal(res["kept"].cpu(), torch.tensor([[777] * Hq, [40] * Hq], dtype=torch.int32))
        assert torch.equal(res["vrows"].cpu(), torch.tensor([[777] * Hkv, [40] * Hkv], dtype=torch.int32))
        check_decode(q, K, V, seq_len, dense, mode, sdc, vmc, mu, res)
    # nothing survives: post + VMC and pre + SDC give mu, pre without SDC gives 0
    for mode, th in ((ref.POST, 1.5), (ref.PRE, 1e4)):
        full = torch.full((Hq, Nmax), th, device="cuda")
        for sdc, vmc in ((ref.SDC_NONE, True), (ref.SDC_EXACT, True), (ref.SDC_NONE, False)):
            res = run_decode(q, K, V, seq_len, full, mode, sdc, vmc, mu)
            assert int(res["kept"].sum()) == 0 and int(res["vrows"].sum()) == 0
            eligible = mode == ref.POST or sdc != ref.SDC_NONE
            want = mu.repeat_interleave(Hq // Hkv, dim=1) if (vmc and eligible) else torch.zeros_like(res["out"])
            torch.testing.assert_close(res["out"], want, rtol=1e-6, atol=1e-6)


def test_decode_bad_seq_len_sets_status():
    B, Hq, Hkv, d, Nmax = 3, 4, 1, 64, 300
    q, K, V, _ = decode_case(41, B, Hq, Hkv, d, Nmax, [300, 300, 300])
    theta = torch.full((Hq, Nmax), float("-inf"), device="cuda")
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    seq_len = torch.tensor([300, 0, 301], device="cuda", dtype=torch.int32)
    out = torch.full((B, Hq, d), 7.0, device="cuda")
    topt.decode(q, K, V, seq_len, theta, mode=ref.POST, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.all(out[1:] == 7.0)                 # skipped units left untouched
    assert torch.isfinite(out[0]).all()


def test_decode_reuses_workspace():
    B, Hq, Hkv, d, Nmax = 2, 8, 2, 128, 2048
    q, K, V, _ = decode_case(51, B, Hq, Hkv, d, Nmax, [2048, 1500])
    seq_len = torch.tensor([2048, 1500], device="cuda", dtype=torch.int32)
    theta, _ = calibrate_prefill_rows(52, 2, Hq, Hkv, d, 512, 32, ref.POST, Nmax)
    args = topt.decode_args(q, K, V, seq_len, theta, mode=ref.POST)
    ws = topt.decode_workspace(args, "cuda")
    a = topt.decode(q, K, V, seq_len, theta, mode=ref.POST, workspace=ws)
    first = a["out"].clone()
    for _ in range(3):
        b = topt.decode(q, K, V, seq_len, theta, mode=ref.POST, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(first, b["out"])              # deterministic: no state kept between calls


# ---------------------------------------------------------------------------
# running mean
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_vmean_running_mean(dtype):
    B, Hkv, d, Nmax = 2, 3, 128, 600
    gen = synth.generator(61, "cuda")
    V = synth.values(gen, B, Hkv, Nmax, d, device="cuda", dtype=dtype)
    mu = torch.zeros((B, Hkv, d), device="cuda")
    n_old = torch.zeros(B, device="cuda", dtype=torch.int32)
    topt.vmean_update(V, n_old, 500, mu)                       # prefill initialisation
    for t in range(500, 600):                                  # then one token at a time
        n_old.fill_(t)
        topt.vmean_update(V, n_old, 1, mu)
    torch.cuda.synchronize()
    want = np.mean(synth.as_f64(V), axis=2)
    np.testing.assert_allclose(mu.cpu().double().numpy(), want, rtol=0, atol=1e-5)
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    n_old.fill_(600)
    topt.vmean_update(V, n_old, 1, mu, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1


def test_vmean_prepared_args_reused():
    """topt.vmean_args prepares the call once; calling the C ABI with the same
    struct for consecutive tokens gives the running mean (the serving-loop use)."""
    import ctypes
    B, Hkv, d, Nmax = 2, 2, 64, 300
    gen = synth.generator(62, "cuda")
    V = synth.values(gen, B, Hkv, Nmax, d, device="cuda")
    mu = torch.zeros((B, Hkv, d), device="cuda")
    n_old = torch.zeros(B, device="cuda", dtype=torch.int32)
    topt.vmean_update(V, n_old, 200, mu)
    a = topt.vmean_args(V, n_old, 1, mu)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for t in range(200, 300):
        n_old.fill_(t)
        assert topt.lib().topt_vmean_update(ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()
    np.testing.assert_allclose(mu.cpu().double().numpy(), np.mean(synth.as_f64(V), axis=2), rtol=0, atol=1e-5)


@pytest.mark.parametrize("dtype,t", [(torch.bfloat16, 1), (torch.float32, 3), (torch.bfloat16, 70)])
def test_vmean_appends_new_rows(dtype, t):
    """With k_new / v_new the same launch writes the new rows into both caches
    at rows n_old.. (bit for bit, nothing else touched) and averages them: mu
    then equals the update of a cache that already held those rows."""
    B, Hkv, d, Nmax = 2, 3, 128, 400
    gen = synth.generator(63, "cuda")
    K = synth.iid_normal(gen, (B, Hkv, Nmax, d), "cuda", dtype)
    V = synth.values(gen, B, Hkv, Nmax, d, device="cuda", dtype=dtype)
    k_new = synth.iid_normal(gen, (B, Hkv, t, d), "cuda", dtype)
    v_new = synth.iid_normal(gen, (B, Hkv, t, d), "cuda", dtype)
    n_old = torch.tensor([250, 399 - t], device="cuda", dtype=torch.int32)
    mu0 = torch.zeros((B, Hkv, d), device="cuda")
    for b in range(B):
        topt.vmean_update(V[b:b + 1], n_old[b:b + 1].clone().zero_(), int(n_old[b]), mu0[b:b + 1])
    K2, V2, mu = K.clone(), V.clone(), mu0.clone()
    topt.vmean_update(V2, n_old, t, mu, k_cache=K2, k_new=k_new, v_new=v_new)
    # reference: the rows written by hand, then the plain update
    K3, V3, mu_ref = K.clone(), V.clone(), mu0.clone()
    for b in range(B):
        n0 = int(n_old[b])
        K3[b, :, n0:n0 + t] = k_new[b]
        V3[b, :, n0:n0 + t] = v_new[b]
    topt.vmean_update(V3, n_old, t, mu_ref)
    torch.cuda.synchronize()
    assert torch.equal(K2, K3) and torch.equal(V2, V3)
    assert torch.equal(mu, mu_ref)
    # and against the float64 mean of the prefix plus the new rows
    want = np.stack([np.mean(synth.as_f64(V3)[b, :, :int(n_old[b]) + t], axis=1) for b in range(B)])
    np.testing.assert_allclose(mu.cpu().double().numpy(), want, rtol=0, atol=1e-5)


def test_vmean_append_rejects_missing_k_cache():
    import ctypes
    B, Hkv, d, Nmax = 1, 1, 64, 16
    V = torch.zeros((B, Hkv, Nmax, d), device="cuda", dtype=torch.bfloat16)
    mu = torch.zeros((B, Hkv, d), device="cuda")
    n_old = torch.zeros(B, device="cuda", dtype=torch.int32)
    k_new = torch.zeros((B, Hkv, 1, d), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        topt.vmean_args(V, n_old, 1, mu, k_new=k_new)
    a = topt.vmean_args(V, n_old, 1, mu)
    a.k_new = ctypes.c_void_p(k_new.data_ptr())          # k_cache left NULL
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert topt.lib().topt_vmean_update(ctypes.byref(a), stream) == 1   # TOPT_EINVAL, nothing launched


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
PREFILL_MODES = [
    (ref.PRE, ref.SDC_NONE, False), (ref.PRE, ref.SDC_EXACT, True), (ref.PRE, ref.SDC_EXPTH, True),
    (ref.POST, ref.SDC_NONE, True), (ref.POST, ref.SDC_NONE, False),
]


@pytest.mark.parametrize("d,dtype,B,Hq,Hkv,S", [
    (64, torch.float32, 2, 4, 2, 100),
    (128, torch.bfloat16, 2, 4, 2, 100),
    (64, torch.bfloat16, 2, 4, 2, 100),
    (128, torch.bfloat16, 1, 4, 1, 300),    # three 128-row blocks, ragged last block and key tile
    (64, torch.bfloat16, 1, 2, 2, 257),     # one KV head per query head, ragged
    (128, torch.bfloat16, 1, 3, 1, 200),    # odd GQA group: one head per CTA in the single-pass kernel
])
def test_prefill_matches_oracle(d, dtype, B, Hq, Hkv, S):
    k = 8
    Q, K, V = prefill_case(71, B, Hq, Hkv, d, S, dtype)
    for mode, sdc, vmc in PREFILL_MODES:
        theta, _ = calibrate_prefill_rows(72, 2, Hq, Hkv, d, S, k, mode, 80, dtype=dtype)
        mask = torch.full((B, Hq, S, mask_words(S)), -1, device="cuda", dtype=torch.int32)
        tiles = torch.zeros(2, device="cuda", dtype=torch.int64)
        res = topt.prefill(Q, K, V, theta, mode=mode, sdc=sdc, vmc=vmc, mask=mask, tiles=tiles)
        torch.cuda.synchronize()
        n, n_band, worst, keep_rows = check_prefill(Q, K, V, theta, mode, sdc, vmc, res)
        tm, tn = topt.prefill_tile_shape(topt.prefill_args(Q, K, V, theta, mode=mode))
        hit = total = 0
        for b in range(B):
            for h in range(Hq):
                kr = {i: keep_rows[(b, h, i)] for i in range(S)}
                hh, tt = ref.tile_counts_ref(kr, S, tm, tn)
                hit += hh
                total += tt
        assert tiles.tolist() == [hit, total]


@pytest.mark.parametrize("d,dtype,S", [(128, torch.bfloat16, 129), (64, torch.bfloat16, 1),
                                       (64, torch.float32, 129)])
def test_prefill_dense_and_empty(d, dtype, S):
    """theta = -inf keeps every causal key (dense attention, every tile executed);
    a threshold nothing reaches skips every P.V tile: post-softmax and pre-softmax
    with SDC give the prefix mean of V under VMC, the rest give 0."""
    B, Hq, Hkv = 1, 4, 2
    Q, K, V = prefill_case(81, B, Hq, Hkv, d, S, dtype)
    dense = torch.full((Hq, S), float("-inf"), device="cuda")
    for mode, sdc, vmc in PREFILL_MODES:
        mask = torch.full((B, Hq, S, mask_words(S)), -1, device="cuda", dtype=torch.int32)
        tiles = torch.zeros(2, device="cuda", dtype=torch.int64)
        res = topt.prefill(Q, K, V, dense, mode=mode, sdc=sdc, vmc=vmc, mask=mask, tiles=tiles)
        torch.cuda.synchronize()
        want_kept = torch.arange(1, S + 1, dtype=torch.int32).expand(B, Hq, S)
        assert torch.equal(res["kept"].cpu(), want_kept)
        assert tiles[0].item() == tiles[1].item() > 0
        check_prefill(Q, K, V, dense, mode, sdc, vmc, res)
    Vf = V.double()
    mu = Vf.cumsum(dim=2) / torch.arange(1, S + 1, device="cuda", dtype=torch.float64)[:, None]
    mu_q = mu.repeat_interleave(Hq // Hkv, dim=1).float()
    for mode, th in ((ref.POST, 1.5), (ref.PRE, 1e4)):
        full = torch.full((Hq, S), th, device="cuda")
        for sdc, vmc in ((ref.SDC_NONE, True), (ref.SDC_EXACT, True), (ref.SDC_NONE, False)):
            tiles = torch.zeros(2, device="cuda", dtype=torch.int64)
            res = topt.prefill(Q, K, V, full, mode=mode, sdc=sdc, vmc=vmc, tiles=tiles)
            torch.cuda.synchronize()
            assert int(res["kept"].sum()) == 0
            assert tiles[0].item() == 0 and tiles[1].item() > 0
            eligible = mode == ref.POST or sdc != ref.SDC_NONE
            want = mu_q if (vmc and eligible) else torch.zeros_like(res["out"])
            torch.testing.assert_close(res["out"], want, rtol=2e-5, atol=2e-5)


@pytest.mark.parametrize("mode", [ref.PRE, ref.POST])
def test_prefill_wait_runs_out_and_context_survives(mode):
    """A wait of a tensor-core kernel (pre-softmax: the single-pass kernel;
    post-softmax: the two-pass one) that never completes (the test hook never
    loads the first K tile of a block) gives up after its time limit: the call
    reports TOPT_ETIMEOUT, nothing faults, and the next call is correct."""
    import ctypes
    B, Hq, Hkv, d, S = 1, 2, 1, 128, 200
    Q, K, V = prefill_case(91, B, Hq, Hkv, d, S)
    dense = torch.full((Hq, S), float("-inf") if mode == ref.PRE else 0.0, device="cuda")
    status = torch.zeros(1, device="cuda", dtype=torch.int32)
    out = torch.empty((B, Hq, S, d), device="cuda")
    a = topt.prefill_args(Q, K, V, dense, mode=mode, out=out, status=status)
    ws = torch.empty(max(1, topt.prefill_workspace_bytes(a)), device="cuda", dtype=torch.uint8)
    a.workspace = ctypes.c_void_p(ws.data_ptr())
    a.workspace_bytes = ws.numel()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert topt.lib().topt_prefill_test_timeout(ctypes.byref(a), stream) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 5                               # TOPT_ETIMEOUT
    status.zero_()
    mask = torch.full((B, Hq, S, mask_words(S)), -1, device="cuda", dtype=torch.int32)
    res = topt.prefill(Q, K, V, dense, mode=mode, mask=mask, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_prefill(Q, K, V, dense, mode, ref.SDC_NONE, False, res)
