"""GPU parity of the GQA group policies of decode (Top-Theta §4.6): every
head's final kept set under UNION and VOTE against the float64 oracle.

A key whose threshold decision falls inside the 1e-3 band for any head of
its group may go either way (the policy spreads one head's decision to the
group), so final masks are compared outside those keys, the count is
reported, and the outputs are checked with the kernel's final sets adopted.
"""
import numpy as np
import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt

from gpu_cases import calibrate_prefill_rows, decode_case, mask_words
from parity import OUT_TOL, require_cuda, unpack_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_cuda()
    build.build()
    topt.lib()


def _check_policy(q, K, V, seq_len, theta, mode, sdc, vmc, mu, res, policy, t):
    qn = synth.as_f64(q)
    B, Hq, _ = qn.shape
    g = Hq // K.shape[1]
    sl = seq_len.cpu().numpy()
    th = theta.cpu().double().numpy()
    mun = None if mu is None else mu.cpu().double().numpy()
    out = res["out"].cpu().double().numpy()
    kept = res["kept"].cpu().numpy()
    vrows = res["vrows"].cpu().numpy()
    mask = res["mask"].cpu().numpy()
    n_band = 0
    for b in range(B):
        L = int(sl[b])
        for kv in range(K.shape[1]):
            Kn = synth.as_f64(K[b, kv, :L])
            Vn = synth.as_f64(V[b, kv, :L])
            hs = [kv * g + i for i in range(g)]
            own = [ref.attend_row(ref.row_scores(qn[b, h], Kn, L), Vn, ref.theta_for_row(th[h], L),
                                  mode, sdc, vmc, None if mun is None else mun[b, kv]) for h in hs]
            band = np.any([r["band"] for r in own], axis=0)
            n_band += int(band.sum())
            want = ref.group_policy([r["keep"] for r in own], policy, t)
            got = np.array([unpack_mask(mask[b, h], L) for h in hs])
            mism = (got != want) & ~band[None, :]
            assert not mism.any(), (b, kv, np.argwhere(mism)[:5])
            assert vrows[b, kv] == int(got.any(axis=0).sum())
            for i, h in enumerate(hs):
                a = ref.row_scores(qn[b, h], Kn, L)
                r = ref.attend_row(a, Vn, ref.theta_for_row(th[h], L), mode, sdc, vmc,
                                   None if mun is None else mun[b, kv], keep=got[i])
                assert kept[b, h] == r["kept"]
                err = ref.output_rel_error(out[b, h], r["out"])
                assert err <= OUT_TOL, (b, h, err)
    return n_band


MODES = [(ref.PRE, ref.SDC_NONE, False), (ref.PRE, ref.SDC_EXACT, True), (ref.POST, ref.SDC_NONE, True)]


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (6, 2), (16, 2)])
@pytest.mark.parametrize("policy,t", [(ref.GQA_UNION, 1), (ref.GQA_VOTE, 2), (ref.GQA_VOTE, 3)])
def test_decode_gqa_policy_matches_oracle(Hq, Hkv, policy, t):
    B, d, Nmax, k = 3, 128, 700, 16
    seq = [700, 1, 333]
    q, K, V, _ = decode_case(91, B, Hq, Hkv, d, Nmax, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = torch.stack([V[b, :, :int(L)].float().mean(dim=1) for b, L in enumerate(seq)])
    for mode, sdc, vmc in MODES:
        theta, _ = calibrate_prefill_rows(92, 2, Hq, Hkv, d, 512, k, mode, Nmax)
        mask = torch.zeros((B, Hq, mask_words(Nmax)), device="cuda", dtype=torch.int32) - 1
        res = topt.decode(q, K, V, seq_len, theta, mode=mode, sdc=sdc, vmc=vmc, mu=mu, mask=mask,
                          gqa=policy, gqa_min_heads=t)
        torch.cuda.synchronize()
        _check_policy(q, K, V, seq_len, theta, mode, sdc, vmc, mu if vmc else None, res, policy, t)


def test_decode_gqa_vote_one_is_own_selection_and_union_reads_no_more_rows():
    B, Hq, Hkv, d, Nmax, k = 4, 32, 8, 128, 2048, 64
    seq = [2048, 1500, 77, 1]
    q, K, V, _ = decode_case(93, B, Hq, Hkv, d, Nmax, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    theta, _ = calibrate_prefill_rows(94, 2, Hq, Hkv, d, 2048, k, ref.PRE, Nmax)
    own = topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_EXACT)
    one = topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_EXACT, gqa=ref.GQA_VOTE,
                      gqa_min_heads=1)
    uni = topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_EXACT, gqa=ref.GQA_UNION)
    big = topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, sdc=ref.SDC_EXACT, gqa=ref.GQA_VOTE,
                      gqa_min_heads=Hq // Hkv + 1)
    torch.cuda.synchronize()
    assert torch.equal(one["kept"], own["kept"]) and torch.equal(one["vrows"], own["vrows"])
    torch.testing.assert_close(one["out"], own["out"], rtol=0, atol=0)
    assert torch.equal(uni["vrows"], own["vrows"])
    assert torch.all(uni["kept"] >= own["kept"])
    assert int(big["kept"].abs().sum()) == 0 and int(big["vrows"].abs().sum()) == 0
    with pytest.raises(topt.ToptError):
        topt.decode(q, K, V, seq_len, theta, mode=ref.PRE, gqa=ref.GQA_VOTE, gqa_min_heads=0)
