"""Parity helpers shared by the GPU tests: compare CUDA results with the oracle.

Bars (from the method's statement of the workloads):
  * masks and kept counts: bit-exact, except elements whose thresholded value
    lies within 1e-3 (relative) of theta; those are counted and the oracle
    adopts the kernel's decision there before computing its outputs;
  * outputs: per row  max|p - p_ref| / max|p_ref| <= 2e-3.
"""
import json
import os

import numpy as np
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import synth

OUT_TOL = 2e-3
BAND_BOUND = 1e-3          # at most this fraction of the compared elements may fall in the band
RECORD = os.environ.get("TOPT_PARITY_RECORD",
                        os.path.join(os.path.dirname(os.path.abspath(__file__)), "records",
                                     "parity_bands.json"))


# Counts of the last check: elements compared, in the band, and band elements
# the kernel decides differently from the oracle (excluded from the bit-exact
# comparison, reported).
LAST = {"elements": 0, "band": 0, "band_disagree": 0}


def record_band(config, case, stats=None):
    """Asserts the band bound and adds (config, case) to the JSON record of
    decisions excluded from the bit-exact mask comparison."""
    st = dict(LAST if stats is None else stats)
    n_band, n_elem = st["band"], st["elements"]
    frac = n_band / max(1, n_elem)
    assert frac <= BAND_BOUND, f"{config} {case}: {n_band} of {n_elem} elements in the band"
    os.makedirs(os.path.dirname(RECORD), exist_ok=True)
    try:
        with open(RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    rec.setdefault(config, {})[case] = {"band_elements": int(n_band), "elements_compared": int(n_elem),
                                        "fraction": frac,
                                        "band_decided_otherwise": int(st["band_disagree"])}
    with open(RECORD, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)


def unpack_mask(words, L):
    """int32 bitmap words -> bool [L]."""
    w = np.asarray(words, dtype=np.int64) & 0xFFFFFFFF
    bits = ((w[:, None] >> np.arange(32)[None, :]) & 1).astype(bool).reshape(-1)
    return bits[:L]


def check_decode(q, Kc, Vc, seq_len, theta, mode, sdc, vmc, mu, res, gamma=ref.GAMMA, heads=None,
                 out_tol=OUT_TOL, e_tilde=None):
    """Compare topt.decode results (dict of tensors incl. mask) with decode_ref.

    Returns (n_rows_checked, n_band_elements, max_rel_err).
    """
    qn = synth.as_f64(q)
    B, Hq, _ = qn.shape
    Hkv = Kc.shape[1]
    g = Hq // Hkv
    sl = seq_len.cpu().numpy()
    th = theta.cpu().double().numpy()
    et = None if e_tilde is None else e_tilde.cpu().double().numpy()
    mun = None if mu is None else mu.cpu().double().numpy()
    out = res["out"].cpu().double().numpy()
    kept = res["kept"].cpu().numpy()
    vrows = res["vrows"].cpu().numpy()
    mask = res["mask"].cpu().numpy()
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    by_pair = {}
    for (b, h) in heads:
        by_pair.setdefault((b, h // g), []).append(h)
    n_band = n_elem = n_dis = 0
    worst = 0.0
    for (b, kv), hs in by_pair.items():
        L = int(sl[b])
        n_elem += L * len(hs)
        Kn = synth.as_f64(Kc[b, kv, :L])
        Vn = synth.as_f64(Vc[b, kv, :L])
        union = np.zeros(L, dtype=bool)
        for h in hs:
            a = ref.row_scores(qn[b, h], Kn, L)
            gpu_keep = unpack_mask(mask[b, h], L)
            e_off = 0.0 if et is None else ref.theta_for_row(et[h], L)
            r0 = ref.attend_row(a, Vn, ref.theta_for_row(th[h], L), mode, sdc, vmc,
                                None if mun is None else mun[b, kv], gamma, e_tilde=e_off)
            band = r0["band"]
            n_band += int(band.sum())
            n_dis += int(((gpu_keep != r0["keep"]) & band).sum())
            mism = (gpu_keep != r0["keep"]) & ~band
            assert not mism.any(), f"mask mismatch (b={b}, h={h}) at {np.flatnonzero(mism)[:10]}"
            assert not unpack_mask(mask[b, h], mask.shape[-1] * 32)[L:].any(), "bits beyond L"
            r = ref.attend_row(a, Vn, ref.theta_for_row(th[h], L), mode, sdc, vmc,
                               None if mun is None else mun[b, kv], gamma, decide=gpu_keep,
                               e_tilde=e_off)
            assert kept[b, h] == r["kept"], (b, h, kept[b, h], r["kept"])
            err = ref.output_rel_error(out[b, h], r["out"])
            worst = max(worst, err)
            assert err <= out_tol, f"output error {err:.3e} (b={b}, h={h})"
            union |= gpu_keep
        if len(hs) == g:
            assert vrows[b, kv] == int(union.sum()), (b, kv, vrows[b, kv], int(union.sum()))
    LAST.update(elements=n_elem, band=n_band, band_disagree=n_dis)
    return len(heads), n_band, worst


def check_prefill(Q, K, V, theta, mode, sdc, vmc, res, rows=None, gamma=ref.GAMMA, out_tol=OUT_TOL,
                  e_tilde=None):
    """Compare topt.prefill results (with mask) with prefill_ref on the given rows."""
    Qn, Kn, Vn = synth.as_f64(Q), synth.as_f64(K), synth.as_f64(V)
    B, Hq, S, _ = Qn.shape
    g = Hq // Kn.shape[1]
    th = theta.cpu().double().numpy()
    et = None if e_tilde is None else e_tilde.cpu().double().numpy()
    out = res["out"].cpu().double().numpy()
    kept = res["kept"].cpu().numpy()
    mask = res["mask"].cpu().numpy()
    if rows is None:
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(S)]
    n_band = n_elem = n_dis = 0
    worst = 0.0
    keep_rows = {}
    for (b, h, i) in rows:
        L = i + 1
        kv = h // g
        a = ref.row_scores(Qn[b, h, i], Kn[b, kv], L)
        mu = ref.vmean_ref(Vn[b, kv, :L]) if vmc else None
        gk = unpack_mask(mask[b, h, i], L)
        e_off = 0.0 if et is None else ref.theta_for_row(et[h], L)
        r0 = ref.attend_row(a, Vn[b, kv, :L], ref.theta_for_row(th[h], L), mode, sdc, vmc, mu, gamma,
                            e_tilde=e_off)
        band = r0["band"]
        n_band += int(band.sum())
        n_elem += L
        n_dis += int(((gk != r0["keep"]) & band).sum())
        mism = (gk != r0["keep"]) & ~band
        assert not mism.any(), f"mask mismatch (b={b}, h={h}, i={i}) at {np.flatnonzero(mism)[:10]}"
        assert not unpack_mask(mask[b, h, i], mask.shape[-1] * 32)[L:].any(), "bits beyond row"
        r = ref.attend_row(a, Vn[b, kv, :L], ref.theta_for_row(th[h], L), mode, sdc, vmc, mu,
                           gamma, decide=gk, e_tilde=e_off)
        assert kept[b, h, i] == r["kept"], (b, h, i)
        err = ref.output_rel_error(out[b, h, i], r["out"])
        worst = max(worst, err)
        assert err <= out_tol, f"output error {err:.3e} (b={b}, h={h}, i={i})"
        keep_rows[(b, h, i)] = gk
    LAST.update(elements=n_elem, band=n_band, band_disagree=n_dis)
    return len(rows), n_band, worst, keep_rows


def theta_from_gpu(calibrator_theta):
    return calibrator_theta.detach().clone()


def require_cuda():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("CUDA GPU not available")


def unpack_rows(words, S):
    """int32 bitmap [S][W] -> bool [S][S] (bit j%32 of word j/32 of row i)."""
    w = np.asarray(words, dtype=np.int64) & 0xFFFFFFFF
    bits = ((w[:, :, None] >> np.arange(32)[None, None, :]) & 1).astype(bool)
    return bits.reshape(w.shape[0], -1)[:, :S]


def check_prefill_all_masks(Q, K, theta, mode, res):
    """Masks and kept counts of every row of every head of a prefill against
    the oracle's whole-matrix decisions; returns the counts (as LAST)."""
    Qn, Kn = synth.as_f64(Q), synth.as_f64(K)
    B, Hq, S, _ = Qn.shape
    g = Hq // Kn.shape[1]
    th = theta.cpu().double().numpy()
    mask = res["mask"].cpu().numpy()
    kept = res["kept"].cpu().numpy()
    n_band = n_elem = n_dis = 0
    for b in range(B):
        for h in range(Hq):
            keep, band = ref.prefill_decisions(Qn[b, h], Kn[b, h // g], th[h], mode)
            gk = unpack_rows(mask[b, h], S)
            mism = (gk != keep) & ~band
            assert not mism.any(), f"mask mismatch (b={b}, h={h}) at {np.argwhere(mism)[:5]}"
            assert not np.triu(gk, 1).any(), f"bits beyond the row (b={b}, h={h})"
            assert np.array_equal(kept[b, h], gk.sum(axis=1)), f"kept counts (b={b}, h={h})"
            n_band += int(band.sum())
            n_dis += int(((gk != keep) & band).sum())
            n_elem += S * (S + 1) // 2
    return {"elements": n_elem, "band": n_band, "band_disagree": n_dis}
