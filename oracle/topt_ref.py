"""Plain float64 CPU oracle for Top-theta attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Sources (cited below by short name):

* [TopTheta] "Top-Theta Attention: Sparsifying Transformers by Compensated
  Thresholding" (arXiv 2502.08363v2, HTML).  §2.2 Eq. 1-3 (attention),
  §3.1 Algorithm 1 (threshold calibration), §3.2.1 Eq. 4 and the three
  estimators of the discarded mass (SDC), §3.2.2 Eq. 5-7 (VMC), §4.6 (GQA:
  V rows are counted per group).
* [Verdict] pith.science verdict on arXiv 2502.08363, "load_bearing_attack":
  rows longer than the calibrated ones use the nearest calibrated threshold.

Readings where the pages are silent or garbled (each one is listed with its
reason in the design notes of the repository):

* c1  an element is kept iff x >= theta (ties are kept).
* c2  the per-sample "(n-k)/n quantile" is the k-th largest valid element
      (order statistic, no interpolation).
* c3  a row is keyed by L, the number of keys it sees; the threshold table
      holds the row with L keys at index L-1.
* c4  rows with L <= k are dense (theta = -inf).
* c5  a row id that was never calibrated takes the nearest calibrated row id
      (ties go to the shorter row); a head with no calibrated row is dense.
* c6  scores are scaled by 1/sqrt(d); causally masked keys do not exist.
* c7  post-softmax thresholds are the arithmetic mean of probabilities.
* c8  the exp-threshold estimate uses the same max-shifted units as R:
      E~ = gamma (L - k~) exp(theta - m).
* c9  m is the true row maximum over all valid keys.
* c10 beta = 1 - sum of the final (after SDC) kept probabilities.
* c11 mu in causal prefill is the prefix mean of V rows 0..L-1.
* c12 an empty selection gives num = 0 and R = 0 (pre without SDC: out = 0).
* c13 std uses ddof = 1; a single sample has std 0.
* c16 post-softmax with SDC is post-softmax (SDC maps pre onto post).
* c19 MKC: theta_r(k) = sup{theta : k_bar_r(theta) >= k} (App. D leaves the
      inverse of a fractional, not always monotone k_bar open); Eq. 8 averages
      only over the intervals that contain theta, as printed.
* c20 offline-calibrated E~ (estimator 1 of §3.2.1) is the mean, over the
      calibration rows of a row id, of the exact discarded sum E of each row
      under the inference thresholds, in the max-shifted units of reading c8;
      rows with theta = -inf get 0; row ids without samples take the nearest
      sampled one (reading c5), none at all 0.  At inference it is used as
      it is, whatever the row itself keeps.
* c22 fitted theta(L): the pages mention a function of the sequence length
      fitted to the calibrated thresholds without its form; here a least-
      squares line (degree min(1, n - 1)) in ln L through the n calibrated
      row ids L > k, fitted to theta (pre) or to ln theta (post, positive
      values only), and used for every row id L > k.  A quadratic in ln L
      was tried first and extrapolated badly past the calibrated lengths.
      The post-softmax value is kept between the smallest normal float32 and
      the largest calibrated value (a probability threshold of 1 or more
      would drop every key of a row, one of 0 would keep them all).
* c21 GQA group policies (§4.6, the two alternatives): UNION gives every head
      of a group the union of the group's kept sets; VOTE keeps a key for a
      head only if the head keeps it and at least t heads of the group do.
      Each head then normalises over its final set (R, k~, SDC, beta).
"""
from __future__ import annotations

import math

import numpy as np

PRE, POST = 0, 1
SDC_NONE, SDC_EXACT, SDC_EXPTH, SDC_OFFLINE = 0, 1, 2, 3
GQA_OWN, GQA_UNION, GQA_VOTE = 0, 1, 2
GAMMA = 0.05          # [TopTheta §3.2.1, exp-threshold estimator]
BAND_REL = 1e-3       # decisions within this relative distance of theta are not compared
FLT32_MIN_NORMAL = 2.0 ** -126


# ---------------------------------------------------------------------------
# Eq. 1: scores of one query row against the keys it sees.
# ---------------------------------------------------------------------------
def row_scores(q, K, L):
    """a_j = q . K_j / sqrt(d) for j < L  ([TopTheta §2.2 Eq. 1], reading c6)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    d = q.shape[-1]
    return (K[:L] @ q) / math.sqrt(d)


def row_softmax(a):
    """Eq. 2 with the row maximum subtracted first (Eq. 4 writes it this way)."""
    m = np.max(a)
    e = np.exp(a - m)
    return e / e.sum()


# ---------------------------------------------------------------------------
# Algorithm 1: calibration.
# ---------------------------------------------------------------------------
def kth_largest(x, k):
    """The k-th largest element of x (1-based), reading c2."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[0]
    return np.partition(x, n - k)[n - k]


def calibration_sample(a, k, mode):
    """One observed threshold of a calibration row ([TopTheta §3.1, Algorithm 1]).

    Pre-softmax: the quantile is taken on the scores a.  Post-softmax: the same
    quantile is taken on s = softmax(a) instead ([TopTheta §3.1], the remark
    after Figure 2).
    """
    if mode == PRE:
        return kth_largest(a, k)
    return kth_largest(row_softmax(a), k)


def collect_thresholds(Qc, Kc, row_len, k, mode, sets=None):
    """Gather the sets Theta_r of Algorithm 1 for one layer.

    Qc [N][Hq][R][d], Kc [N][Hkv][Nk][d]; query row i of sequence n sees keys
    0..row_len[i]-1.  Query head h reads KV head h // (Hq // Hkv) (GQA,
    [TopTheta §2.2]).  ``sets`` maps (h, L) to the list of observed thresholds
    and is extended in place, so several calls accumulate like one.
    """
    Qc = np.asarray(Qc, dtype=np.float64)
    Kc = np.asarray(Kc, dtype=np.float64)
    N, Hq, R, _ = Qc.shape
    Hkv = Kc.shape[1]
    g = Hq // Hkv
    if sets is None:
        sets = {}
    for n in range(N):
        for h in range(Hq):
            for i in range(R):
                L = int(row_len[i])
                if L <= k:               # Algorithm 1 starts at row k (reading c4)
                    continue
                a = row_scores(Qc[n, h, i], Kc[n, h // g], L)
                sets.setdefault((h, L), []).append(calibration_sample(a, k, mode))
    return sets


def finalize_thresholds(sets, Hq, Lmax, k, alpha):
    """theta_r = mean(Theta_r) + alpha * std(Theta_r) ([TopTheta §3.1, Algorithm 1]).

    Returns the table [Hq][Lmax]; entry L-1 belongs to rows with L keys.
    Rows with L <= k are dense (-inf, reading c4).  Uncalibrated rows take the
    nearest calibrated row id, ties to the shorter row ([Verdict], reading c5).
    """
    theta = np.full((Hq, Lmax), -np.inf)
    for h in range(Hq):
        seen = sorted(L for (hh, L) in sets if hh == h and L <= Lmax)
        value = {}
        for L in seen:
            obs = np.asarray(sets[(h, L)], dtype=np.float64)
            std = float(np.std(obs, ddof=1)) if obs.size > 1 else 0.0
            value[L] = float(np.mean(obs)) + alpha * std
        theta[h] = fill_row_ids(value, Lmax, k)
    return theta


def fill_row_ids(value, Lmax, k):
    """One head's row of the table from the calibrated row ids ``value`` (L -> theta).

    Rows with L <= k are dense (-inf, reading c4); a row id that was not
    calibrated takes the value of the nearest calibrated one, ties to the
    shorter row ([Verdict], reading c5); no calibrated row at all: dense.
    """
    row = np.full(Lmax, -np.inf)
    seen = sorted(value)
    if not seen:
        return row
    for L in range(k + 1, Lmax + 1):
        if L in value:
            row[L - 1] = value[L]
        else:
            best = min(seen, key=lambda c: (abs(c - L), c))
            row[L - 1] = value[best]
    return row


def fit_row_ids(value, Lmax, k, mode):
    """One head's row of the table from a function of ln L fitted to the
    calibrated row ids ``value`` (L -> theta), reading c22.

    y = theta (PRE) or ln theta (POST, theta > 0 only) is fitted by least
    squares with a line (degree min(1, n - 1)) in x = ln L over the n usable
    row ids; every L > k takes the fitted value (exp of it for POST, kept
    between the smallest normal float32 and the largest calibrated value, so an
    extrapolated post-softmax threshold never reaches 1, which would drop every
    key, nor 0, which would keep them all), L <= k stays dense, and a head
    without usable row ids is dense.
    """
    row = np.full(Lmax, -np.inf)
    pts = [(L, v) for L, v in sorted(value.items()) if L > k and (mode == PRE or v > 0)]
    if not pts:
        return row
    x = np.log(np.array([L for L, _ in pts], dtype=np.float64))
    y = np.array([v for _, v in pts], dtype=np.float64)
    if mode == POST:
        y = np.log(y)
    deg = min(1, len(pts) - 1)
    coef = np.polynomial.polynomial.polyfit(x, y, deg)
    Ls = np.arange(k + 1, Lmax + 1, dtype=np.float64)
    fitted = np.polynomial.polynomial.polyval(np.log(Ls), coef)
    if mode == POST:
        row[k:] = np.clip(np.exp(fitted), FLT32_MIN_NORMAL, max(v for _, v in pts))
    else:
        row[k:] = fitted
    return row


def finalize_fitted(sets, Hq, Lmax, k, alpha, mode):
    """theta [Hq][Lmax] from the fitted function of ln L (reading c22); the
    calibrated values are the Algorithm 1 statistics of ``finalize_thresholds``."""
    theta = np.full((Hq, Lmax), -np.inf)
    for h in range(Hq):
        value = {}
        for (hh, L), obs in sets.items():
            if hh != h or L > Lmax:
                continue
            obs = np.asarray(obs, dtype=np.float64)
            std = float(np.std(obs, ddof=1)) if obs.size > 1 else 0.0
            value[L] = float(np.mean(obs)) + alpha * std
        theta[h] = fit_row_ids(value, Lmax, k, mode)
    return theta


def calibrate_ref(Qc, Kc, row_len, k, mode, alpha, Lmax, fit=False):
    """Algorithm 1 for one layer: returns (theta [Hq][Lmax], sets); ``fit``
    replaces the nearest-row fill with the fitted function of ln L."""
    sets = collect_thresholds(Qc, Kc, row_len, k, mode)
    if fit:
        return finalize_fitted(sets, Qc.shape[1], Lmax, k, alpha, mode), sets
    return finalize_thresholds(sets, Qc.shape[1], Lmax, k, alpha), sets


# ---------------------------------------------------------------------------
# §3.2.1 estimator 1: offline-calibrated discarded sum E~.
# ---------------------------------------------------------------------------
def discarded_sum(a, theta):
    """E of one pre-softmax row under theta: the exponent sum of the keys that
    are not kept, in the units of Eq. 4 (row maximum subtracted, reading c8)."""
    a = np.asarray(a, dtype=np.float64)
    m = float(np.max(a))
    return float(np.exp(a[a < theta] - m).sum())


def collect_discarded(Qc, Kc, row_len, theta, sets=None):
    """Observed E of every calibration row under the (pre-softmax) threshold
    table theta [Hq][Lmax], keyed by (head, L); rows whose threshold is -inf
    keep everything and give no sample.  Indexing as in ``collect_thresholds``."""
    Qc = np.asarray(Qc, dtype=np.float64)
    Kc = np.asarray(Kc, dtype=np.float64)
    N, Hq, R, _ = Qc.shape
    g = Hq // Kc.shape[1]
    if sets is None:
        sets = {}
    for n in range(N):
        for h in range(Hq):
            for i in range(R):
                L = int(row_len[i])
                th = theta_for_row(theta[h], L)
                if not np.isfinite(th):
                    continue
                a = row_scores(Qc[n, h, i], Kc[n, h // g], L)
                sets.setdefault((h, L), []).append(discarded_sum(a, th))
    return sets


def finalize_discarded(sets, theta):
    """E~ [Hq][Lmax]: the mean of each sampled row id, the nearest sampled row
    id elsewhere (reading c5), 0 where theta is -inf or nothing was sampled
    (reading c20)."""
    Hq, Lmax = theta.shape
    et = np.zeros((Hq, Lmax))
    for h in range(Hq):
        value = {L: float(np.mean(v)) for (hh, L), v in sets.items() if hh == h and L <= Lmax}
        row = fill_row_ids(value, Lmax, 0)
        row[~np.isfinite(row)] = 0.0
        row[~np.isfinite(theta[h])] = 0.0
        et[h] = row
    return et


def calibrate_discarded_ref(Qc, Kc, row_len, theta):
    """Offline E~ table beside a pre-softmax theta table: (E~ [Hq][Lmax], sets)."""
    sets = collect_discarded(Qc, Kc, row_len, theta)
    return finalize_discarded(sets, np.asarray(theta, dtype=np.float64)), sets


# ---------------------------------------------------------------------------
# Appendix D, Algorithm 2: multi-k cumulative calibration (MKC).
# ---------------------------------------------------------------------------
def mkc_interval_sequence(x):
    """The interval sequence of one calibration row ([TopTheta App. D, Algorithm 2]).

    The row is sorted ascending into v_0..v_{r-1}; interval j is [v_j, v_{j+1})
    with effective k r-1-j, the number of elements of the row above any
    threshold inside it.  Returned as (t0, lo, hi) triples, j = 0..r-2.
    """
    v = np.sort(np.asarray(x, dtype=np.float64))
    r = v.shape[0]
    return [(r - 1 - j, float(v[j]), float(v[j + 1])) for j in range(r - 1)]


def mkc_collect(Qc, Kc, row_len, mode, sets=None):
    """The sets Theta_r of Algorithm 2 for one layer, keyed by (head, r).

    Every calibration row of every sequence contributes the interval sequence
    of its scores (PRE) or of its softmax values (POST; Figure 15 of the same
    appendix calibrates both).  Unlike Algorithm 1 no row is skipped: the
    target k is not known yet.  Same indexing as ``collect_thresholds``.
    """
    Qc = np.asarray(Qc, dtype=np.float64)
    Kc = np.asarray(Kc, dtype=np.float64)
    N, Hq, R, _ = Qc.shape
    g = Hq // Kc.shape[1]
    if sets is None:
        sets = {}
    for n in range(N):
        for h in range(Hq):
            for i in range(R):
                L = int(row_len[i])
                a = row_scores(Qc[n, h, i], Kc[n, h // g], L)
                x = a if mode == PRE else row_softmax(a)
                sets.setdefault((h, L), []).append(mkc_interval_sequence(x))
    return sets


def merge_intervals(seqs):
    """MergeIntervals of Algorithm 2: the step function k_bar(theta) of Eq. 8.

    On every elementary piece [lo, hi) between consecutive endpoints of all
    intervals, k_bar is the mean effective k of the intervals that contain the
    piece (at most one per sequence).  Pieces no interval contains are left
    out: k_bar is undefined there.  Returns (lo, hi, sum_t0, n_intervals)
    with the mean kept as an exact ratio of integers.
    """
    ends = np.unique(np.array([e for seq in seqs for (_, lo, hi) in seq for e in (lo, hi)],
                              dtype=np.float64))
    lo, hi = ends[:-1], ends[1:]
    tot = np.zeros(lo.shape[0], dtype=np.int64)
    cnt = np.zeros(lo.shape[0], dtype=np.int64)
    for seq in seqs:
        if not seq:
            continue
        t0 = np.array([t for (t, _, _) in seq], dtype=np.int64)
        a = np.array([x for (_, x, _) in seq], dtype=np.float64)
        b = np.array([x for (_, _, x) in seq], dtype=np.float64)
        # the last interval of the sequence starting at or below lo is the only
        # one that can contain the piece
        j = np.searchsorted(a, lo, side="right") - 1
        jj = np.maximum(j, 0)
        inside = (j >= 0) & (lo < b[jj])
        tot += np.where(inside, t0[jj], 0)
        cnt += inside
    keep = cnt > 0
    return [(float(l), float(h), int(t), int(c))
            for l, h, t, c in zip(lo[keep], hi[keep], tot[keep], cnt[keep])]


def mkc_theta(pieces, k):
    """theta_r(k), the inverse of k_bar_r at k (reading c19).

    The largest threshold up to which the calibration rows keep at least k
    elements on average: sup{theta : k_bar(theta) >= k}, the upper end of the
    highest piece whose mean effective k is at least k.  A threshold equal to
    that end keeps the same elements of the calibration rows as the inside of
    the piece, because an element equal to theta is kept (reading c1).  -inf
    when no piece reaches k (every row of length r <= k).
    """
    best = -np.inf
    for lo, hi, tot, cnt in pieces:
        if tot >= k * cnt:
            best = max(best, hi)
    return best


def mkc_ref(Qc, Kc, row_len, mode, ks, Hq_Lmax=None):
    """Algorithm 2 for one layer: theta [len(ks)][Hq][Lmax] and the sets.

    ``Hq_Lmax`` defaults to (Hq, max row length).  Each table is filled like
    Algorithm 1's (``fill_row_ids``): dense rows with L <= k, nearest
    calibrated row id elsewhere.
    """
    Qc = np.asarray(Qc, dtype=np.float64)
    Hq = Qc.shape[1]
    Lmax = int(max(row_len)) if Hq_Lmax is None else Hq_Lmax[1]
    sets = mkc_collect(Qc, Kc, row_len, mode)
    return mkc_finalize(sets, Hq, Lmax, ks), sets


def mkc_finalize(sets, Hq, Lmax, ks):
    """The per-k threshold tables from the merged sets (Algorithm 2, last step)."""
    merged = {key: merge_intervals(seqs) for key, seqs in sets.items() if key[1] <= Lmax}
    theta = np.full((len(ks), Hq, Lmax), -np.inf)
    for ki, k in enumerate(ks):
        for h in range(Hq):
            value = {L: mkc_theta(pc, k) for (hh, L), pc in merged.items() if hh == h and L > k}
            theta[ki, h] = fill_row_ids(value, Lmax, k)
    return theta


def theta_for_row(theta_row, L):
    """Look up the threshold of a row with L keys (readings c3, c5)."""
    Lmax = theta_row.shape[-1]
    return float(theta_row[min(L, Lmax) - 1])


# ---------------------------------------------------------------------------
# Inference on one attention row: threshold, SDC, VMC.
# ---------------------------------------------------------------------------
def attend_row(a, Vrows, theta, mode, sdc=SDC_NONE, vmc=False, mu=None,
               gamma=GAMMA, decide=None, e_tilde=0.0, keep=None):
    """Top-theta attention of one row.

    a      scores of the L visible keys (Eq. 1)
    Vrows  [L][d] value rows
    theta  the row's calibrated threshold (pre: on a, post: on s)
    decide optional bool [L]; inside the band |x - theta| <= 1e-3 |theta| the
           oracle adopts these decisions instead of its own.
    e_tilde the row's offline-calibrated estimate (SDC_OFFLINE, reading c20)
    keep   optional bool [L]: the final kept set, replacing the comparison with
           theta (a GQA group policy decided it, reading c21)

    Returns a dict with out [d], keep [L], kept (k~), band [L], m, Z, R, E, beta.
    """
    a = np.asarray(a, dtype=np.float64)
    V = np.asarray(Vrows, dtype=np.float64)
    L = a.shape[0]
    m = float(np.max(a))
    e = np.exp(a - m)                       # e^{a_j - max_l a_l}, Eq. 4
    Z = float(e.sum())
    s = e / Z                               # Eq. 2
    x = a if mode == PRE else s
    forced = keep
    keep = x >= theta                       # reading c1
    if np.isfinite(theta):
        band = np.abs(x - theta) <= BAND_REL * abs(theta)
    else:
        band = np.zeros(L, dtype=bool)
    if decide is not None:
        keep = np.where(band, np.asarray(decide, dtype=bool), keep)
    if forced is not None:
        keep = np.asarray(forced, dtype=bool).copy()
    kt = int(keep.sum())
    R = float(e[keep].sum())                # Eq. 4: selected exponent sum
    E = Z - R                               # Eq. 4: discarded exponent sum

    if mode == POST:
        # post-softmax: the kept s are not renormalised ([TopTheta §3.2.2 case i]);
        # SDC is the identity here (reading c16).
        s_kept = e[keep] / Z
    elif sdc == SDC_NONE:
        # softmax over the kept scores only ([TopTheta §3 Fig. 1, pre variant]).
        s_kept = e[keep] / R if R > 0 else np.zeros(kt)
    else:
        if sdc == SDC_EXACT:                # [TopTheta §3.2.1, estimator 3]
            E_est = E
        elif sdc == SDC_OFFLINE:            # [TopTheta §3.2.1, estimator 1], reading c20
            E_est = float(e_tilde)
        else:                               # [TopTheta §3.2.1, estimator 2], reading c8
            E_est = gamma * (L - kt) * math.exp(theta - m) if L > kt else 0.0
        # Eq. 4: softmax(a~)_i * R/(R + E~) = e_i / (R + E~)
        denom = R + E_est
        s_kept = e[keep] / denom if denom > 0 else np.zeros(kt)

    out = s_kept @ V[keep] if kt else np.zeros(V.shape[1])   # Eq. 7 first term
    vmc_eligible = mode == POST or sdc != SDC_NONE
    beta = 1.0 - float(s_kept.sum()) if vmc_eligible else 0.0  # Eq. 6, reading c10
    if vmc:
        out = out + beta * np.asarray(mu, dtype=np.float64)    # Eq. 7
    return dict(out=out, keep=keep, kept=kt, band=band, m=m, Z=Z, R=R, E=E,
                beta=beta)


def prefill_decisions(Q, K, theta_row, mode):
    """The keep and band decisions of every causal row of one head at once.

    Row i of a causal prefill sees keys 0..i (reading c6), so L = i + 1 and its
    threshold is theta_for_row(theta_row, L) (readings c3, c5).  The element
    x_ij is a_ij (PRE) or softmax(a_i)_j (POST) and is kept iff x_ij >= theta
    (reading c1); band marks |x - theta| <= 1e-3 |theta| for finite theta.
    These are attend_row's decisions, computed for all rows as whole matrices.
    Q, K [S][d]; returns keep [S][S], band [S][S] (False above the diagonal).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    S, d = Q.shape
    causal = np.tril(np.ones((S, S), dtype=bool))
    a = np.where(causal, (Q @ K[:S].T) / math.sqrt(d), -np.inf)
    theta = np.array([theta_for_row(theta_row, i + 1) for i in range(S)])[:, None]
    if mode == PRE:
        x = a
    else:
        e = np.exp(a - a.max(axis=1, keepdims=True))
        x = e / e.sum(axis=1, keepdims=True)
    keep = (x >= theta) & causal
    with np.errstate(invalid="ignore"):     # -inf - (-inf) above the diagonal of dense rows
        band = np.isfinite(theta) & (np.abs(x - theta) <= BAND_REL * np.abs(theta)) & causal
    return keep, band


def vmean_ref(Vrows):
    """Eq. 5: mean V row."""
    return np.mean(np.asarray(Vrows, dtype=np.float64), axis=0)


def vmean_update_ref(mu, n_old, new_rows):
    """Running mean of [TopTheta §3.2.2]: mu over n_old rows, then t rows appended."""
    new_rows = np.asarray(new_rows, dtype=np.float64)
    t = new_rows.shape[0]
    return (n_old * np.asarray(mu, dtype=np.float64) + new_rows.sum(axis=0)) / (n_old + t)


# ---------------------------------------------------------------------------
# Decode and prefill drivers (loops over rows, heads and batches).
# ---------------------------------------------------------------------------
def group_policy(keeps, policy, min_heads=1):
    """Final kept sets of the g heads of one GQA group ([TopTheta §4.6]).

    keeps [g][L] are the heads' own threshold decisions.  GQA_OWN keeps them
    (the paper's experiments); GQA_UNION gives every head the union, so the
    heads use V rows the group loads anyway; GQA_VOTE drops keys that fewer
    than ``min_heads`` heads keep (reading c21).
    """
    K = np.asarray(keeps, dtype=bool)
    if policy == GQA_OWN:
        return K.copy()
    if policy == GQA_UNION:
        return np.repeat(K.any(axis=0)[None, :], K.shape[0], axis=0)
    votes = K.sum(axis=0)
    return K & (votes >= min_heads)[None, :]


def decode_ref(q, Kc, Vc, seq_len, theta, mode, sdc=SDC_NONE, vmc=False,
               mu=None, gamma=GAMMA, decide=None, heads=None, e_tilde=None,
               gqa=GQA_OWN, gqa_min_heads=1):
    """One generated token per sequence ([TopTheta §2.2, generative decoding]).

    q [B][Hq][d]; Kc, Vc [B][Hkv][Nmax][d]; seq_len [B] (keys incl. the current
    token); theta [Hq][Lmax]; mu [B][Hkv][d] (when vmc); e_tilde [Hq][Lmax]
    (SDC_OFFLINE, looked up like theta); gqa / gqa_min_heads the group policy
    (``group_policy``; a policy other than GQA_OWN computes whole groups).
    ``decide`` is an
    optional bool [B][Hq][Nmax] of decisions adopted inside the band.
    ``heads`` optionally restricts the work to a list of (b, h) pairs.

    Returns dicts keyed by (b, h) of attend_row results, and the union size
    per (b, kv head) over the heads computed ([TopTheta §4.6]).
    """
    B, Hq, _ = q.shape
    Hkv = Kc.shape[1]
    g = Hq // Hkv
    res = {}
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(Hq)]
    if gqa != GQA_OWN:
        groups = sorted({(b, h // g) for (b, h) in heads})
        heads = [(b, kv * g + i) for (b, kv) in groups for i in range(g)]
    for (b, h) in heads:
        L = int(seq_len[b])
        kv = h // g
        a = row_scores(q[b, h], Kc[b, kv], L)
        th = theta_for_row(theta[h], L)
        dec = None if decide is None else decide[b, h, :L]
        et = 0.0 if e_tilde is None else theta_for_row(e_tilde[h], L)
        res[(b, h)] = attend_row(a, Vc[b, kv, :L], th, mode, sdc, vmc,
                                 None if mu is None else mu[b, kv], gamma, dec, et)
    if gqa != GQA_OWN:
        for (b, kv) in groups:
            L = int(seq_len[b])
            hs = [kv * g + i for i in range(g)]
            final = group_policy([res[(b, h)]["keep"] for h in hs], gqa, gqa_min_heads)
            for i, h in enumerate(hs):
                a = row_scores(q[b, h], Kc[b, kv], L)
                th = theta_for_row(theta[h], L)
                et = 0.0 if e_tilde is None else theta_for_row(e_tilde[h], L)
                res[(b, h)] = attend_row(a, Vc[b, kv, :L], th, mode, sdc, vmc,
                                         None if mu is None else mu[b, kv], gamma, None, et,
                                         keep=final[i])
    union = {}
    for (b, h), r in res.items():
        key = (b, h // g)
        u = union.get(key)
        union[key] = r["keep"].copy() if u is None else (u | r["keep"])
    vrows = {key: int(u.sum()) for key, u in union.items()}
    return res, vrows


def prefill_ref(Q, K, V, theta, mode, sdc=SDC_NONE, vmc=False, gamma=GAMMA,
                decide=None, rows=None, e_tilde=None):
    """Causal prefill ([TopTheta §2.2, prefill phase]); row i sees keys 0..i.

    Q [B][Hq][S][d]; K, V [B][Hkv][S][d]; theta [Hq][Lmax].  mu for row i is
    the mean of V rows 0..i (reading c11).  ``rows`` optionally restricts the
    work to a list of (b, h, i).  e_tilde [Hq][Lmax] as in ``decode_ref``.
    Returns a dict keyed by (b, h, i).
    """
    B, Hq, S, _ = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    res = {}
    if rows is None:
        rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(S)]
    for (b, h, i) in rows:
        L = i + 1
        kv = h // g
        a = row_scores(Q[b, h, i], K[b, kv], L)
        th = theta_for_row(theta[h], L)
        mu = vmean_ref(V[b, kv, :L]) if vmc else None
        dec = None if decide is None else decide[b, h, i, :L]
        et = 0.0 if e_tilde is None else theta_for_row(e_tilde[h], L)
        res[(b, h, i)] = attend_row(a, V[b, kv, :L], th, mode, sdc, vmc, mu,
                                    gamma, dec, et)
    return res


def tile_counts_ref(keep_rows, S, tile_m, tile_n):
    """Count causal (row block, key block) tiles and those holding a kept element.

    keep_rows maps row i to its bool mask over keys 0..i.  A tile is causal if
    any of its (i, j) has j <= i.  Returns (tiles_with_survivor, causal_tiles).
    """
    hit = 0
    total = 0
    for rb in range(0, S, tile_m):
        for cb in range(0, S, tile_n):
            if cb > min(rb + tile_m, S) - 1:
                continue
            total += 1
            any_kept = False
            for i in range(rb, min(rb + tile_m, S)):
                row = keep_rows[i]
                hi = min(cb + tile_n, i + 1)
                if hi > cb and bool(np.any(row[cb:hi])):
                    any_kept = True
                    break
            hit += int(any_kept)
    return hit, total


def output_rel_error(out, ref):
    """max |out - ref| / max |ref| over one output row (the parity metric)."""
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(np.asarray(out, dtype=np.float64) - ref)))
    return err / scale if scale > 0 else err
