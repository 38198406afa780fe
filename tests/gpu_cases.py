"""Seeded GPU inputs and GPU-side calibration used by the GPU parity tests."""
import numpy as np
import torch

from calibrated_thresholding_gb300 import synth, topt


def decode_case(seed, B, Hq, Hkv, d, Nmax, seq_len, values="normal"):
    gen = synth.generator(seed, "cuda")
    ch = synth.outlier_channels(seed, Hkv, d)
    K = synth.keys(gen, B, Hkv, Nmax, d, ch, device="cuda")
    V = synth.values(gen, B, Hkv, Nmax, d, values, device="cuda")
    q = synth.decode_queries(gen, K, Hq, seq_len)
    return q, K, V, ch


def prefill_case(seed, B, Hq, Hkv, d, S, dtype=torch.bfloat16, iid=False, channels=None):
    gen = synth.generator(seed, "cuda")
    if iid:
        Q = synth.iid_normal(gen, (B, Hq, S, d), "cuda", dtype)
        K = synth.iid_normal(gen, (B, Hkv, S, d), "cuda", dtype)
        V = synth.iid_normal(gen, (B, Hkv, S, d), "cuda", dtype)
        return Q, K, V
    ch = synth.outlier_channels(seed, Hkv, d) if channels is None else channels
    K = synth.keys(gen, B, Hkv, S, d, ch, device="cuda", dtype=dtype)
    V = synth.values(gen, B, Hkv, S, d, device="cuda", dtype=dtype)
    Q = synth.prefill_queries(gen, K, Hq, dtype=dtype)
    return Q, K, V


def calibrate_prefill_rows(seed, n_cal, Hq, Hkv, d, S, k, mode, Lmax, alpha=0.0,
                           dtype=torch.bfloat16, iid=False, channels=None):
    """theta [Hq][Lmax] from n_cal causal sequences of length S (all rows)."""
    cal = topt.Calibrator(Hq, Lmax, k, mode, alpha)
    row_len = torch.arange(1, S + 1, device="cuda", dtype=torch.int32)
    for n in range(n_cal):
        Q, K, _ = prefill_case(seed * 1000 + n, 1, Hq, Hkv, d, S, dtype, iid, channels)
        cal.add(Q, K, row_len, reset=(n == 0))
    return cal.finalize().clone(), cal


def calibrate_decode_rows(seed, n_cal, Hq, Hkv, d, L, k, mode, Lmax, channels, values="normal"):
    """theta from n_cal decode rows that see L keys each."""
    cal = topt.Calibrator(Hq, Lmax, k, mode)
    row_len = torch.tensor([L], device="cuda", dtype=torch.int32)
    for n in range(n_cal):
        gen = synth.generator(seed * 1000 + n, "cuda")
        K = synth.keys(gen, 1, Hkv, L, d, channels, device="cuda")
        q = synth.decode_queries(gen, K, Hq, [L])
        cal.add(q[:, :, None, :].contiguous(), K, row_len, reset=(n == 0))
    return cal.finalize().clone(), cal


def mask_words(n):
    return (n + 31) // 32


def np_seq(x):
    return np.asarray(x, dtype=np.int32)
