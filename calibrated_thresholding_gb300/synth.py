"""Seeded synthetic inputs shaped like the workloads of the Top-theta pages.

This module holds random draws and bf16 rounding only; none of the method's
arithmetic lives here.  Both the CUDA path and the float64 oracle consume the
same tensors produced here (the oracle gets them converted to float64).

Distributions (the pages evaluate LLaMA-2/3 models on Q&A and LongBench; no
weights or datasets are available, so these stand in for them):

* keys: iid N(0, 1); per KV head four channels, drawn once from the workload
  seed and shared by calibration and evaluation, are scaled by 8 (outlier
  channels of real K caches).
* queries: 0.5 * (a uniformly chosen earlier key of the same KV head) + N(0, 1),
  which makes each score row peaked.
* values: iid N(0, 1), or (long-context decode) a random direction with a
  per-token log-normal(0, 0.5) norm.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch


def seed_of(*parts) -> int:
    """A stable 63-bit seed from any printable parts (workload, role, index...)."""
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_channels(workload_seed: int, n_kv_heads: int, d: int, count: int = 4) -> np.ndarray:
    """[Hkv][count] distinct channel indices per KV head."""
    rng = np.random.default_rng(workload_seed)
    return np.stack([rng.choice(d, size=count, replace=False) for _ in range(n_kv_heads)])


def iid_normal(gen, shape, device="cpu", dtype=torch.float32):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype)


def keys(gen, B, Hkv, n, d, channels, scale=8.0, device="cpu", dtype=torch.bfloat16):
    """K [B][Hkv][n][d]: N(0, 1) with the given outlier channels scaled."""
    x = torch.randn((B, Hkv, n, d), generator=gen, device=device, dtype=torch.float32)
    mult = torch.ones((Hkv, d), device=device, dtype=torch.float32)
    idx = torch.as_tensor(np.asarray(channels), device=device, dtype=torch.int64)
    mult.scatter_(1, idx, float(scale))
    x.mul_(mult[None, :, None, :])
    return x.to(dtype)


def values(gen, B, Hkv, n, d, kind="normal", device="cpu", dtype=torch.bfloat16):
    """V [B][Hkv][n][d]: N(0, 1), or ``kind='lognormal_norm'``."""
    z = torch.randn((B, Hkv, n, d), generator=gen, device=device, dtype=torch.float32)
    if kind == "lognormal_norm":
        r = torch.exp(0.5 * torch.randn((B, Hkv, n, 1), generator=gen, device=device,
                                        dtype=torch.float32))
        z = z / z.norm(dim=-1, keepdim=True) * r
    elif kind != "normal":
        raise ValueError(kind)
    return z.to(dtype)


def decode_queries(gen, K, Hq, seq_len, dtype=torch.bfloat16):
    """q [B][Hq][d]: 0.5 * K[b, kv, j] + N(0, 1), j uniform over [0, L_b - 1)."""
    B, Hkv, _, d = K.shape
    g = Hq // Hkv
    dev = K.device
    L = torch.as_tensor(np.asarray(seq_len), device=dev, dtype=torch.int64)
    span = torch.clamp(L - 1, min=1)
    u = torch.rand((B, Hq), generator=gen, device=dev, dtype=torch.float64)
    j = torch.minimum((u * span[:, None]).to(torch.int64), (span - 1)[:, None])
    kv = torch.arange(Hq, device=dev) // g
    src = K[torch.arange(B, device=dev)[:, None], kv[None, :], j].float()
    noise = torch.randn((B, Hq, d), generator=gen, device=dev, dtype=torch.float32)
    return (0.5 * src + noise).to(dtype)


def prefill_queries(gen, K, Hq, dtype=torch.bfloat16):
    """Q [B][Hq][S][d]: row t is 0.5 * K[b, kv, j] + N(0, 1), j uniform over [0, t)."""
    B, Hkv, S, d = K.shape
    g = Hq // Hkv
    dev = K.device
    t = torch.arange(S, device=dev, dtype=torch.int64)
    span = torch.clamp(t, min=1)
    u = torch.rand((B, Hq, S), generator=gen, device=dev, dtype=torch.float64)
    j = torch.minimum((u * span).to(torch.int64), span - 1)
    kv = (torch.arange(Hq, device=dev) // g)[None, :, None].expand(B, Hq, S)
    bb = torch.arange(B, device=dev)[:, None, None].expand(B, Hq, S)
    src = K[bb, kv, j].float()
    noise = torch.randn((B, Hq, S, d), generator=gen, device=dev, dtype=torch.float32)
    return (0.5 * src + noise).to(dtype)


def as_f64(x) -> np.ndarray:
    """The exact values of a (bf16 or fp32) tensor as a float64 numpy array."""
    return x.detach().to("cpu", torch.float64).numpy()
