"""GPU check of topt_decode_noalloc, the decode entry point that allocates nothing.

Some callers cannot allocate device memory themselves (a fixed memory budget
set at start-up, or a host framework whose allocator owns all device memory);
this entry point uses a scratch array the library holds instead of a caller
workspace.  Its results must match topt_decode's on the same inputs, on two
calls in a row (the array keeps the previous call's contents, so the second
call checks that nothing left over from the first one leaks into it).

The file name puts it last in collection order, so a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle.topt_ref as ref
from calibrated_thresholding_gb300 import build, synth, topt

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-3   # the output tolerance of the parity tests


def _inputs(seed, B, Hq, Hkv, d, n, seq):
    gen = synth.generator(seed, "cuda")
    ch = synth.outlier_channels(seed, Hkv, d)
    K = synth.keys(gen, B, Hkv, n, d, ch, device="cuda")
    V = synth.values(gen, B, Hkv, n, d, device="cuda")
    q = synth.decode_queries(gen, K, Hq, seq)
    seq_len = torch.tensor(seq, device="cuda", dtype=torch.int32)
    mu = torch.stack([V[b, :, :L].float().mean(dim=1) for b, L in enumerate(seq)])
    theta = torch.full((Hq, n), 1e-3, device="cuda")      # post-softmax threshold
    theta[:, :16] = float("-inf")
    return q, K, V, seq_len, mu, theta


def _max_rel_err(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    scale = b.abs().amax(dim=-1).clamp_min(1e-30)
    return float(((a - b).abs().amax(dim=-1) / scale).max())


def test_noalloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("CUDA GPU not available")
    build.build()
    L = topt.lib()
    B, Hq, Hkv, d, n = 3, 16, 4, 128, 1500
    q, K, V, seq_len, mu, theta = _inputs(7, B, Hq, Hkv, d, n, [1500, 733, 1])

    # reference: the workspace entry point
    want = topt.decode(q, K, V, seq_len, theta, mode=ref.POST, vmc=True, mu=mu)
    torch.cuda.synchronize()

    # the no-allocation entry point, called through the C ABI twice in a row
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((B, Hq, d), float("nan"), device="cuda")
        kept = torch.full((B, Hq), -1, device="cuda", dtype=torch.int32)
        vrows = torch.full((B, Hkv), -1, device="cuda", dtype=torch.int32)
        a = topt.decode_args(q, K, V, seq_len, theta, mode=ref.POST, vmc=True, mu=mu, out=out,
                             kept=kept, vrows=vrows)
        assert a.workspace is None
        rc = L.topt_decode_noalloc(ctypes.byref(a), stream)
        assert rc == 0, topt.ToptError("topt_decode_noalloc", rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"call {call}"
        assert _max_rel_err(out, want["out"]) <= OUT_TOL, f"call {call}"
        assert torch.equal(kept.cpu(), want["kept"].cpu()), f"call {call}"
        assert torch.equal(vrows.cpu(), want["vrows"].cpu()), f"call {call}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("CUDA GPU not available")
    build.build()
    L = topt.lib()
    a = topt.DecodeArgs()
    a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim = 8, 64, 8, 128
    a.cache_len, a.theta_len, a.mode = 32768, 32768, ref.POST
    need = ctypes.c_size_t(0)
    assert L.topt_decode_workspace(ctypes.byref(a), ctypes.byref(need)) == 0
    assert need.value > 32 << 20
    # pointers that pass the host checks; nothing is launched for this shape
    dummy = torch.empty(16, device="cuda", dtype=torch.uint8)
    for f in ("q", "k_cache", "v_cache", "seq_len", "theta", "out"):
        setattr(a, f, ctypes.c_void_p(dummy.data_ptr()))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.topt_decode_noalloc(ctypes.byref(a), stream) == 6   # TOPT_EWORKSPACE
