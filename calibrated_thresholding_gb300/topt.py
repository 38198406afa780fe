"""Thin Python binding of libtopt.so (argument marshalling only).

Every step of the computation runs in the CUDA library; this module passes
torch tensors' device pointers and the current CUDA stream through the C ABI
declared in ``include/topt.h``.  If the library is missing the first call
raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

PRE, POST = 0, 1
SDC_NONE, SDC_EXACT, SDC_EXPTH, SDC_OFFLINE = 0, 1, 2, 3
GQA_OWN, GQA_UNION, GQA_VOTE = 0, 1, 2
BF16, F32 = 0, 1
CALIB_RESET, CALIB_FINALIZE, CALIB_FIT = 1, 2, 4
GAMMA = 0.05

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported dtype", 3: "unsupported shape",
           4: "CUDA error", 5: "device wait timed out", 6: "workspace too small"}


class ToptError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn}: {_STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


i32, f32, vp, sz = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class DecodeArgs(ctypes.Structure):
    _fields_ = [("batch", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("cache_len", i32), ("theta_len", i32), ("mode", i32), ("sdc", i32), ("vmc", i32),
                ("gamma", f32), ("q", vp), ("k_cache", vp), ("v_cache", vp), ("seq_len", vp),
                ("theta", vp), ("e_tilde", vp), ("mu", vp), ("out", vp), ("kept", vp), ("vrows", vp), ("mask", vp),
                ("status", vp), ("workspace", vp), ("workspace_bytes", sz), ("events", vp * 3),
                ("gqa_policy", i32), ("gqa_min_heads", i32)]


class PrefillArgs(ctypes.Structure):
    _fields_ = [("batch", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("seq", i32), ("theta_len", i32), ("dtype", i32), ("mode", i32), ("sdc", i32),
                ("vmc", i32), ("gamma", f32), ("q", vp), ("k", vp), ("v", vp), ("theta", vp),
                ("e_tilde", vp), ("out", vp), ("kept", vp), ("mask", vp), ("tiles", vp), ("status", vp),
                ("workspace", vp), ("workspace_bytes", sz), ("events", vp * 2)]


class CalibArgs(ctypes.Structure):
    _fields_ = [("n_seqs", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("n_rows", i32), ("n_keys", i32), ("theta_len", i32), ("dtype", i32),
                ("mode", i32), ("k", i32), ("alpha", f32), ("flags", i32), ("q", vp),
                ("keys", vp), ("row_len", vp), ("acc", vp), ("count", vp), ("theta", vp),
                ("status", vp), ("workspace", vp), ("workspace_bytes", sz)]


class SdcCalibArgs(ctypes.Structure):
    _fields_ = [("n_seqs", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("n_rows", i32), ("n_keys", i32), ("theta_len", i32), ("dtype", i32),
                ("flags", i32), ("q", vp), ("keys", vp), ("row_len", vp), ("theta", vp),
                ("acc", vp), ("count", vp), ("e_tilde", vp), ("status", vp), ("workspace", vp),
                ("workspace_bytes", sz)]


class MkcArgs(ctypes.Structure):
    _fields_ = [("n_seqs", i32), ("n_q_heads", i32), ("n_kv_heads", i32), ("head_dim", i32),
                ("n_rows", i32), ("n_keys", i32), ("theta_len", i32), ("dtype", i32),
                ("mode", i32), ("n_k", i32), ("ks", vp), ("q", vp), ("keys", vp),
                ("row_len", vp), ("theta", vp), ("status", vp), ("workspace", vp),
                ("workspace_bytes", sz)]


class VmeanArgs(ctypes.Structure):
    _fields_ = [("batch", i32), ("n_kv_heads", i32), ("head_dim", i32), ("cache_len", i32),
                ("dtype", i32), ("n_new", i32), ("v_cache", vp), ("n_old", vp), ("mu", vp),
                ("status", vp), ("k_cache", vp), ("k_new", vp), ("v_new", vp)]


_lib = None
_lock = threading.Lock()

SYMBOLS = ["topt_decode_workspace", "topt_decode", "topt_decode_noalloc", "topt_prefill_workspace",
           "topt_prefill_tile_shape", "topt_prefill", "topt_prefill_test_timeout", "topt_calibrate_workspace",
           "topt_calibrate", "topt_calibrate_sdc_workspace", "topt_calibrate_sdc",
           "topt_calibrate_multik_workspace", "topt_calibrate_multik", "topt_select_kth", "topt_vmean_update", "topt_version",
           "topt_status_string"]


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libtopt.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(f"libtopt.so is not built ({path}); run "
                                   "calibrated_thresholding_gb300.build.build() first")
            L = ctypes.CDLL(path)
            P = ctypes.POINTER
            L.topt_decode_workspace.argtypes = [P(DecodeArgs), P(sz)]
            L.topt_decode.argtypes = [P(DecodeArgs), vp]
            L.topt_decode_noalloc.argtypes = [P(DecodeArgs), vp]
            L.topt_prefill_workspace.argtypes = [P(PrefillArgs), P(sz)]
            L.topt_prefill_tile_shape.argtypes = [P(PrefillArgs), P(i32), P(i32)]
            L.topt_prefill.argtypes = [P(PrefillArgs), vp]
            L.topt_prefill_test_timeout.argtypes = [P(PrefillArgs), vp]
            L.topt_calibrate_workspace.argtypes = [P(CalibArgs), P(sz)]
            L.topt_calibrate.argtypes = [P(CalibArgs), vp]
            L.topt_select_kth.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp]
            L.topt_vmean_update.argtypes = [P(VmeanArgs), vp]
            L.topt_status_string.restype = ctypes.c_char_p
            for name in SYMBOLS:
                if name not in ("topt_status_string",):
                    getattr(L, name).restype = ctypes.c_int
            L.topt_version.argtypes = []
            _lib = L
        return _lib


def _check(fn, code):
    if code != 0:
        raise ToptError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
def decode_args(q, k_cache, v_cache, seq_len, theta, *, mode, sdc=SDC_NONE, vmc=False, mu=None,
                gamma=GAMMA, out=None, kept=None, vrows=None, mask=None, status=None,
                workspace=None, e_tilde=None, gqa=GQA_OWN, gqa_min_heads=1):
    B, Hq, d = q.shape
    _, Hkv, Nmax, _ = k_cache.shape
    a = DecodeArgs()
    a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim = B, Hq, Hkv, d
    a.cache_len, a.theta_len = Nmax, theta.shape[-1]
    a.mode, a.sdc, a.vmc, a.gamma = int(mode), int(sdc), int(bool(vmc)), float(gamma)
    a.gqa_policy, a.gqa_min_heads = int(gqa), int(gqa_min_heads)
    a.q = _ptr(_dev(q, "q", torch.bfloat16))
    a.k_cache = _ptr(_dev(k_cache, "k_cache", torch.bfloat16))
    a.v_cache = _ptr(_dev(v_cache, "v_cache", torch.bfloat16))
    a.seq_len = _ptr(_dev(seq_len, "seq_len", torch.int32))
    a.theta = _ptr(_dev(theta, "theta", torch.float32))
    a.e_tilde = _ptr(_dev(e_tilde, "e_tilde", torch.float32))
    a.mu = _ptr(_dev(mu, "mu", torch.float32))
    a.out = _ptr(_dev(out, "out", torch.float32))
    a.kept = _ptr(_dev(kept, "kept", torch.int32))
    a.vrows = _ptr(_dev(vrows, "vrows", torch.int32))
    a.mask = _ptr(_dev(mask, "mask", torch.int32))
    a.status = _ptr(_dev(status, "status", torch.int32))
    if workspace is not None:
        a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
        a.workspace_bytes = workspace.numel()
    return a


def decode_workspace_bytes(a: DecodeArgs) -> int:
    n = sz(0)
    _check("topt_decode_workspace", lib().topt_decode_workspace(ctypes.byref(a), ctypes.byref(n)))
    return n.value


def decode_workspace(a: DecodeArgs, device) -> torch.Tensor:
    """A workspace for topt_decode (it needs no initialisation)."""
    return torch.empty(decode_workspace_bytes(a), device=device, dtype=torch.uint8)


def decode(q, k_cache, v_cache, seq_len, theta, *, mode, sdc=SDC_NONE, vmc=False, mu=None,
           gamma=GAMMA, out=None, kept=None, vrows=None, mask=None, status=None,
           workspace=None, stream=None, e_tilde=None, gqa=GQA_OWN, gqa_min_heads=1):
    """Top-theta decode through ``topt_decode``; see include/topt.h for shapes.

    Allocates (with torch) the outputs and the workspace that are not given.
    Returns a dict with out, kept, vrows (and mask when given).
    """
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty((B, Hq, d), device=dev, dtype=torch.float32)
    if kept is None:
        kept = torch.empty((B, Hq), device=dev, dtype=torch.int32)
    if vrows is None:
        vrows = torch.empty((B, Hkv), device=dev, dtype=torch.int32)
    a = decode_args(q, k_cache, v_cache, seq_len, theta, mode=mode, sdc=sdc, vmc=vmc, mu=mu,
                    gamma=gamma, out=out, kept=kept, vrows=vrows, mask=mask, status=status,
                    e_tilde=e_tilde, gqa=gqa, gqa_min_heads=gqa_min_heads)
    if workspace is None:
        workspace = decode_workspace(a, dev)
    a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
    a.workspace_bytes = workspace.numel()
    _check("topt_decode", lib().topt_decode(ctypes.byref(a), _stream(stream)))
    return dict(out=out, kept=kept, vrows=vrows, mask=mask)


def decode_noalloc(q, k_cache, v_cache, seq_len, theta, *, mode, sdc=SDC_NONE, vmc=False, mu=None,
                   gamma=GAMMA, out=None, kept=None, vrows=None, mask=None, status=None,
                   stream=None, e_tilde=None, gqa=GQA_OWN, gqa_min_heads=1):
    """Top-theta decode through ``topt_decode_noalloc`` (library-held scratch).

    For callers that must not allocate device scratch; see include/topt.h for
    the limit and the rule that calls must not overlap.  Outputs that are not
    given are allocated here with torch (the C entry point allocates nothing).
    """
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty((B, Hq, d), device=dev, dtype=torch.float32)
    if kept is None:
        kept = torch.empty((B, Hq), device=dev, dtype=torch.int32)
    if vrows is None:
        vrows = torch.empty((B, Hkv), device=dev, dtype=torch.int32)
    a = decode_args(q, k_cache, v_cache, seq_len, theta, mode=mode, sdc=sdc, vmc=vmc, mu=mu,
                    gamma=gamma, out=out, kept=kept, vrows=vrows, mask=mask, status=status,
                    e_tilde=e_tilde, gqa=gqa, gqa_min_heads=gqa_min_heads)
    _check("topt_decode_noalloc", lib().topt_decode_noalloc(ctypes.byref(a), _stream(stream)))
    return dict(out=out, kept=kept, vrows=vrows, mask=mask)


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
def prefill_args(q, k, v, theta, *, mode, sdc=SDC_NONE, vmc=False, gamma=GAMMA, out=None,
                 kept=None, mask=None, tiles=None, status=None, e_tilde=None):
    B, Hq, S, d = q.shape
    Hkv = k.shape[1]
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k and v must share one dtype")
    a = PrefillArgs()
    a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.seq = B, Hq, Hkv, d, S
    a.theta_len, a.dtype = theta.shape[-1], _dtype_code(q)
    a.mode, a.sdc, a.vmc, a.gamma = int(mode), int(sdc), int(bool(vmc)), float(gamma)
    a.q, a.k, a.v = _ptr(_dev(q, "q")), _ptr(_dev(k, "k")), _ptr(_dev(v, "v"))
    a.theta = _ptr(_dev(theta, "theta", torch.float32))
    a.e_tilde = _ptr(_dev(e_tilde, "e_tilde", torch.float32))
    a.out = _ptr(_dev(out, "out", torch.float32))
    a.kept = _ptr(_dev(kept, "kept", torch.int32))
    a.mask = _ptr(_dev(mask, "mask", torch.int32))
    a.tiles = _ptr(_dev(tiles, "tiles", torch.int64))
    a.status = _ptr(_dev(status, "status", torch.int32))
    return a


def prefill_workspace_bytes(a: PrefillArgs) -> int:
    n = sz(0)
    _check("topt_prefill_workspace", lib().topt_prefill_workspace(ctypes.byref(a), ctypes.byref(n)))
    return n.value


def prefill_tile_shape(a: PrefillArgs):
    r, c = i32(0), i32(0)
    _check("topt_prefill_tile_shape",
           lib().topt_prefill_tile_shape(ctypes.byref(a), ctypes.byref(r), ctypes.byref(c)))
    return r.value, c.value


def prefill(q, k, v, theta, *, mode, sdc=SDC_NONE, vmc=False, gamma=GAMMA, out=None, kept=None,
            mask=None, tiles=None, status=None, workspace=None, stream=None, e_tilde=None):
    """Causal Top-theta prefill through ``topt_prefill``."""
    B, Hq, S, d = q.shape
    dev = q.device
    if out is None:
        out = torch.empty((B, Hq, S, d), device=dev, dtype=torch.float32)
    if kept is None:
        kept = torch.empty((B, Hq, S), device=dev, dtype=torch.int32)
    a = prefill_args(q, k, v, theta, mode=mode, sdc=sdc, vmc=vmc, gamma=gamma, out=out, kept=kept,
                     mask=mask, tiles=tiles, status=status, e_tilde=e_tilde)
    need = prefill_workspace_bytes(a)
    if workspace is None and need > 0:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    if workspace is not None:
        a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
        a.workspace_bytes = workspace.numel()
    _check("topt_prefill", lib().topt_prefill(ctypes.byref(a), _stream(stream)))
    return dict(out=out, kept=kept, mask=mask, tiles=tiles)


# ---------------------------------------------------------------------------
# calibration
# ---------------------------------------------------------------------------
class Calibrator:
    """Accumulators of one layer's calibration [TopTheta §3.1, Algorithm 1].

    ``add`` runs topt_calibrate on a batch of calibration sequences; ``finalize``
    writes and returns theta [Hq][Lmax].  ``fit`` makes finalize write the
    fitted function of ln L (TOPT_CALIB_FIT) instead of the nearest-row fill.
    """

    def __init__(self, n_q_heads, theta_len, k, mode, alpha=0.0, device="cuda", fit=False):
        self.Hq, self.Lmax, self.k, self.mode, self.alpha = n_q_heads, theta_len, k, mode, alpha
        self.fit = bool(fit)
        self.acc = torch.zeros((2, n_q_heads, theta_len), device=device, dtype=torch.float64)
        self.count = torch.zeros((n_q_heads, theta_len), device=device, dtype=torch.int32)
        self.theta = torch.empty((n_q_heads, theta_len), device=device, dtype=torch.float32)
        self.device = device

    def _args(self, q, keys, row_len, flags, status):
        a = CalibArgs()
        a.n_q_heads, a.theta_len = self.Hq, self.Lmax
        a.mode, a.k, a.alpha, a.flags = int(self.mode), int(self.k), float(self.alpha), int(flags)
        a.acc, a.count, a.theta = _ptr(self.acc), _ptr(self.count), _ptr(self.theta)
        a.status = _ptr(_dev(status, "status", torch.int32))
        if q is None:
            a.n_seqs, a.n_kv_heads, a.head_dim, a.dtype = 0, self.Hq, 128, BF16
            return a
        N, Hq, R, d = q.shape
        a.n_seqs, a.n_kv_heads, a.head_dim, a.n_rows, a.n_keys = N, keys.shape[1], d, R, keys.shape[2]
        a.dtype = _dtype_code(q)
        a.q, a.keys = _ptr(_dev(q, "q")), _ptr(_dev(keys, "keys"))
        a.row_len = _ptr(_dev(row_len, "row_len", torch.int32))
        return a

    def add(self, q, keys, row_len, reset=False, status=None, workspace=None, stream=None):
        a = self._args(q, keys, row_len, CALIB_RESET if reset else 0, status)
        if workspace is None:
            n = sz(0)
            _check("topt_calibrate_workspace",
                   lib().topt_calibrate_workspace(ctypes.byref(a), ctypes.byref(n)))
            workspace = torch.empty(n.value, device=q.device, dtype=torch.uint8)
        a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
        a.workspace_bytes = workspace.numel()
        _check("topt_calibrate", lib().topt_calibrate(ctypes.byref(a), _stream(stream)))

    def finalize(self, status=None, stream=None):
        a = self._args(None, None, None, CALIB_FINALIZE | (CALIB_FIT if self.fit else 0), status)
        _check("topt_calibrate", lib().topt_calibrate(ctypes.byref(a), _stream(stream)))
        return self.theta


class SdcCalibrator:
    """Offline E~ of one layer beside a pre-softmax theta [TopTheta §3.2.1, estimator 1].

    ``add`` runs topt_calibrate_sdc on a batch of calibration sequences;
    ``finalize`` writes and returns E~ [Hq][Lmax] (pass it as ``e_tilde``
    with ``sdc=SDC_OFFLINE``).
    """

    def __init__(self, theta, device="cuda"):
        self.theta = _dev(theta, "theta", torch.float32)
        self.Hq, self.Lmax = theta.shape
        self.acc = torch.zeros((self.Hq, self.Lmax), device=device, dtype=torch.float64)
        self.count = torch.zeros((self.Hq, self.Lmax), device=device, dtype=torch.int32)
        self.e_tilde = torch.empty((self.Hq, self.Lmax), device=device, dtype=torch.float32)

    def _args(self, q, keys, row_len, flags, status):
        a = SdcCalibArgs()
        a.n_q_heads, a.theta_len, a.flags = self.Hq, self.Lmax, int(flags)
        a.theta, a.acc, a.count = _ptr(self.theta), _ptr(self.acc), _ptr(self.count)
        a.e_tilde = _ptr(self.e_tilde)
        a.status = _ptr(_dev(status, "status", torch.int32))
        if q is None:
            a.n_seqs, a.n_kv_heads, a.head_dim, a.dtype = 0, self.Hq, 128, BF16
            return a
        N, Hq, R, d = q.shape
        a.n_seqs, a.n_kv_heads, a.head_dim, a.n_rows, a.n_keys = N, keys.shape[1], d, R, keys.shape[2]
        a.dtype = _dtype_code(q)
        a.q, a.keys = _ptr(_dev(q, "q")), _ptr(_dev(keys, "keys"))
        a.row_len = _ptr(_dev(row_len, "row_len", torch.int32))
        return a

    def add(self, q, keys, row_len, reset=False, status=None, workspace=None, stream=None):
        a = self._args(q, keys, row_len, CALIB_RESET if reset else 0, status)
        if workspace is None:
            n = sz(0)
            _check("topt_calibrate_sdc_workspace",
                   lib().topt_calibrate_sdc_workspace(ctypes.byref(a), ctypes.byref(n)))
            workspace = torch.empty(n.value, device=q.device, dtype=torch.uint8)
        a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
        a.workspace_bytes = workspace.numel()
        _check("topt_calibrate_sdc", lib().topt_calibrate_sdc(ctypes.byref(a), _stream(stream)))

    def finalize(self, status=None, stream=None):
        a = self._args(None, None, None, CALIB_FINALIZE, status)
        _check("topt_calibrate_sdc", lib().topt_calibrate_sdc(ctypes.byref(a), _stream(stream)))
        return self.e_tilde


def calibrate_multik(q, keys, row_len, ks, mode, theta_len, theta=None, status=None,
                     workspace=None, stream=None):
    """Multi-k cumulative calibration of one layer [TopTheta App. D, Algorithm 2].

    q [N][Hq][R][d] and keys [N][Hkv][Nk][d] on the GPU, row_len [R] int32,
    ks [n_k] int32 target k values.  Returns theta [n_k][Hq][theta_len]:
    theta[ki] is the table for ks[ki] (topt_calibrate_multik).
    """
    N, Hq, R, d = q.shape
    ks = _dev(ks, "ks", torch.int32)
    n_k = ks.numel()
    if theta is None:
        theta = torch.empty((n_k, Hq, theta_len), device=q.device, dtype=torch.float32)
    a = MkcArgs()
    a.n_seqs, a.n_q_heads, a.n_kv_heads, a.head_dim = N, Hq, keys.shape[1], d
    a.n_rows, a.n_keys, a.theta_len = R, keys.shape[2], int(theta_len)
    a.dtype, a.mode, a.n_k = _dtype_code(q), int(mode), n_k
    a.ks, a.q, a.keys = _ptr(ks), _ptr(_dev(q, "q")), _ptr(_dev(keys, "keys"))
    a.row_len = _ptr(_dev(row_len, "row_len", torch.int32))
    a.theta = _ptr(_dev(theta, "theta", torch.float32))
    a.status = _ptr(_dev(status, "status", torch.int32))
    if workspace is None:
        n = sz(0)
        _check("topt_calibrate_multik_workspace",
               lib().topt_calibrate_multik_workspace(ctypes.byref(a), ctypes.byref(n)))
        workspace = torch.empty(n.value, device=q.device, dtype=torch.uint8)
    a.workspace = _ptr(_dev(workspace, "workspace", torch.uint8))
    a.workspace_bytes = workspace.numel()
    _check("topt_calibrate_multik", lib().topt_calibrate_multik(ctypes.byref(a), _stream(stream)))
    return theta


def select_kth(x, row_len, k, out=None, status=None, stream=None):
    """out[r] = k-th largest of x[r, :row_len[r]] through ``topt_select_kth``."""
    rows, stride = x.shape
    if out is None:
        out = torch.empty(rows, device=x.device, dtype=torch.float32)
    _dev(x, "x", torch.float32)
    _dev(row_len, "row_len", torch.int32)
    _check("topt_select_kth", lib().topt_select_kth(
        _ptr(x), rows, stride, _ptr(row_len), int(k), _ptr(out),
        _ptr(_dev(status, "status", torch.int32)), _stream(stream)))
    return out


def vmean_args(v_cache, n_old, n_new, mu, status=None, k_cache=None, k_new=None, v_new=None) -> VmeanArgs:
    """The topt_vmean_update arguments for these tensors (validated once; the
    struct can be passed to ``lib().topt_vmean_update`` for every step).
    k_new / v_new [B][Hkv][n_new][d] (optional): the step's new rows, appended
    to k_cache / v_cache at rows n_old.. by the same launch."""
    B, Hkv, Nmax, d = v_cache.shape
    a = VmeanArgs()
    a.batch, a.n_kv_heads, a.head_dim, a.cache_len = B, Hkv, d, Nmax
    a.dtype, a.n_new = _dtype_code(v_cache), int(n_new)
    a.v_cache = _ptr(_dev(v_cache, "v_cache"))
    a.n_old = _ptr(_dev(n_old, "n_old", torch.int32))
    a.mu = _ptr(_dev(mu, "mu", torch.float32))
    a.status = _ptr(_dev(status, "status", torch.int32))
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t is not None and (tuple(t.shape) != (B, Hkv, int(n_new), d) or t.dtype != v_cache.dtype
                              or not t.is_contiguous()):
            raise ValueError(f"{name}: a contiguous [{B}][{Hkv}][{int(n_new)}][{d}] {v_cache.dtype} tensor")
    if k_new is not None and (k_cache is None or tuple(k_cache.shape) != tuple(v_cache.shape)
                              or k_cache.dtype != v_cache.dtype):
        raise ValueError("k_new needs k_cache shaped and typed as v_cache")
    a.k_cache = _ptr(_dev(k_cache, "k_cache"))
    a.k_new = _ptr(_dev(k_new, "k_new"))
    a.v_new = _ptr(_dev(v_new, "v_new"))
    return a


def vmean_update(v_cache, n_old, n_new, mu, status=None, stream=None, k_cache=None, k_new=None, v_new=None):
    """mu <- running mean after appending rows n_old..n_old+n_new-1 (topt_vmean_update);
    with k_new / v_new the rows are first written into k_cache / v_cache."""
    a = vmean_args(v_cache, n_old, n_new, mu, status, k_cache, k_new, v_new)
    _check("topt_vmean_update", lib().topt_vmean_update(ctypes.byref(a), _stream(stream)))
    return mu
