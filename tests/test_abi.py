"""Host-side checks of the C ABI (no GPU needed).

The library loads, exports every function include/topt.h declares, and
rejects bad arguments on the host before touching the GPU.
"""
import ctypes
import os
import re

import pytest

from calibrated_thresholding_gb300 import build, topt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return topt.lib()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:topt_status|int32_t|const char\*)\s+(topt_\w+)\s*\(",
                                    text, flags=re.M))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("topt_calibrate", "topt_prefill", "topt_decode", "topt_vmean_update"):
        assert n in names
    assert set(topt.SYMBOLS) >= names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    assert L.topt_version() == 100
    assert L.topt_status_string(3) == b"unsupported shape"


def _decode_args(**kw):
    a = topt.DecodeArgs()
    a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim = 2, 8, 2, 128
    a.cache_len, a.theta_len, a.mode, a.sdc, a.vmc, a.gamma = 64, 64, topt.POST, 0, 0, 0.05
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_decode_validation_rejects_on_host(L):
    n = ctypes.c_size_t(0)
    assert L.topt_decode_workspace(ctypes.byref(_decode_args()), ctypes.byref(n)) == 0
    assert n.value > 0
    # workspace covers the fp32 score block of every head
    assert n.value >= 2 * 8 * 64 * 4
    bad = [dict(head_dim=96), dict(n_q_heads=6, n_kv_heads=4), dict(n_q_heads=32, n_kv_heads=2),
           dict(batch=0), dict(cache_len=0)]
    for kw in bad:
        assert L.topt_decode_workspace(ctypes.byref(_decode_args(**kw)), ctypes.byref(n)) == 3, kw
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(mode=7)), ctypes.byref(n)) == 1
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(sdc=4)), ctypes.byref(n)) == 1
    # the offline estimator is a valid mode; its table is checked at the call
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(sdc=3)), ctypes.byref(n)) == 0
    # GQA policies: unknown policy and VOTE without a head count are refused
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(gqa_policy=3)), ctypes.byref(n)) == 1
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(gqa_policy=2)), ctypes.byref(n)) == 1
    assert L.topt_decode_workspace(ctypes.byref(_decode_args(gqa_policy=2, gqa_min_heads=2)),
                                   ctypes.byref(n)) == 0
    # NULL tensors: rejected before any launch
    assert L.topt_decode(ctypes.byref(_decode_args()), None) == 1


def test_prefill_and_calibrate_validation(L):
    a = topt.PrefillArgs()
    a.batch, a.n_q_heads, a.n_kv_heads, a.head_dim, a.seq, a.theta_len = 1, 4, 2, 64, 100, 100
    a.dtype, a.mode = topt.BF16, topt.PRE
    r, c = ctypes.c_int32(0), ctypes.c_int32(0)
    assert L.topt_prefill_tile_shape(ctypes.byref(a), ctypes.byref(r), ctypes.byref(c)) == 0
    assert r.value > 0 and c.value > 0
    a.dtype = 9
    assert L.topt_prefill(ctypes.byref(a), None) == 2
    a.dtype = topt.F32
    assert L.topt_prefill(ctypes.byref(a), None) == 1          # NULL tensors

    c = topt.CalibArgs()
    c.n_seqs, c.n_q_heads, c.n_kv_heads, c.head_dim, c.n_rows, c.n_keys = 2, 4, 2, 64, 10, 10
    c.theta_len, c.dtype, c.mode, c.k, c.alpha = 10, topt.BF16, topt.PRE, 0, 0.0
    assert L.topt_calibrate(ctypes.byref(c), None) == 1        # k < 1
    c.k = 3
    n = ctypes.c_size_t(0)
    assert L.topt_calibrate_workspace(ctypes.byref(c), ctypes.byref(n)) == 0
    assert n.value >= 2 * 4 * 10 * 10 * 4
    c.flags = 8
    assert L.topt_calibrate(ctypes.byref(c), None) == 1
    assert L.topt_select_kth(None, 3, 4, None, 1, None, None, None) == 1

    e = topt.SdcCalibArgs()
    e.n_seqs, e.n_q_heads, e.n_kv_heads, e.head_dim, e.n_rows, e.n_keys = 2, 4, 2, 64, 10, 10
    e.theta_len, e.dtype = 10, topt.BF16
    assert L.topt_calibrate_sdc_workspace(ctypes.byref(e), ctypes.byref(n)) == 0
    assert n.value >= 2 * 4 * 10 * 10 * 4
    assert L.topt_calibrate_sdc(ctypes.byref(e), None) == 1    # NULL theta / accumulators
    e.n_kv_heads = 3
    assert L.topt_calibrate_sdc_workspace(ctypes.byref(e), ctypes.byref(n)) == 3

    m = topt.MkcArgs()
    m.n_seqs, m.n_q_heads, m.n_kv_heads, m.head_dim, m.n_rows, m.n_keys = 2, 4, 2, 64, 10, 10
    m.theta_len, m.dtype, m.mode, m.n_k = 10, topt.BF16, topt.PRE, 3
    assert L.topt_calibrate_multik_workspace(ctypes.byref(m), ctypes.byref(n)) == 0
    assert n.value >= 2 * 10 * 10 * 4 + 3 * 4 * 10 * 4
    assert L.topt_calibrate_multik(ctypes.byref(m), None) == 1  # NULL tensors
    m.n_k = 0
    assert L.topt_calibrate_multik_workspace(ctypes.byref(m), ctypes.byref(n)) == 1
    m.n_k, m.n_keys = 3, 1 << 20
    assert L.topt_calibrate_multik_workspace(ctypes.byref(m), ctypes.byref(n)) == 3

    v = topt.VmeanArgs()
    v.batch, v.n_kv_heads, v.head_dim, v.cache_len, v.dtype, v.n_new = 1, 1, 64, 8, topt.BF16, 9
    assert L.topt_vmean_update(ctypes.byref(v), None) == 3     # t > capacity


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(topt, "_lib", None)
    monkeypatch.setattr(topt, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        topt.lib()


STRUCTS = {"topt_decode_args": "DecodeArgs", "topt_prefill_args": "PrefillArgs",
           "topt_calib_args": "CalibArgs", "topt_sdc_calib_args": "SdcCalibArgs",
           "topt_mkc_args": "MkcArgs", "topt_vmean_args": "VmeanArgs"}


def test_header_is_c99_and_binding_layouts_match(tmp_path):
    """include/topt.h compiles as strict C99, and every argument struct of the
    ctypes binding has the C struct's size and field offsets."""
    gcc = "gcc"
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "topt.h"', "int main(void) {"]
    for cname, pyname in STRUCTS.items():
        cls = getattr(topt, pyname)
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    import subprocess
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for ln in out:
        if ln:
            parts = ln.split()
            got[(parts[0], parts[1])] = int(parts[2])
    for cname, pyname in STRUCTS.items():
        cls = getattr(topt, pyname)
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)
