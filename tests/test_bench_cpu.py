"""The arithmetic behind bench.py's reported numbers, on CPU: flop and byte
counts of one call checked against sizes worked out by hand for the
LLaMA-3-8B-shaped workloads, and the rule that recorded DRAM traffic is
reported only for the kernel sources it was measured on."""
import os
import sys
from types import SimpleNamespace

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from calibrated_thresholding_gb300 import workloads  # noqa: E402


def test_prefill_flop_counts():
    wl = workloads.CFG3                                  # 1 x 4096 rows, 32 heads, d = 128
    causal_elems = 32 * 4096 * 4097 // 2                 # 268,500,992 (i, j <= i) pairs
    assert causal_elems == 268_500_992
    assert bench.causal_flops(wl) == 4 * 128 * causal_elems
    assert bench.kept_elem_flops(wl, 0) == 2 * 128 * causal_elems
    assert bench.kept_elem_flops(wl, 1000) - bench.kept_elem_flops(wl, 0) == 2 * 128 * 1000
    # 128 x 128 tiles: 32 heads x 528 causal tiles = 16,896; every tile executed gives the
    # 141.7 GFLOP per launch of the prefill profile
    st = SimpleNamespace(wl=wl, tile_rows=128, tile_keys=128)
    tiles = 32 * (32 * 33 // 2)
    assert tiles == 16_896
    useful, issued = bench.prefill_flops(st, (tiles, tiles))
    assert abs(useful - 141.73e9) < 0.01e9
    assert issued == useful * 1.5


def test_decode_algorithmic_bytes():
    wl = workloads.CFG2                                  # B = 16, 8 KV heads, 8192 tokens, d = 128
    vrows = torch.full((wl.B, wl.Hkv), 300, dtype=torch.int32)
    st = SimpleNamespace(wl=wl, layers=2, vrows=[vrows, vrows * 0])
    k_bytes, per_layer = bench.algorithmic_bytes(st)
    assert k_bytes == 268_435_456                        # the whole K cache of one layer, bf16
    small = 16 * 32 * 128 * 2 + 16 * 8 * 128 * 4 + 16 * 32 * 128 * 4   # q, mu, out
    theta = 16 * 32 * 4
    assert per_layer[1] == k_bytes + theta + small       # nothing kept: no V row read
    assert per_layer[0] - per_layer[1] == 16 * 8 * 300 * 128 * 2


def test_recorded_traffic_only_for_the_measured_sources():
    for known in (bench.DECODE_TRAFFIC, bench.PREFILL_TRAFFIC):
        rec = {"sources": known["sources"], "source_sha256": bench.source_sha(known["sources"]),
               "bytes_per_launch": 123}
        assert bench.recorded_traffic(rec) == 123
        rec["source_sha256"] = "0" * 64
        assert bench.recorded_traffic(rec) is None
