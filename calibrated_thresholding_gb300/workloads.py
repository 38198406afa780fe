"""The five synthetic workloads, shapes and seeds only.

They stand in for the pages' LLaMA-2/3 evaluations (Q&A suites, HumanEval,
LongBench), which need weights and datasets that are not available here;
inputs come from :mod:`calibrated_thresholding_gb300.synth` with these shapes.
"""
from __future__ import annotations

from dataclasses import dataclass

PRE, POST = 0, 1
SDC_NONE, SDC_EXACT, SDC_EXPTH = 0, 1, 2


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    n: int                 # tokens in each cache (incl. the current one)
    k: int
    mode: int = POST
    sdc: int = SDC_EXACT   # post-softmax ignores SDC (it already is the target)
    vmc: bool = True
    layers: int = 1
    k_first_layers: int = 0  # k of layers 0 and 1 when nonzero
    n_cal: int = 64
    cal_len: int = 0       # 0: calibrate decode rows at L = n; else prefill rows 1..cal_len
    values: str = "normal"

    def k_of(self, layer: int) -> int:
        return self.k_first_layers if (self.k_first_layers and layer < 2) else self.k


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    S: int
    k: int
    dtype: str = "bf16"
    n_cal: int = 8
    iid: bool = False      # iid N(0,1) Q, K, V instead of the peaked recipe


CFG1 = PrefillWorkload("single-head-fp32-S256-d64", B=1, Hq=1, Hkv=1, d=64, S=256, k=32,
                       dtype="f32", n_cal=16, iid=True)
CFG2 = DecodeWorkload("llama3-8b-decode-B16-n8192-32layers", B=16, Hq=32, Hkv=8, d=128, n=8192,
                      k=128, layers=32, k_first_layers=512, n_cal=64)
CFG3 = PrefillWorkload("llama3-8b-prefill-S4096", B=1, Hq=32, Hkv=8, d=128, S=4096, k=64, n_cal=8)
CFG4 = DecodeWorkload("llama3-70b-decode-B8-n32768", B=8, Hq=64, Hkv=8, d=128, n=32768, k=128,
                      n_cal=64, cal_len=4096)
CFG5 = DecodeWorkload("llama2-7b-mhsa-decode-n131072", B=1, Hq=32, Hkv=32, d=128, n=131072,
                      k=128, sdc=SDC_NONE, n_cal=16, values="lognormal_norm")

# k~/k buckets of the drift measurement (row length in keys)
BUCKETS = ((1, 511), (512, 2047), (2048, 8191), (8192, 1 << 30))
# ~16 lengths spread over the buckets (drift sweep of the 70B-shaped decode)
DRIFT_LENGTHS = (200, 300, 400, 500, 600, 900, 1400, 2000, 2100, 3000, 4096, 6000,
                 8200, 12000, 20000, 32768)
