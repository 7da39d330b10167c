"""The synthetic MoE-layer workloads: shapes, routing structure and input recipe.

Sizes follow the layers named on the expert-parallelism pages (Mixtral 8x7B,
DeepSeek-V3 routed experts, Switch-Base) plus a tiny all-float32 layer.  The
recipe for every workload: x ~ N(0,1); router weight ~ N(0, 1/h); expert
gate/up/down weights ~ N(0, 1/h); selection bias ~ U(-0.1, 0.1) where the
layer uses one; seed 0.  "N" is the Irwin-Hall normal of :mod:`synth`.

Layouts (row-major, the last index contiguous):
  x [T, h]; router weight [E, h]; w13 [E, 2I, h] (gate rows 0..I-1 then up rows
  I..2I-1 of each expert); w2 [E, h, I]; selection bias [E] float32; logit
  offset [E] float32; shared expert w13s [2*shared_I, h], w2s [h, shared_I]
  ~ N(0, 1/h).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import numpy as np

import synth


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    K: int
    I: int
    dtype: str                  # "f32" | "bf16"
    score: str                  # "softmax" | "sigmoid"
    renormalize: int = 1
    scale: float = 1.0
    n_groups: int = 0
    topk_groups: int = 0
    group_topn: int = 0
    capacity: int = 0           # <= 0: dropless
    pad: int = 0
    ep_size: int = 1
    sel_bias: Optional[Tuple[float, float]] = None   # U(lo, hi) selection bias
    zipf_s: Optional[float] = None                   # Zipf logit offsets
    shared_I: int = 0                                # shared expert intermediate (0: none)
    n_redundant: int = 0                             # EPLB: physical replicas beyond E (0: none)
    fp8: bool = False                                # experts in FP8 (E4M3, row scales)
    seed: int = 0

    @property
    def ds(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def rows(self) -> int:
        """Rows of the permuted buffer: T*K, or E*capacity when padded."""
        return self.E * self.capacity if (self.pad and self.capacity > 0) else self.T * self.K


def capacity_for(factor: float, T: int, K: int, E: int) -> int:
    return int(math.ceil(factor * T * K / E))


TINY = Workload("tiny_f32", T=256, h=256, E=8, K=2, I=512, dtype="f32", score="softmax",
                capacity=capacity_for(1.25, 256, 2, 8), ep_size=4)
MIXTRAL = Workload("mixtral_8x7b", T=4096, h=4096, E=8, K=2, I=14336, dtype="bf16",
                   score="softmax", ep_size=4)
DSV3 = Workload("deepseek_v3", T=4096, h=7168, E=256, K=8, I=2048, dtype="bf16",
                score="sigmoid", scale=2.5, n_groups=8, topk_groups=4, group_topn=2,
                ep_size=64, sel_bias=(-0.1, 0.1))
SWITCH = Workload("switch_base", T=16384, h=768, E=128, K=1, I=3072, dtype="bf16",
                  score="softmax", capacity=capacity_for(1.0, 16384, 1, 128), ep_size=16,
                  zipf_s=1.1)
DECODE = tuple(DSV3.replace(name=f"deepseek_v3_decode_T{t}", T=t) for t in (32, 256, 1024))
# The whole DeepSeek-V3 MoE block: the routed layer plus its one shared expert
# (intermediate 2048, like a routed expert), which every token passes through.
DSV3_BLOCK = DSV3.replace(name="deepseek_v3_block", shared_I=2048)

# The DeepSeek-V3 expert shape (h=7168, I=2048, ~128 rows per expert) with 16
# experts: 1.4 GB of weights, small enough for a profiler capture that replays a
# kernel many times, yet larger than the 126 MB L2.
PROFILE_DSV3 = DSV3.replace(name="deepseek_v3_e16_T256", T=256, E=16, ep_size=16)

# The same shape with 32 experts and 512 tokens (2.8 GB of weights): enough
# tiles for several waves of the grouped FFN on 148 SMs.
PROFILE_DSV3_E32 = DSV3.replace(name="deepseek_v3_e32_T512", T=512, E=32, ep_size=32)

ALL = {w.name: w for w in (TINY, MIXTRAL, DSV3, SWITCH) + DECODE}
# Expert-parallel load balancing: redundant replicas so that the physical
# experts fill every rank evenly (16 per 16 ranks for the Zipf-skewed Switch
# layer: 144 physical, 9 per rank; 64 for DeepSeek-V3: 320 physical, 5 per rank).
SWITCH_EPLB = SWITCH.replace(name="switch_base_eplb", n_redundant=16)
DSV3_EPLB = DSV3.replace(name="deepseek_v3_eplb", n_redundant=64)

# FP8 experts (E4M3 weights and expert inputs, float32 row scales) on the
# weight-bound DeepSeek-V3 shapes.
DSV3_FP8 = DSV3.replace(name="deepseek_v3_fp8", fp8=True)
DECODE_FP8 = DECODE[1].replace(name="deepseek_v3_decode_T256_fp8", fp8=True)

# Profiling cases: the DeepSeek-V3 token count and width with 16 experts (1.4 GB
# of weights; permuted buffers of 470 MB, larger than L2; 2048 rows per expert,
# so the tokens-as-M FFN) plus the shared expert; and the 32-expert case in FP8.
PROFILE_DSV3_E16_BLOCK = DSV3.replace(name="deepseek_v3_e16_T4096_block", E=16, ep_size=16, shared_I=2048)
PROFILE_DSV3_E32_FP8 = PROFILE_DSV3_E32.replace(name="deepseek_v3_e32_T512_fp8", fp8=True)

EXTRA = {w.name: w for w in (PROFILE_DSV3, PROFILE_DSV3_E32, DSV3_BLOCK, SWITCH_EPLB, DSV3_EPLB, DSV3_FP8,
                             DECODE_FP8, PROFILE_DSV3_E16_BLOCK, PROFILE_DSV3_E32_FP8)}


def sigma_in(w: Workload) -> float:
    return 1.0 / math.sqrt(w.h)


# ---------------------------------------------------------------- host side
def host_x(w: Workload, rows=None) -> np.ndarray:
    """x [T, h] (or the listed token rows), float32 or bf16 bits."""
    if rows is None:
        return synth.normal(w.seed, synth.TID_X, (w.T, w.h), 1.0, w.dtype)
    rows = np.asarray(rows, dtype=np.int64)
    idx = (rows[:, None] * w.h + np.arange(w.h)[None, :]).reshape(-1)
    return synth.normal_at(w.seed, synth.TID_X, idx, 1.0, w.dtype).reshape(len(rows), w.h)


def host_router_weight(w: Workload) -> np.ndarray:
    return synth.normal(w.seed, synth.TID_WR, (w.E, w.h), sigma_in(w), w.dtype)


def host_w13(w: Workload, e: int) -> np.ndarray:
    """Expert e's gate/up weight [2I, h]."""
    n = 2 * w.I * w.h
    return synth.normal(w.seed, synth.TID_W13, (2 * w.I, w.h), sigma_in(w), w.dtype, start=e * n)


def host_w2(w: Workload, e: int) -> np.ndarray:
    """Expert e's down weight [h, I]."""
    n = w.h * w.I
    return synth.normal(w.seed, synth.TID_W2, (w.h, w.I), sigma_in(w), w.dtype, start=e * n)


def host_w13s(w: Workload) -> np.ndarray:
    """The shared expert's gate/up weight [2*shared_I, h]."""
    return synth.normal(w.seed, synth.TID_W13S, (2 * w.shared_I, w.h), sigma_in(w), w.dtype)


def host_w2s(w: Workload) -> np.ndarray:
    """The shared expert's down weight [h, shared_I]."""
    return synth.normal(w.seed, synth.TID_W2S, (w.h, w.shared_I), sigma_in(w), w.dtype)


def host_sel_bias(w: Workload) -> Optional[np.ndarray]:
    if w.sel_bias is None:
        return None
    return synth.uniform(w.seed, synth.TID_SEL_BIAS, w.E, w.sel_bias[0], w.sel_bias[1])


_ZIPF_CACHE: dict = {}


def host_logit_offset(w: Workload) -> Optional[np.ndarray]:
    if w.zipf_s is None:
        return None
    key = (w.seed, w.E, w.zipf_s)
    if key not in _ZIPF_CACHE:
        _ZIPF_CACHE[key] = synth.zipf_logit_offsets(w.seed, w.E, w.zipf_s)
    return _ZIPF_CACHE[key]
