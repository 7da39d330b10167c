"""Shared helpers of the GPU parity tests: host/device conversions, oracle inputs
and cached oracle results.  Nothing here runs a step of the layer."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth
from synth import workloads


def np_of(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def dev_of(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.to_f64(a, dtype) if a.dtype != np.float64 else a


def half_ulp(r: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of the storage type at each value: the error
    that rounding an exact result to that type alone may add."""
    mant = 7 if dtype == "bf16" else 23
    mag = np.maximum(np.abs(r), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(mag)).astype(np.int64) - mant - 1)


def rel_err(got: np.ndarray, ref: np.ndarray, dtype: str, storage_rounding: bool = True) -> float:
    """max |got - ref| / rms(ref) in float64, where ``ref`` is the oracle's exact
    (unrounded) value.  With ``storage_rounding`` each element's error is first
    reduced by half an ulp of the output type at ``ref``: a result stored in
    bf16 cannot be closer than that to the exact value, whatever the arithmetic
    (at max|y| just above a power of two that alone is about 5.5 * 2**-8 of the
    RMS of a Gaussian-like output, more than 2e-2)."""
    g, r = f64(got, dtype), f64(ref, dtype)
    if r.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(r * r))
    d = np.abs(g - r)
    if storage_rounding:
        d = np.maximum(d - half_ulp(r, dtype), 0.0)
    return float(d.max() / max(rms, 1e-30))


# Max-abs error relative to the output RMS: 2e-2 for bf16 data with float32
# accumulation, 1e-4 for float32 data.
TOL = {"f32": 1e-4, "bf16": 2e-2}


@functools.lru_cache(maxsize=8)
def host_inputs(name: str):
    w = workloads.ALL[name] if isinstance(name, str) else name
    return {"x": workloads.host_x(w), "w_r": workloads.host_router_weight(w),
            "sel_bias": workloads.host_sel_bias(w), "logit_offset": workloads.host_logit_offset(w)}


@functools.lru_cache(maxsize=8)
def oracle_routing(name: str):
    """Oracle logits, routing and layout of a named workload (cached)."""
    w = workloads.ALL[name]
    h = host_inputs(name)
    L = oracle.router_logits(h["x"], h["w_r"], w.dtype, h["logit_offset"])
    ids, wts, keys, allowed = oracle.route(L, w, h["sel_bias"])
    lay = oracle.dispatch_layout(ids, w)
    return {"logits": L, "ids": ids, "w": wts, "keys": keys, "allowed": allowed, "layout": lay}


def expert_weights(w: workloads.Workload, e: int):
    return workloads.host_w13(w, e), workloads.host_w2(w, e)


# Routing differences seen by the end-to-end tests, printed in pytest's terminal
# summary (tests/conftest.py): (test, tokens, near-tie tokens of the oracle,
# tokens the GPU routed differently, tokens compared in float).
NEAR_TIE_LOG = []


def log_near_ties(name: str, tokens: int, near_tie: int, routed_differently: int, compared: int) -> None:
    NEAR_TIE_LOG.append((name, tokens, near_tie, routed_differently, compared))
