"""Device side of the seeded input generator (ctypes binding of synth/libsynth.so).

Fills torch tensors in device memory with exactly the values synth's host
functions produce for the same (seed, tensor id, element index)."""
from __future__ import annotations

import ctypes
import math
import os

import torch

import synth
from synth import workloads

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python expert_dispatch_bias_b300/build.py`")
_lib = ctypes.CDLL(_LIB_PATH)
_lib.synth_fill_normal.restype = ctypes.c_int
_lib.synth_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64,
                                   ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p]
_lib.synth_fill_uniform.restype = ctypes.c_int
_lib.synth_fill_uniform.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                    ctypes.c_double, ctypes.c_double, ctypes.c_void_p]


def fill_normal(t: torch.Tensor, seed: int, tensor_id: int, sigma: float, start: int = 0) -> torch.Tensor:
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.float32, torch.bfloat16)
    rc = _lib.synth_fill_normal(t.data_ptr(), t.numel(), 1 if t.dtype == torch.bfloat16 else 0, seed, tensor_id,
                                start, float(sigma), torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal: cuda error {rc}")
    return t


def fill_uniform(t: torch.Tensor, seed: int, tensor_id: int, lo: float, hi: float) -> torch.Tensor:
    assert t.is_cuda and t.is_contiguous() and t.dtype == torch.float32
    rc = _lib.synth_fill_uniform(t.data_ptr(), t.numel(), seed, tensor_id, float(lo), float(hi) - float(lo),
                                 torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_uniform: cuda error {rc}")
    return t


def shared_weights(w: workloads.Workload, device="cuda") -> dict:
    """The shared expert's w13s [2*shared_I, h] and w2s [h, shared_I] on the device."""
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    s = workloads.sigma_in(w)
    return {"w13s": fill_normal(torch.empty(2 * w.shared_I, w.h, dtype=dt, device=device), w.seed, synth.TID_W13S, s),
            "w2s": fill_normal(torch.empty(w.h, w.shared_I, dtype=dt, device=device), w.seed, synth.TID_W2S, s)}


def layer_inputs(w: workloads.Workload, device="cuda", weights=True) -> dict:
    """The workload's inputs on the device: x, w_r, w13, w2, sel_bias, logit_offset."""
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    s = workloads.sigma_in(w)
    out = {
        "x": fill_normal(torch.empty(w.T, w.h, dtype=dt, device=device), w.seed, synth.TID_X, 1.0),
        "w_r": fill_normal(torch.empty(w.E, w.h, dtype=dt, device=device), w.seed, synth.TID_WR, s),
        "sel_bias": None,
        "logit_offset": None,
    }
    if weights:
        out["w13"] = fill_normal(torch.empty(w.E, 2 * w.I, w.h, dtype=dt, device=device), w.seed, synth.TID_W13, s)
        out["w2"] = fill_normal(torch.empty(w.E, w.h, w.I, dtype=dt, device=device), w.seed, synth.TID_W2, s)
    if weights and w.shared_I > 0:
        out.update(shared_weights(w, device))
    if w.sel_bias is not None:
        out["sel_bias"] = fill_uniform(torch.empty(w.E, dtype=torch.float32, device=device), w.seed,
                                       synth.TID_SEL_BIAS, *w.sel_bias)
    off = workloads.host_logit_offset(w)
    if off is not None:
        out["logit_offset"] = torch.from_numpy(off).to(device)
    return out
