"""ctypes binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every function below passes device pointers, sizes
and the current CUDA stream to the C entry point of the same name and raises
MoeError on a non-zero status.  No step of the layer runs here.  If the
library is missing the import fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_SOFTMAX, MOE_SIGMOID = 0, 1
MOE_OP_LAYOUT, MOE_OP_FFN, MOE_OP_LAYER, MOE_OP_LAYER_HOST = 0, 1, 2, 3
MOE_OP_SHARED, MOE_OP_BLOCK, MOE_OP_BLOCK_HOST = 4, 5, 6
MOE_OP_FFN_FP8, MOE_OP_LAYER_FP8, MOE_OP_LOGITS, MOE_OP_FFN_COMBINE = 7, 8, 9, 10

STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
    4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_TIMEOUT",
    7: "MOE_ERR_DEVICE_BAD_INDEX",
}

# Every symbol the header declares (checked by the tests).
EXPORTS = (
    "moe_status_string", "moe_validate_config", "moe_rows", "moe_workspace_size", "moe_workspace_init",
    "moe_router_logits", "moe_route", "moe_dispatch_layout", "moe_dispatch_layout_static", "moe_permute",
    "moe_grouped_ffn",
    "moe_combine", "moe_layer_forward", "moe_layer_forward_host", "moe_check",
    "moe_shared_ffn", "moe_combine_add", "moe_block_forward", "moe_block_forward_host",
    "moe_eplb_plan", "moe_eplb_map", "moe_grouped_ffn_mapped", "moe_layer_forward_eplb",
    "moe_quantize_fp8", "moe_permute_fp8", "moe_grouped_ffn_fp8", "moe_layer_forward_fp8",
    "moe_grouped_ffn_gather", "moe_grouped_ffn_combine", "moe_launch_count",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("T", c_int32), ("h", c_int32), ("E", c_int32), ("K", c_int32), ("I", c_int32),
        ("dtype", c_int32), ("score", c_int32), ("renormalize", c_int32), ("scale", c_float),
        ("n_groups", c_int32), ("topk_groups", c_int32), ("group_topn", c_int32),
        ("capacity", c_int32), ("pad", c_int32), ("ep_size", c_int32), ("shared_I", c_int32),
        ("n_redundant", c_int32),
    ]


class MoeLayoutStats(ctypes.Structure):
    _fields_ = [("kept_total", c_int64), ("dropped", c_int64), ("offdiag_rows", c_int64),
                ("experts_touched", c_int32), ("balancedness", c_float)]


class MoeLayerOut(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("logits", "topk_ids", "topk_w", "counts", "kept", "offsets", "slot",
                                         "row_src", "n_ij", "rank_bytes", "stats", "stage_events")]


# Stages of the layer calls (moe_layer_stage); stage_events holds one event more.
LAYER_STAGES = ("logits", "route", "eplb_map", "layout", "permute", "ffn", "shared", "combine")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python expert_dispatch_bias_b300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    cfgp = POINTER(MoeConfig)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [c_int32]),
        "moe_validate_config": (c_int32, [cfgp]),
        "moe_rows": (c_int32, [cfgp, POINTER(c_int64)]),
        "moe_workspace_size": (c_int32, [cfgp, c_int32, POINTER(c_size_t)]),
        "moe_workspace_init": (c_int32, [c_void_p, c_size_t, c_void_p]),
        "moe_router_logits": (c_int32, [cfgp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                        c_void_p]),
        "moe_route": (c_int32, [cfgp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
        "moe_dispatch_layout": (c_int32, [cfgp] + [c_void_p] * 10 + [c_size_t, c_void_p]),
        "moe_dispatch_layout_static": (c_int32, [cfgp] + [c_void_p] * 9 + [c_void_p]),
        "moe_permute": (c_int32, [cfgp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
        "moe_grouped_ffn": (c_int32, [cfgp] + [c_void_p] * 7 + [c_size_t, c_void_p]),
        "moe_combine": (c_int32, [cfgp, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
        "moe_layer_forward": (c_int32, [cfgp] + [c_void_p] * 9 + [c_size_t, c_void_p]),
        "moe_layer_forward_host": (c_int32, [cfgp] + [c_void_p] * 8 + [c_size_t, c_void_p]),
        "moe_check": (c_int32, [c_void_p]),
        "moe_launch_count": (ctypes.c_uint64, []),
        "moe_shared_ffn": (c_int32, [cfgp] + [c_void_p] * 5 + [c_size_t, c_void_p]),
        "moe_combine_add": (c_int32, [cfgp] + [c_void_p] * 6),
        "moe_block_forward": (c_int32, [cfgp] + [c_void_p] * 11 + [c_size_t, c_void_p]),
        "moe_block_forward_host": (c_int32, [cfgp] + [c_void_p] * 10 + [c_size_t, c_void_p]),
        "moe_eplb_plan": (c_int32, [c_int32, c_int32, c_int32] + [c_void_p] * 5),
        "moe_eplb_map": (c_int32, [cfgp] + [c_void_p] * 5),
        "moe_grouped_ffn_mapped": (c_int32, [cfgp] + [c_void_p] * 8 + [c_size_t, c_void_p]),
        "moe_layer_forward_eplb": (c_int32, [cfgp] + [c_void_p] * 11 + [c_size_t, c_void_p]),
        "moe_quantize_fp8": (c_int32, [c_int64, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
        "moe_permute_fp8": (c_int32, [cfgp] + [c_void_p] * 5),
        "moe_grouped_ffn_fp8": (c_int32, [cfgp] + [c_void_p] * 10 + [c_size_t, c_void_p]),
        "moe_layer_forward_fp8": (c_int32, [cfgp] + [c_void_p] * 11 + [c_size_t, c_void_p]),
        "moe_grouped_ffn_gather": (c_int32, [cfgp] + [c_void_p] * 8 + [c_size_t, c_void_p]),
        "moe_grouped_ffn_combine": (c_int32, [cfgp] + [c_void_p] * 11 + [c_size_t, c_void_p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MoeError(status, where)


def make_config(T, h, E, K, I, dtype="bf16", score="softmax", renormalize=1, scale=1.0, n_groups=0,
                topk_groups=0, group_topn=0, capacity=0, pad=0, ep_size=1, shared_I=0, n_redundant=0) -> MoeConfig:
    return MoeConfig(T, h, E, K, I, MOE_F32 if dtype in ("f32", MOE_F32) else MOE_BF16,
                     MOE_SIGMOID if score in ("sigmoid", MOE_SIGMOID) else MOE_SOFTMAX,
                     int(renormalize), float(scale), n_groups, topk_groups, group_topn, capacity, pad, ep_size,
                     shared_I, n_redundant)


def config_from(w) -> MoeConfig:
    """MoeConfig from any object with the layer's attributes (e.g. a synth Workload)."""
    return make_config(w.T, w.h, w.E, w.K, w.I, w.dtype, w.score, w.renormalize, w.scale, w.n_groups,
                       w.topk_groups, w.group_topn, w.capacity, w.pad, w.ep_size, getattr(w, "shared_I", 0),
                       getattr(w, "n_redundant", 0))


# ------------------------------------------------------------------ the C entry points
def moe_validate_config(cfg: MoeConfig) -> int:
    return lib.moe_validate_config(ctypes.byref(cfg))


def moe_rows(cfg: MoeConfig) -> int:
    r = c_int64()
    _check(lib.moe_rows(ctypes.byref(cfg), ctypes.byref(r)), "moe_rows")
    return r.value


def moe_workspace_size(cfg: MoeConfig, op: int) -> int:
    n = c_size_t()
    _check(lib.moe_workspace_size(ctypes.byref(cfg), op, ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_init(ws, stream=None) -> None:
    _check(lib.moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_workspace_init")


def moe_router_logits(cfg, x, w_r, logit_offset, logits, workspace, stream=None) -> None:
    """workspace: moe_workspace_size(cfg, MOE_OP_LOGITS) bytes (alloc_workspace)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.moe_router_logits(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(logits),
                                 _ptr(workspace), nbytes, _stream(stream)), "moe_router_logits")


def moe_route(cfg, logits, sel_bias, topk_ids, topk_w, stream=None) -> None:
    _check(lib.moe_route(ctypes.byref(cfg), _ptr(logits), _ptr(sel_bias), _ptr(topk_ids), _ptr(topk_w),
                         _stream(stream)), "moe_route")


def moe_dispatch_layout(cfg, topk_ids, counts, kept, offsets, slot, row_src, n_ij, rank_bytes, stats, workspace,
                        stream=None) -> None:
    _check(lib.moe_dispatch_layout(ctypes.byref(cfg), _ptr(topk_ids), _ptr(counts), _ptr(kept), _ptr(offsets),
                                   _ptr(slot), _ptr(row_src), _ptr(n_ij), _ptr(rank_bytes), _ptr(stats),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "moe_dispatch_layout")


def moe_dispatch_layout_static(cfg, topk_ids, counts, kept, offsets, slot, row_src, n_ij, rank_bytes, stats,
                               stream=None) -> None:
    """moe_dispatch_layout for callers that cannot allocate: no workspace, the
    library's fixed scratch array instead (see include/moe.h)."""
    _check(lib.moe_dispatch_layout_static(ctypes.byref(cfg), _ptr(topk_ids), _ptr(counts), _ptr(kept),
                                          _ptr(offsets), _ptr(slot), _ptr(row_src), _ptr(n_ij), _ptr(rank_bytes),
                                          _ptr(stats), _stream(stream)), "moe_dispatch_layout_static")


def moe_permute(cfg, x, slot, row_src, xp, stream=None) -> None:
    _check(lib.moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(slot), _ptr(row_src), _ptr(xp), _stream(stream)),
           "moe_permute")


def moe_grouped_ffn(cfg, xp, offsets, kept, w13, w2, yp, workspace, stream=None) -> None:
    _check(lib.moe_grouped_ffn(ctypes.byref(cfg), _ptr(xp), _ptr(offsets), _ptr(kept), _ptr(w13), _ptr(w2),
                               _ptr(yp), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream)), "moe_grouped_ffn")


def moe_grouped_ffn_combine(cfg, xp, offsets, kept, w13, w2, row_src, slot, topk_w, yp, y, workspace,
                            stream=None) -> None:
    """workspace: moe_workspace_size(cfg, MOE_OP_FFN_COMBINE) bytes, zero-filled (alloc_workspace)."""
    _check(lib.moe_grouped_ffn_combine(ctypes.byref(cfg), _ptr(xp), _ptr(offsets), _ptr(kept), _ptr(w13), _ptr(w2),
                                       _ptr(row_src), _ptr(slot), _ptr(topk_w), _ptr(yp), _ptr(y), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_grouped_ffn_combine")


def moe_grouped_ffn_gather(cfg, x, row_src, offsets, kept, w13, w2, yp, workspace, stream=None) -> None:
    _check(lib.moe_grouped_ffn_gather(ctypes.byref(cfg), _ptr(x), _ptr(row_src), _ptr(offsets), _ptr(kept),
                                      _ptr(w13), _ptr(w2), _ptr(yp), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_grouped_ffn_gather")


def moe_combine(cfg, yp, slot, topk_w, y, stream=None) -> None:
    _check(lib.moe_combine(ctypes.byref(cfg), _ptr(yp), _ptr(slot), _ptr(topk_w), _ptr(y), _stream(stream)),
           "moe_combine")


def moe_layer_forward(cfg, x, w_r, logit_offset, sel_bias, w13, w2, y, out: Optional[MoeLayerOut], workspace,
                      stream=None) -> None:
    _check(lib.moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias),
                                 _ptr(w13), _ptr(w2), _ptr(y), ctypes.byref(out) if out is not None else None,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward")


def moe_layer_forward_host(cfg, x_host, w_r, logit_offset, sel_bias, w13, w2, y_host, workspace,
                           stream=None) -> None:
    _check(lib.moe_layer_forward_host(ctypes.byref(cfg), _ptr(x_host), _ptr(w_r), _ptr(logit_offset),
                                      _ptr(sel_bias), _ptr(w13), _ptr(w2), _ptr(y_host), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward_host")


def moe_shared_ffn(cfg, x, w13s, w2s, ys, workspace, stream=None) -> None:
    _check(lib.moe_shared_ffn(ctypes.byref(cfg), _ptr(x), _ptr(w13s), _ptr(w2s), _ptr(ys), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)), "moe_shared_ffn")


def moe_combine_add(cfg, yp, slot, topk_w, ys, y, stream=None) -> None:
    _check(lib.moe_combine_add(ctypes.byref(cfg), _ptr(yp), _ptr(slot), _ptr(topk_w), _ptr(ys), _ptr(y),
                               _stream(stream)), "moe_combine_add")


def moe_block_forward(cfg, x, w_r, logit_offset, sel_bias, w13, w2, w13s, w2s, y, out: Optional[MoeLayerOut],
                      workspace, stream=None) -> None:
    _check(lib.moe_block_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias),
                                 _ptr(w13), _ptr(w2), _ptr(w13s), _ptr(w2s), _ptr(y),
                                 ctypes.byref(out) if out is not None else None, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)), "moe_block_forward")


def moe_block_forward_host(cfg, x_host, w_r, logit_offset, sel_bias, w13, w2, w13s, w2s, y_host, workspace,
                           stream=None) -> None:
    _check(lib.moe_block_forward_host(ctypes.byref(cfg), _ptr(x_host), _ptr(w_r), _ptr(logit_offset),
                                      _ptr(sel_bias), _ptr(w13), _ptr(w2), _ptr(w13s), _ptr(w2s), _ptr(y_host),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "moe_block_forward_host")


def moe_eplb_plan(E: int, ep_size: int, n_redundant: int, counts) -> dict:
    """Host-only replica plan (see include/moe.h); counts: a sequence of E ints.
    Returns numpy arrays rep_offsets, rep_phys, phys_to_log, rank_load."""
    import numpy as np
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int64))
    P = E + n_redundant
    out = {"rep_offsets": np.zeros(E + 1, np.int32), "rep_phys": np.zeros(P, np.int32),
           "phys_to_log": np.zeros(P, np.int32), "rank_load": np.zeros(ep_size, np.int64)}
    _check(lib.moe_eplb_plan(E, ep_size, n_redundant, c.ctypes.data, out["rep_offsets"].ctypes.data,
                             out["rep_phys"].ctypes.data, out["phys_to_log"].ctypes.data,
                             out["rank_load"].ctypes.data), "moe_eplb_plan")
    return out


def moe_eplb_map(cfg, topk_ids, rep_offsets, rep_phys, phys_ids, stream=None) -> None:
    _check(lib.moe_eplb_map(ctypes.byref(cfg), _ptr(topk_ids), _ptr(rep_offsets), _ptr(rep_phys), _ptr(phys_ids),
                            _stream(stream)), "moe_eplb_map")


def moe_grouped_ffn_mapped(cfg, xp, offsets, kept, phys_to_log, w13, w2, yp, workspace, stream=None) -> None:
    _check(lib.moe_grouped_ffn_mapped(ctypes.byref(cfg), _ptr(xp), _ptr(offsets), _ptr(kept), _ptr(phys_to_log),
                                      _ptr(w13), _ptr(w2), _ptr(yp), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_grouped_ffn_mapped")


def moe_layer_forward_eplb(cfg, x, w_r, logit_offset, sel_bias, w13, w2, rep_offsets, rep_phys, phys_to_log, y,
                           out: Optional[MoeLayerOut], workspace, stream=None) -> None:
    _check(lib.moe_layer_forward_eplb(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias),
                                      _ptr(w13), _ptr(w2), _ptr(rep_offsets), _ptr(rep_phys), _ptr(phys_to_log),
                                      _ptr(y), ctypes.byref(out) if out is not None else None, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward_eplb")


def moe_quantize_fp8(src, codes, scales, stream=None) -> None:
    """Row quantisation of a 2-D bf16/float32 tensor into E4M3 codes (uint8) and
    float32 row scales (see include/moe.h)."""
    rows, cols = src.shape[0], src.numel() // max(src.shape[0], 1)
    import torch
    dt = MOE_BF16 if src.dtype == torch.bfloat16 else MOE_F32
    _check(lib.moe_quantize_fp8(rows, cols, dt, _ptr(src), _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8")


def moe_permute_fp8(cfg, x, slot, xq, sx, stream=None) -> None:
    _check(lib.moe_permute_fp8(ctypes.byref(cfg), _ptr(x), _ptr(slot), _ptr(xq), _ptr(sx), _stream(stream)),
           "moe_permute_fp8")


def moe_grouped_ffn_fp8(cfg, xq, sx, offsets, kept, w13q, s13, w2q, s2, yp, workspace, stream=None) -> None:
    _check(lib.moe_grouped_ffn_fp8(ctypes.byref(cfg), _ptr(xq), _ptr(sx), _ptr(offsets), _ptr(kept), _ptr(w13q),
                                   _ptr(s13), _ptr(w2q), _ptr(s2), _ptr(yp), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_grouped_ffn_fp8")


def moe_layer_forward_fp8(cfg, x, w_r, logit_offset, sel_bias, w13q, s13, w2q, s2, y, out: Optional[MoeLayerOut],
                          workspace, stream=None) -> None:
    _check(lib.moe_layer_forward_fp8(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias),
                                     _ptr(w13q), _ptr(s13), _ptr(w2q), _ptr(s2), _ptr(y),
                                     ctypes.byref(out) if out is not None else None, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_layer_forward_fp8")


def moe_check(stream=None) -> int:
    """Synchronises the stream; returns the status (does not raise)."""
    return lib.moe_check(_stream(stream))


def moe_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib.moe_launch_count())


def layer_out(stage_events=None, **tensors) -> MoeLayerOut:
    """Optional outputs of the layer calls.  ``stage_events``: MOE_LAYER_STAGES + 1
    torch.cuda.Event objects or None, each event already recorded once (torch
    creates the CUDA event on its first record); the layer records them around
    its stages and skips the None entries."""
    o = MoeLayerOut()
    for k, v in tensors.items():
        setattr(o, k, _ptr(v))
    if stage_events is not None:
        if len(stage_events) != len(LAYER_STAGES) + 1:
            raise ValueError(f"stage_events needs {len(LAYER_STAGES) + 1} events")
        handles = [None if e is None else e.cuda_event for e in stage_events]
        if not all(h for h, e in zip(handles, stage_events) if e is not None):
            raise ValueError("record every stage event once before passing it (torch creates it lazily)")
        o._events = (c_void_p * len(handles))(*handles)   # kept alive with the struct
        o.stage_events = ctypes.cast(o._events, c_void_p)
    return o
