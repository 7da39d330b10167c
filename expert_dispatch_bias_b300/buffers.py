"""Device buffers for the C entry points, allocated through PyTorch (the library
itself never allocates)."""
from __future__ import annotations

import dataclasses

import torch

from . import _lib


def torch_dtype(cfg: _lib.MoeConfig) -> torch.dtype:
    return torch.float32 if cfg.dtype == _lib.MOE_F32 else torch.bfloat16


def alloc_workspace(cfg: _lib.MoeConfig, op: int, device="cuda", stream=None) -> torch.Tensor:
    """A zero-initialised workspace of moe_workspace_size(cfg, op) bytes."""
    n = _lib.moe_workspace_size(cfg, op)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    _lib.moe_workspace_init(ws, stream)
    return ws


@dataclasses.dataclass
class LayoutBuffers:
    counts: torch.Tensor
    kept: torch.Tensor
    offsets: torch.Tensor
    slot: torch.Tensor
    row_src: torch.Tensor
    n_ij: torch.Tensor
    rank_bytes: torch.Tensor
    stats: torch.Tensor     # 32 raw bytes holding a moe_layout_stats


def alloc_layout(cfg: _lib.MoeConfig, device="cuda") -> LayoutBuffers:
    R = _lib.moe_rows(cfg)
    N = cfg.ep_size
    i32 = dict(dtype=torch.int32, device=device)
    P = cfg.E + cfg.n_redundant  # physical experts (E without replicas)
    return LayoutBuffers(
        counts=torch.empty(P, **i32), kept=torch.empty(P, **i32), offsets=torch.empty(P + 1, **i32),
        slot=torch.empty(max(cfg.T * cfg.K, 1), **i32), row_src=torch.empty(max(R, 1), **i32),
        n_ij=torch.empty(N * N, dtype=torch.int64, device=device),
        rank_bytes=torch.empty(2 * N, dtype=torch.int64, device=device),
        stats=torch.empty(4, dtype=torch.int64, device=device))


def stats_dict(stats: torch.Tensor) -> dict:
    """Decodes the 32-byte moe_layout_stats."""
    raw = stats.cpu().contiguous().numpy().tobytes()
    s = _lib.MoeLayoutStats.from_buffer_copy(raw[:32])
    return {f: getattr(s, f) for f, _ in _lib.MoeLayoutStats._fields_}
