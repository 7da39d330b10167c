"""moe_dispatch_layout_static: the dispatch layout for callers that cannot allocate.

Some callers cannot call cudaMalloc and have no workspace to lend, for example
code inside a host framework that owns every device allocation through its own
allocator, or a latency-critical loop that cannot afford the implicit
synchronisation of cudaMalloc.  For them the library offers a layout call whose
look-back scratch is a fixed device array inside the library.  These tests call
it through the C ABI and require its outputs to equal those of the ordinary
moe_dispatch_layout (bit for bit: every output is an index or a count), on two
calls in a row, and check that layouts too large for the fixed array are refused.

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before it.
"""
import ctypes

import pytest
import torch

import expert_dispatch_bias_b300 as moe
import synth
from synth import workloads

pytestmark = pytest.mark.gpu


def _outputs(buf):
    return [t.cpu().clone() for t in (buf.counts, buf.kept, buf.offsets, buf.slot, buf.row_src, buf.n_ij,
                                      buf.rank_bytes, buf.stats)]


def _call_static(cfg, ids, buf):
    st = moe.lib.moe_dispatch_layout_static(
        ctypes.byref(cfg), ids.data_ptr(), buf.counts.data_ptr(), buf.kept.data_ptr(), buf.offsets.data_ptr(),
        buf.slot.data_ptr(), buf.row_src.data_ptr(), buf.n_ij.data_ptr(), buf.rank_bytes.data_ptr(),
        buf.stats.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, moe.STATUS[st]


CASES = [
    workloads.DSV3,                                                                   # 16 tiles, EP=64
    workloads.SWITCH.replace(capacity=128, pad=1),                                    # drops + pad rows
    workloads.Workload("ragged", T=1000, h=64, E=60, K=3, I=64, dtype="bf16", score="softmax", capacity=45,
                       ep_size=6),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_static_layout_matches_workspace_layout(w):
    cfg = moe.config_from(w)
    ids = torch.from_numpy(synth.uniform_topk_ids(11, synth.TID_TEST + 20, w.T, w.E, w.K)).cuda()
    ref_buf = moe.alloc_layout(cfg)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYOUT)
    moe.moe_dispatch_layout(cfg, ids, ref_buf.counts, ref_buf.kept, ref_buf.offsets, ref_buf.slot, ref_buf.row_src,
                            ref_buf.n_ij, ref_buf.rank_bytes, ref_buf.stats, ws)
    assert moe.moe_check() == 0
    ref = _outputs(ref_buf)
    for _ in range(2):                      # two calls in a row share the fixed array
        buf = moe.alloc_layout(cfg)
        for t in (buf.slot, buf.row_src, buf.n_ij, buf.counts):
            t.fill_(-7)
        _call_static(cfg, ids, buf)
        assert moe.moe_check() == 0
        got = _outputs(buf)
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


SEQUENCE = [
    workloads.DSV3,                                                                   # two passes, 16 tiles
    workloads.DSV3.replace(name="dsv3_decode_T256", T=256),                           # one block (2048 assignments)
    workloads.Workload("mid", T=3000, h=64, E=60, K=4, I=64, dtype="bf16", score="softmax", capacity=220,
                       ep_size=6),                                                    # two passes, 3 tiles, drops
    workloads.DSV3,
    workloads.Workload("mid", T=3000, h=64, E=60, K=4, I=64, dtype="bf16", score="softmax", capacity=220,
                       ep_size=6),
]


def test_static_layout_sequence_of_mixed_configurations():
    """Each call starts clean whatever the previous call left in the shared array:
    a multi-tile layout, then the one-block path, then a smaller multi-tile one
    with drops, and back, each equal to the workspace call."""
    for i, w in enumerate(SEQUENCE):
        cfg = moe.config_from(w)
        ids = torch.from_numpy(synth.uniform_topk_ids(30 + i, synth.TID_TEST + 21, w.T, w.E, w.K)).cuda()
        ref_buf = moe.alloc_layout(cfg)
        moe.moe_dispatch_layout(cfg, ids, ref_buf.counts, ref_buf.kept, ref_buf.offsets, ref_buf.slot,
                                ref_buf.row_src, ref_buf.n_ij, ref_buf.rank_bytes, ref_buf.stats,
                                moe.alloc_workspace(cfg, moe.MOE_OP_LAYOUT))
        buf = moe.alloc_layout(cfg)
        _call_static(cfg, ids, buf)
        assert moe.moe_check() == 0
        for a, b in zip(_outputs(buf), _outputs(ref_buf)):
            assert torch.equal(a, b), (i, w.name)


def test_static_layout_refuses_layouts_above_its_fixed_scratch():
    w = workloads.Workload("big", T=400000, h=64, E=1024, K=8, I=64, dtype="bf16", score="softmax", ep_size=8)
    cfg = moe.config_from(w)
    assert moe.moe_workspace_size(cfg, moe.MOE_OP_LAYOUT) > (1 << 20)
    # valid, aligned device pointers: the size check is what refuses the call,
    # on the host, before anything is launched
    buf = moe.alloc_layout(moe.config_from(workloads.TINY))
    ids = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = moe.lib.moe_dispatch_layout_static(
        ctypes.byref(cfg), ids.data_ptr(), buf.counts.data_ptr(), buf.kept.data_ptr(), buf.offsets.data_ptr(),
        buf.slot.data_ptr(), buf.row_src.data_ptr(), buf.n_ij.data_ptr(), buf.rank_bytes.data_ptr(),
        buf.stats.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 4                          # MOE_ERR_WORKSPACE_TOO_SMALL
    assert moe.moe_check() == 0
