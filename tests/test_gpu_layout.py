"""GPU dispatch layout against the oracle: every index output bit-exact."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import workloads

from gpu_helpers import dev_of, np_of, oracle_routing

pytestmark = pytest.mark.gpu


def run_layout(w, ids_np, ws=None, slot_init=None):
    cfg = moe.config_from(w)
    buf = moe.alloc_layout(cfg)
    if slot_init is not None:
        buf.slot.fill_(slot_init)
    if ws is None:
        ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYOUT)
    ids = dev_of(ids_np.astype(np.int32)) if ids_np.size else torch.empty(1, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_layout(cfg, ids, buf.counts, buf.kept, buf.offsets, buf.slot, buf.row_src, buf.n_ij,
                            buf.rank_bytes, buf.stats, ws)
    return buf, ws


def compare(w, ids_np, buf):
    ref = oracle.dispatch_layout(ids_np, w)
    T, K = ids_np.shape
    R = ref["rows"]
    N = w.ep_size
    assert np.array_equal(np_of(buf.counts), ref["counts"])
    assert np.array_equal(np_of(buf.kept), ref["kept"])
    assert np.array_equal(np_of(buf.offsets), ref["offsets"])
    assert np.array_equal(np_of(buf.slot)[:T * K].reshape(T, K), ref["slot"])
    assert np.array_equal(np_of(buf.row_src)[:R], ref["row_src"])
    assert np.array_equal(np_of(buf.n_ij).reshape(N, N), ref["n_ij"])
    rb = np_of(buf.rank_bytes)
    assert np.array_equal(rb[:N], ref["sent_bytes"]) and np.array_equal(rb[N:], ref["recv_bytes"])
    st = moe.stats_dict(buf.stats)
    assert st["kept_total"] == ref["kept_total"] and st["dropped"] == ref["dropped"]
    assert st["offdiag_rows"] == ref["offdiag_rows"]
    assert st["experts_touched"] == ref["experts_touched"]
    assert np.float32(st["balancedness"]) == ref["balancedness"]


@pytest.mark.parametrize("name", list(workloads.ALL))
def test_layout_workloads_bit_exact(name):
    w = workloads.ALL[name]
    ids = oracle_routing(name)["ids"]
    buf, ws = run_layout(w, ids)
    assert moe.moe_check() == 0
    compare(w, ids, buf)
    # the workspace cleans itself: a second call on it gives the same result
    buf2, _ = run_layout(w, ids, ws=ws)
    assert moe.moe_check() == 0
    compare(w, ids, buf2)


def _wl(T, E, K, cap=0, pad=0, ep=1):
    return workloads.Workload(name="edge", T=T, h=64, E=E, K=K, I=64, dtype="bf16", score="softmax",
                              capacity=cap, pad=pad, ep_size=ep)


EDGE = {
    "uniform_ep64": (_wl(512, 256, 8, ep=64), "uniform"),
    "ragged_capacity": (_wl(1000, 60, 3, cap=45, ep=6), "uniform"),
    "all_to_expert0": (_wl(5000, 16, 1, cap=100, ep=4), "zeros"),
    "pad": (_wl(777, 32, 4, cap=90, pad=1, ep=8), "uniform"),
    "one_token": (_wl(1, 4, 2, ep=2), "uniform"),
    "max_E_K": (_wl(3000, 1024, 16, cap=40, ep=1024), "uniform"),
    "many_tiles": (_wl(65536, 64, 8, ep=8), "uniform"),
    "single_expert": (_wl(333, 1, 1, ep=1), "zeros"),
    "T_below_ep": (_wl(32, 256, 8, ep=64), "uniform"),
    "capacity_one_pad": (_wl(200, 8, 2, cap=1, pad=1, ep=4), "uniform"),
    # up to 8192 assignments take the one-block layout, more the two-pass one:
    # both sides of the boundary, and the drop/pad/skew cases above on the
    # two-pass layout
    "small_limit": (_wl(1024, 256, 8, ep=64), "uniform"),
    "small_limit_plus_one": (_wl(8193, 64, 1, cap=200, ep=8), "uniform"),
    "ragged_capacity_two_pass": (_wl(10000, 60, 3, cap=450, ep=6), "uniform"),
    "all_to_expert0_two_pass": (_wl(20000, 16, 1, cap=1000, ep=4), "zeros"),
    "pad_two_pass": (_wl(2777, 32, 4, cap=300, pad=1, ep=8), "uniform"),
    "T_below_ep_wide": (_wl(40, 1024, 16, ep=64), "uniform"),
    "small_ep128": (_wl(500, 256, 8, ep=128), "uniform"),  # N_EP^2 above the shared n_ij bins
}


@pytest.mark.parametrize("case", list(EDGE))
def test_layout_edge_cases(case):
    w, kind = EDGE[case]
    if kind == "zeros":
        ids = np.zeros((w.T, w.K), dtype=np.int32)
    else:
        ids = synth.uniform_topk_ids(7, synth.TID_TEST + 3, w.T, w.E, w.K)
    buf, _ = run_layout(w, ids)
    assert moe.moe_check() == 0
    compare(w, ids, buf)


def test_layout_empty_batch():
    w = _wl(0, 8, 2, cap=3, pad=1, ep=2)
    buf, _ = run_layout(w, np.zeros((0, 2), dtype=np.int32))
    assert moe.moe_check() == 0
    assert np_of(buf.counts).tolist() == [0] * 8
    assert np_of(buf.offsets).tolist() == [3 * e for e in range(9)]
    assert np_of(buf.row_src)[:24].tolist() == [-1] * 24
    assert moe.stats_dict(buf.stats)["kept_total"] == 0


def test_layout_bad_expert_id_reported():
    w = _wl(100, 8, 2, ep=2)
    ids = synth.uniform_topk_ids(1, synth.TID_TEST, w.T, w.E, w.K)
    ids[17, 1] = 8          # out of range
    run_layout(w, ids)
    assert moe.moe_check() == 7   # MOE_ERR_DEVICE_BAD_INDEX
    assert moe.moe_check() == 0   # cleared


def test_lookback_wait_times_out_with_status():
    """A tile whose predecessor never publishes: the bounded look-back gives up
    after about a second, sets the sticky error and the kernel returns; the
    context stays usable and the next call is correct."""
    w = _wl(1280, 32, 8, ep=4)     # 10240 assignments: the two-pass layout, five tiles
    ids = synth.uniform_topk_ids(2, synth.TID_TEST, w.T, w.E, w.K)
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYOUT)
    ws[:4].view(torch.int32).fill_(1)   # the tile counter starts at 1: tile 0 is never taken
    run_layout(w, ids, ws=ws, slot_init=0)
    assert moe.moe_check() == 6          # MOE_ERR_DEVICE_TIMEOUT
    moe.moe_workspace_init(ws)
    buf, _ = run_layout(w, ids, ws=ws)
    assert moe.moe_check() == 0
    compare(w, ids, buf)
