"""GPU parity of router logits and routing against the oracle, at full workload sizes."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import workloads

from gpu_helpers import dev_of, host_inputs, np_of, oracle_routing, rel_err

pytestmark = pytest.mark.gpu
NAMES = list(workloads.ALL)


@pytest.mark.parametrize("name", NAMES)
def test_router_logits(name):
    w = workloads.ALL[name]
    h = host_inputs(name)
    ref = oracle_routing(name)["logits"]
    cfg = moe.config_from(w)
    L = torch.empty(w.T, w.E, dtype=torch.float32, device="cuda")
    off = dev_of(h["logit_offset"]) if h["logit_offset"] is not None else None
    moe.moe_router_logits(cfg, dev_of(h["x"]), dev_of(h["w_r"]), off, L, moe.alloc_workspace(cfg, moe.MOE_OP_LOGITS))
    assert moe.moe_check() == 0
    # float32 accumulation of exact bf16/f32 products vs float64 sums
    assert rel_err(np_of(L), ref, "f32") < 1e-4


# (T, h, E): partial row blocks, expert counts that do not fill a column tile,
# every column-tile width; h of 1024 and more also slices the sum over h
# (1 row tile of 8 experts at h=4096: 8 slices; 2 row tiles x 8 column tiles of
# 128 at h=7168: 8; 33 tiles of 256 at h=7168: 4).
@pytest.mark.parametrize("T,h,E", [(1, 64, 8), (130, 128, 5), (300, 192, 33), (129, 64, 1000), (1200, 128, 256),
                                   (2500, 64, 1000), (40, 768, 128), (130, 1024, 5), (1, 4096, 8),
                                   (300, 2048, 33), (129, 7168, 1000), (4100, 7168, 256)])
@pytest.mark.parametrize("offset", [False, True])
def test_router_logits_ragged(T, h, E, offset):
    """bf16 logits on the tensor cores, with and without offsets.  A second call
    on the same workspace gives the same bits (the slice counters are reset and
    the slices are added in a fixed order)."""
    w = workloads.Workload("logits_case", T=T, h=h, E=E, K=1, I=64, dtype="bf16", score="softmax")
    x = synth.normal(3, synth.TID_TEST + 20, (T, h), 1.0, "bf16")
    wr = synth.normal(3, synth.TID_TEST + 21, (E, h), 1.0 / np.sqrt(h), "bf16")
    off = synth.uniform(3, synth.TID_TEST + 22, E, -2.0, 2.0) if offset else None
    ref = oracle.router_logits(x, wr, "bf16", off)
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LOGITS)
    L = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    args = (cfg, dev_of(x), dev_of(wr), dev_of(off) if offset else None)
    moe.moe_router_logits(*args, L, ws)
    assert moe.moe_check() == 0
    assert rel_err(np_of(L), ref, "f32") < 1e-4
    L2 = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(*args, L2, ws)
    assert moe.moe_check() == 0
    assert torch.equal(L, L2)


@pytest.mark.parametrize("name", NAMES)
def test_route_bit_exact_from_oracle_logits(name):
    w = workloads.ALL[name]
    o = oracle_routing(name)
    h = host_inputs(name)
    cfg = moe.config_from(w)
    ids = torch.empty(w.T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(w.T, w.K, dtype=torch.float32, device="cuda")
    bias = dev_of(h["sel_bias"]) if h["sel_bias"] is not None else None
    moe.moe_route(cfg, dev_of(o["logits"]), bias, ids, wt)
    assert moe.moe_check() == 0
    got = np_of(ids)
    mism = np.argwhere(got != o["ids"])
    assert len(mism) == 0, f"{len(mism)} id mismatches, first at {mism[:4].tolist()}"
    # weights: float64 evaluation on both sides, one rounding to float32
    np.testing.assert_allclose(np_of(wt), o["w"], rtol=3e-7, atol=0)


def _route_case(cfg_kw, L, bias=None):
    T, E = L.shape
    base = dict(T=T, h=64, E=E, K=2, I=64, dtype="bf16", score="softmax")
    base.update(cfg_kw)
    w = workloads.Workload(name="case", **base)
    ids_o, w_o, _, _ = oracle.route(L, w, bias)
    cfg = moe.config_from(w)
    ids = torch.empty(T, w.K, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, w.K, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dev_of(L), dev_of(bias) if bias is not None else None, ids, wt)
    assert moe.moe_check() == 0
    assert np.array_equal(np_of(ids), ids_o)
    np.testing.assert_allclose(np_of(wt), w_o, rtol=3e-7, atol=0)


@pytest.mark.parametrize("E,K", [(1, 1), (5, 3), (32, 32 // 2), (33, 7), (1000, 16), (1024, 1)])
def test_route_shapes_and_ties(E, K):
    """Odd expert counts, K up to 16, E up to 1024, and heavy exact ties (quantised
    logits) for softmax, sigmoid+bias and group-limited sigmoid."""
    rng = np.random.default_rng(E * 31 + K)
    T = 301
    L = (rng.integers(-6, 7, size=(T, E)) / 8.0).astype(np.float32)
    _route_case(dict(K=K), L)
    bias = (rng.integers(-3, 4, size=E) / 32.0).astype(np.float32)
    _route_case(dict(K=K, score="sigmoid", scale=2.5), L, bias)
    _route_case(dict(K=K, score="softmax", renormalize=0), L, bias)
    for G in (2, 4, 8, 32):
        if E % G == 0 and E // G >= 2 and (G // 2) * (E // G) >= K:
            _route_case(dict(K=K, score="sigmoid", n_groups=G, topk_groups=G // 2, group_topn=2), L, bias)


def test_route_empty_batch():
    w = workloads.TINY.replace(T=0)
    cfg = moe.config_from(w)
    moe.moe_route(cfg, torch.empty(0, device="cuda"), None, torch.empty(0, dtype=torch.int32, device="cuda"),
                  torch.empty(0, device="cuda"))
    assert moe.moe_check() == 0


@pytest.mark.parametrize("E,K,G,topn", [(64, 6, 8, 2), (256, 8, 8, 2), (40, 3, 0, 2), (256, 8, 8, 1),
                                        (128, 8, 16, 2)])
def test_route_sigmoid_near_ties(E, K, G, topn):
    """Sigmoid routing whose keys sit a few float32 ulps apart: float32 keys may
    order such experts differently from the exact ones, and the selection must
    still equal the oracle's (the near-ties have to be recognised and settled
    on exact keys)."""
    rng = np.random.default_rng(E + K)
    T = 512
    L = rng.standard_normal((T, E)).astype(np.float32)
    for t in range(T):                      # clusters of logits 1..40 ulps apart
        base = rng.choice(E, size=6, replace=False)
        for j, e in enumerate(base[1:]):
            L[t, e] = np.nextafter(L[t, base[0]], np.float32(np.inf) if j % 2 else np.float32(-np.inf))
            for _ in range(int(rng.integers(0, 40))):
                L[t, e] = np.nextafter(L[t, e], np.float32(np.inf))
    bias = (rng.integers(-3, 4, size=E) / 64.0).astype(np.float32)
    bias[rng.choice(E, size=E // 4, replace=False)] += np.float32(2.0 ** -22)
    kw = dict(K=K, score="sigmoid", scale=2.5)
    if G:
        kw.update(n_groups=G, topk_groups=G // 2, group_topn=topn)
    _route_case(kw, L, bias)


def test_top1_weight_of_non_finite_logits_is_nan():
    """Renormalised top-1 on the logits writes the scale as the weight without
    evaluating s / s; rows whose logits are NaN or all -inf still get NaN, as
    the oracle's float64 evaluation gives, so bad router input is not hidden."""
    w = workloads.SWITCH.replace(name="switch_nan", T=64)
    cfg = moe.config_from(w)
    L = synth.normal(4, synth.TID_TEST + 23, (w.T, w.E), 1.0, "f32").astype(np.float32)
    L[3, :] = np.nan
    L[9, :] = -np.inf
    ids = torch.empty(w.T, 1, dtype=torch.int32, device="cuda")
    wts = torch.empty(w.T, 1, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dev_of(L), None, ids, wts)
    assert moe.moe_check() == 0
    got = np_of(wts)[:, 0]
    _, ref, _, _ = oracle.route(L, w)
    bad = [3, 9]
    assert np.isnan(ref[bad, 0]).all() and np.isnan(got[bad]).all()
    good = np.setdiff1d(np.arange(w.T), bad)
    assert np.array_equal(got[good], ref[good, 0]) and (got[good] == w.scale).all()
