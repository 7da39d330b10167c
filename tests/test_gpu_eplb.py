"""Expert-parallel load balancing on the GPU against the oracle: the replica
map bit-exact, the FFN of replicas sharing their logical expert's weights, and
the routed layer over physical experts (index outputs bit-exact from the GPU's
routing, outputs within tolerance)."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import log_near_ties, TOL, dev_of, host_inputs, np_of, rel_err
from test_gpu_layer import NEAR_TIE

pytestmark = pytest.mark.gpu


def _plan_dev(plan):
    return {k: dev_of(plan[k]) for k in ("rep_offsets", "rep_phys", "phys_to_log")}


@pytest.mark.parametrize("T,E,K,n_ep,R", [(1, 8, 2, 2, 2), (333, 16, 4, 4, 4), (4096, 256, 8, 64, 64),
                                          (16384, 128, 1, 16, 16)])
def test_eplb_map_bit_exact(T, E, K, n_ep, R):
    ids = synth.uniform_topk_ids(7, synth.TID_TEST + 40, T, E, K)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    plan = oracle.eplb_plan(counts, n_ep, R)
    w = workloads.Workload("map", T=T, h=64, E=E, K=K, I=64, dtype="bf16", score="softmax", ep_size=n_ep,
                           n_redundant=R)
    pd = _plan_dev(plan)
    out = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    moe.moe_eplb_map(moe.config_from(w), dev_of(ids), pd["rep_offsets"], pd["rep_phys"], out)
    assert moe.moe_check() == 0
    assert np.array_equal(np_of(out), oracle.eplb_map(ids, plan["rep_offsets"], plan["rep_phys"]))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_grouped_ffn_mapped(dtype):
    """Replicas run their logical expert's weights (one copy in memory)."""
    w = workloads.Workload("ffn_mapped", T=300, h=256, E=6, K=2, I=128, dtype=dtype, score="softmax", ep_size=2,
                           n_redundant=2)
    ids = synth.uniform_topk_ids(8, synth.TID_TEST + 41, w.T, w.E, w.K)
    ids[: w.T // 2, 0] = 0                                    # expert 0 hot
    plan = oracle.eplb_plan(np.bincount(ids.reshape(-1), minlength=w.E), w.ep_size, w.n_redundant)
    pids = oracle.eplb_map(ids, plan["rep_offsets"], plan["rep_phys"])
    pcfg = w.replace(E=w.E + w.n_redundant)
    lay = oracle.dispatch_layout(pids, pcfg)
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    xp = device.fill_normal(torch.empty(lay["rows"], w.h, dtype=dt, device="cuda"), 8, synth.TID_TEST + 42, 1.0)
    inp = device.layer_inputs(w)
    yp = torch.full((lay["rows"], w.h), float("nan"), dtype=dt, device="cuda")
    cfg = moe.config_from(w)
    moe.moe_grouped_ffn_mapped(cfg, xp, dev_of(lay["offsets"]), dev_of(lay["kept"]), _plan_dev(plan)["phys_to_log"],
                               inp["w13"], inp["w2"], yp, moe.alloc_workspace(cfg, moe.MOE_OP_FFN))
    assert moe.moe_check() == 0
    p2l = plan["phys_to_log"]
    W13, W2 = np_of(inp["w13"]), np_of(inp["w2"])
    ref = oracle.grouped_ffn(np_of(xp), lay["offsets"], lay["kept"], lambda p: W13[p2l[p]], lambda p: W2[p2l[p]],
                             pcfg, rounded=False)
    got = np_of(yp)
    worst = max(rel_err(got[idx], val, dtype) for idx, val in ref.values() if len(idx))
    assert worst <= TOL[dtype]


def check_layer_eplb(w, sample=None, seed=0):
    inp = device.layer_inputs(w)
    h = {k: (np_of(v) if v is not None else None) for k, v in inp.items() if k in ("x", "w_r", "sel_bias",
                                                                                      "logit_offset")}
    L = oracle.router_logits(h["x"], h["w_r"], w.dtype, h["logit_offset"])
    ids, wts, keys, allowed = oracle.route(L, w, h["sel_bias"])
    plan = oracle.eplb_plan(np.bincount(ids.reshape(-1), minlength=w.E), w.ep_size, w.n_redundant)
    pd = _plan_dev(plan)
    cfg = moe.config_from(w)
    T, K, P, N = w.T, w.K, w.E + w.n_redundant, w.ep_size
    R = moe.moe_rows(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(topk_ids=torch.empty(T, K, **i32), topk_w=torch.empty(T, K, device="cuda"),
             counts=torch.empty(P, **i32), kept=torch.empty(P, **i32), offsets=torch.empty(P + 1, **i32),
             slot=torch.empty(T, K, **i32), row_src=torch.empty(max(R, 1), **i32),
             n_ij=torch.empty(N * N, dtype=torch.int64, device="cuda"),
             rank_bytes=torch.empty(2 * N, dtype=torch.int64, device="cuda"),
             stats=torch.empty(4, dtype=torch.int64, device="cuda"))
    y = torch.empty(T, w.h, dtype=inp["x"].dtype, device="cuda")
    moe.moe_layer_forward_eplb(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                               inp["w2"], pd["rep_offsets"], pd["rep_phys"], pd["phys_to_log"], y,
                               moe.layer_out(**o), moe.alloc_workspace(cfg, moe.MOE_OP_LAYER))
    assert moe.moe_check() == 0
    gids = np_of(o["topk_ids"])
    bad = np.nonzero((gids != ids).any(axis=1))[0]
    margin = oracle.near_tie_margin(keys, allowed, w)
    assert np.all(margin[bad] < NEAR_TIE), f"routing differs away from a near-tie at tokens {bad[:8]}"
    # the layout over physical experts, bit-exact against the oracle's from the GPU's logical ids
    pcfg = w.replace(E=P, n_groups=0, topk_groups=0, group_topn=0)
    pids = oracle.eplb_map(gids, plan["rep_offsets"], plan["rep_phys"])
    lay = oracle.dispatch_layout(pids, pcfg)
    for k in ("counts", "kept", "offsets", "slot"):
        assert np.array_equal(np_of(o[k]), lay[k]), k
    assert np.array_equal(np_of(o["row_src"])[:lay["rows"]], lay["row_src"])
    assert np.array_equal(np_of(o["n_ij"]).reshape(N, N), lay["n_ij"])
    stats = moe.stats_dict(o["stats"])
    assert abs(stats["balancedness"] - float(lay["balancedness"])) < 1e-6
    tokens = np.setdiff1d(np.arange(T), bad)
    if sample is not None:
        tokens = np.sort(np.random.default_rng(seed).choice(tokens, size=min(sample, len(tokens)), replace=False))
    need = {}
    for t in tokens:
        for k in range(K):
            s = lay["slot"][t, k]
            if s >= 0:
                need.setdefault(int(pids[t, k]), []).append(int(s))
    p2l = plan["phys_to_log"]
    xp = oracle.permute(h["x"], lay["row_src"])
    parts = oracle.grouped_ffn(xp, lay["offsets"], lay["kept"],
                               lambda p: workloads.host_w13(w, int(p2l[p])), lambda p: workloads.host_w2(w, int(p2l[p])),
                               pcfg, experts=sorted(need), rows={e: sorted(set(r)) for e, r in need.items()})
    yp = np.zeros(xp.shape, dtype=xp.dtype)
    for e, (idx, val) in parts.items():
        yp[idx] = val
    # the oracle's own weights (the GPU's routed like the oracle at these tokens)
    ref = oracle.combine(yp, lay["slot"], wts, pcfg, tokens=list(tokens), rounded=False)
    err = rel_err(np_of(y)[tokens], ref, w.dtype)
    log_near_ties(w.name, T, int((margin < NEAR_TIE).sum()), len(bad), len(tokens))
    assert err <= TOL[w.dtype], err
    return stats


EPLB_SMALL = [
    workloads.SWITCH_EPLB.replace(name="switch_eplb_small", T=2048, h=256, I=256, capacity=20),
    workloads.DSV3_EPLB.replace(name="dsv3_eplb_small", T=256, h=512, I=256),
    workloads.TINY.replace(name="tiny_eplb_f32", n_redundant=4),
]


@pytest.mark.parametrize("w", EPLB_SMALL, ids=[w.name for w in EPLB_SMALL])
def test_layer_eplb_small(w):
    check_layer_eplb(w)


@pytest.mark.parametrize("name", ["switch_base_eplb", "deepseek_v3_eplb"])
def test_layer_eplb_full_size_sampled(name):
    w = workloads.EXTRA[name]
    stats = check_layer_eplb(w, sample=6)
    if name == "switch_base_eplb":  # the Zipf-skewed layer is far better balanced with replicas
        assert stats["balancedness"] > 0.9


def test_layer_without_plan_refuses_replicas():
    w = EPLB_SMALL[1]
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    with pytest.raises(moe.MoeError):
        moe.moe_layer_forward(cfg, inp["x"], inp["w_r"], None, inp["sel_bias"], inp["w13"], inp["w2"],
                              torch.empty_like(inp["x"]), None, moe.alloc_workspace(cfg, moe.MOE_OP_LAYER))
