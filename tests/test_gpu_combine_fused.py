"""The weighted combine fused into the grouped FFN's down projection
(moe_grouped_ffn_combine) against the oracle, and against the unfused path:
the fused y must equal moe_combine of the same expert rows bit for bit (same
float32 fused multiply-adds in k order), and a second call on the same
workspace must give the same bits (the arrival counters reset themselves)."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import TOL, dev_of, expert_weights, np_of, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    workloads.DSV3.replace(name="dsv3_small", T=256, h=512, I=256),
    workloads.Workload("ragged_h384", T=300, h=384, E=16, K=2, I=384, dtype="bf16", score="softmax"),
    workloads.Workload("top1", T=500, h=256, E=32, K=1, I=256, dtype="bf16", score="softmax"),
    workloads.ALL["deepseek_v3"],
    workloads.ALL["deepseek_v3_decode_T32"],
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_fused_combine(w):
    cfg = moe.config_from(w)
    inp = device.layer_inputs(w)
    ids = synth.uniform_topk_ids(13, synth.TID_TEST + 70, w.T, w.E, w.K)
    lay = oracle.dispatch_layout(ids, w)
    wts = synth.uniform(13, synth.TID_TEST + 71, w.T * w.K, 0.05, 1.0).astype(np.float32).reshape(w.T, w.K)
    R = lay["rows"]
    slot, row_src, twt = dev_of(lay["slot"]), dev_of(lay["row_src"]), dev_of(wts)
    offsets, kept = dev_of(lay["offsets"]), dev_of(lay["kept"])
    xp = torch.zeros(R, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, inp["x"], slot, row_src, xp)
    # unfused: FFN, then combine
    ya_p = torch.zeros(R, w.h, dtype=torch.bfloat16, device="cuda")
    ya = torch.zeros(w.T, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn(cfg, xp, offsets, kept, inp["w13"], inp["w2"], ya_p, moe.alloc_workspace(cfg, moe.MOE_OP_FFN))
    moe.moe_combine(cfg, ya_p, slot, twt, ya)
    # fused, twice on one workspace
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_FFN_COMBINE)
    outs = []
    for _ in range(2):
        yb_p = torch.full((R, w.h), float("nan"), dtype=torch.bfloat16, device="cuda")
        yb = torch.full((w.T, w.h), float("nan"), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_ffn_combine(cfg, xp, offsets, kept, inp["w13"], inp["w2"], row_src, slot, twt, yb_p, yb, ws)
        assert moe.moe_check() == 0
        outs.append(yb)
        assert torch.equal(yb_p, ya_p)
        assert torch.equal(yb, ya)
    assert torch.equal(outs[0], outs[1])
    # against the oracle: every token of the small cases, a sample at full size
    full_size = w.h * w.I > 4 << 20
    tokens = np.arange(w.T)
    if full_size:
        tokens = np.sort(np.random.default_rng(3).choice(w.T, size=min(8, w.T), replace=False))
    need = {}
    for t in tokens:
        for k in range(w.K):
            need.setdefault(int(ids[t, k]), []).append(int(lay["slot"][t, k]))
    get13 = (lambda e: expert_weights(w, e)[0]) if full_size else (lambda e: np_of(inp["w13"][e]))
    get2 = (lambda e: expert_weights(w, e)[1]) if full_size else (lambda e: np_of(inp["w2"][e]))
    xp_ref = oracle.permute(np_of(inp["x"]), lay["row_src"])
    parts = oracle.grouped_ffn(xp_ref, lay["offsets"], lay["kept"], get13, get2, w, experts=sorted(need),
                               rows={e: sorted(set(r)) for e, r in need.items()})
    yp_ref = np.zeros(xp_ref.shape, dtype=xp_ref.dtype)
    for e, (idx, val) in parts.items():
        yp_ref[idx] = val
    ref = oracle.combine(yp_ref, lay["slot"], wts, w, tokens=list(tokens), rounded=False)
    err = rel_err(np_of(outs[0])[tokens], ref, w.dtype)
    assert err <= TOL[w.dtype], err


def test_fused_combine_refuses_unsupported():
    w = workloads.Workload("drops", T=300, h=256, E=16, K=2, I=256, dtype="bf16", score="softmax", capacity=30)
    cfg = moe.config_from(w)
    inp = device.layer_inputs(w)
    z = torch.zeros(1024, dtype=torch.int32, device="cuda")
    y = torch.empty_like(inp["x"])
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):   # capacity drops leave tokens without K arrivals
        moe.moe_grouped_ffn_combine(cfg, inp["x"], z, z, inp["w13"], inp["w2"], z, z, z.float(), y, y, ws)
    w2 = workloads.MIXTRAL.replace(name="mixtral_small", T=4096, h=256, I=256)   # tokens-as-M layer
    cfg2 = moe.config_from(w2)
    inp2 = device.layer_inputs(w2)
    y2 = torch.empty_like(inp2["x"])
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_ffn_combine(cfg2, inp2["x"], z, z, inp2["w13"], inp2["w2"], z, z, z.float(), y2, y2, ws)
