"""The permutation fused into the grouped FFN (rows gathered from x through
row_src) against the oracle: the oracle permutes x by row_src and runs every
expert's FFN (a sample of experts, every row of each, at full size).  The
two-step path (explicit permute, then the FFN on the permuted copy) must also
give bit-identical expert outputs, since only the load path differs."""
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
    workloads.Workload("ragged", T=300, h=384, E=16, K=2, I=384, dtype="bf16", score="softmax", capacity=30),
    workloads.Workload("pad", T=250, h=256, E=16, K=2, I=256, dtype="bf16", score="softmax", capacity=40, pad=1),
    workloads.Workload("empty_experts", T=40, h=768, E=32, K=1, I=256, dtype="bf16", score="softmax"),
    workloads.DSV3.replace(name="dsv3_decode_T1", T=1),
    workloads.ALL["deepseek_v3"],
    workloads.ALL["switch_base"],
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_gather_equals_permute_then_ffn(w):
    cfg = moe.config_from(w)
    inp = device.layer_inputs(w)
    ids = synth.uniform_topk_ids(12, synth.TID_TEST + 60, w.T, w.E, w.K)
    if w.name == "empty_experts":
        ids = (ids % 5).astype(np.int32)
    lay = oracle.dispatch_layout(ids, w)
    R = lay["rows"]
    slot, row_src = dev_of(lay["slot"]), dev_of(lay["row_src"])
    offsets, kept = dev_of(lay["offsets"]), dev_of(lay["kept"])
    xp = torch.zeros(R, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, inp["x"], slot, row_src, xp)
    ya = torch.zeros(R, w.h, dtype=torch.bfloat16, device="cuda")
    yb = torch.zeros(R, w.h, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_FFN)
    moe.moe_grouped_ffn(cfg, xp, offsets, kept, inp["w13"], inp["w2"], ya, ws)
    moe.moe_grouped_ffn_gather(cfg, inp["x"], row_src, offsets, kept, inp["w13"], inp["w2"], yb, ws)
    assert moe.moe_check() == 0
    rows = torch.from_numpy(lay["row_src"] >= 0).cuda()
    assert torch.equal(ya[rows], yb[rows])
    # against the oracle on the oracle's own permutation of x
    xp_ref = oracle.permute(np_of(inp["x"]), lay["row_src"])
    nz = np.nonzero(lay["kept"])[0]
    full_size = w.h * w.I > 4 << 20
    if full_size:
        experts = sorted({int(nz[0]), int(nz[len(nz) // 2]), int(nz[-1])})
        get13, get2 = (lambda e: expert_weights(w, e)[0]), (lambda e: expert_weights(w, e)[1])
    else:
        experts = [int(e) for e in nz]
        get13, get2 = (lambda e: np_of(inp["w13"][e])), (lambda e: np_of(inp["w2"][e]))
    ref = oracle.grouped_ffn(xp_ref, lay["offsets"], lay["kept"], get13, get2, w, experts=experts, rounded=False)
    got = np_of(yb)
    worst = max(rel_err(got[idx], val, w.dtype) for idx, val in ref.values() if len(idx))
    assert worst <= TOL[w.dtype], worst


def test_gather_refuses_tokens_as_m_layers():
    w = workloads.MIXTRAL.replace(name="mixtral_small", T=4096, h=256, I=256)  # 1024 rows per expert
    cfg = moe.config_from(w)
    inp = device.layer_inputs(w)
    z = torch.zeros(8192, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_ffn_gather(cfg, inp["x"], z, z, z, inp["w13"], inp["w2"], torch.empty_like(inp["x"]),
                                   moe.alloc_workspace(cfg, moe.MOE_OP_FFN))
