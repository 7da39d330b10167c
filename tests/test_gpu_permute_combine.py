"""GPU permute (bit-exact copies) and combine (tolerance) against the oracle."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import TOL, dev_of, np_of, oracle_routing, rel_err

pytestmark = pytest.mark.gpu


def _layout_for(w, routed):
    if routed:
        o = oracle_routing(w.name)
        return o["ids"], o["w"], o["layout"]
    ids = synth.uniform_topk_ids(3, synth.TID_TEST + 5, w.T, w.E, w.K)
    wts = synth.uniform(3, synth.TID_TEST + 6, w.T * w.K, 0.0, 1.0).reshape(w.T, w.K)
    return ids, wts, oracle.dispatch_layout(ids, w)


CASES = {
    "tiny_f32": (workloads.TINY, True),
    "mixtral_8x7b": (workloads.MIXTRAL, True),
    "deepseek_v3": (workloads.DSV3, True),
    "switch_base": (workloads.SWITCH, True),
    "deepseek_v3_decode_T32": (workloads.DECODE[0], True),
    "pad_f32": (workloads.Workload("pad_f32", T=300, h=128, E=16, K=3, I=64, dtype="f32", score="softmax",
                                   capacity=50, pad=1, ep_size=4), False),
    "pad_bf16_wide": (workloads.Workload("pad_bf16", T=129, h=28672, E=8, K=2, I=64, dtype="bf16",
                                         score="softmax", capacity=20, pad=1, ep_size=2), False),
}


@pytest.mark.parametrize("case", list(CASES))
def test_permute_bit_exact(case):
    w, routed = CASES[case]
    ids, _, lay = _layout_for(w, routed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    x = device.fill_normal(torch.empty(w.T, w.h, dtype=dt, device="cuda"), 0, synth.TID_X, 1.0)
    R = lay["rows"]
    xp = torch.full((R, w.h), float("nan"), dtype=dt, device="cuda")
    moe.moe_permute(moe.config_from(w), x, dev_of(lay["slot"]), dev_of(lay["row_src"]), xp)
    assert moe.moe_check() == 0
    ref = oracle.permute(np_of(x), lay["row_src"])
    got = np_of(xp)
    rs = lay["row_src"]
    written = rs >= 0
    if w.pad and w.capacity > 0:
        written = np.ones(R, dtype=bool)          # pad rows are zero-filled
    assert np.array_equal(got[written], ref[written])


@pytest.mark.parametrize("case", list(CASES))
def test_combine(case):
    w, routed = CASES[case]
    ids, wts, lay = _layout_for(w, routed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    R = lay["rows"]
    yp = device.fill_normal(torch.empty(R, w.h, dtype=dt, device="cuda"), 0, synth.TID_TEST + 7, 1.0)
    y = torch.empty(w.T, w.h, dtype=dt, device="cuda")
    moe.moe_combine(moe.config_from(w), yp, dev_of(lay["slot"]), dev_of(wts.astype(np.float32)), y)
    assert moe.moe_check() == 0
    ref = oracle.combine(np_of(yp), lay["slot"], wts, w, rounded=False)
    err = rel_err(np_of(y), ref, w.dtype)
    assert err <= TOL[w.dtype], err


def test_identity_experts_roundtrip():
    """permute then combine with identity experts gives (sum of kept weights) * x."""
    w = workloads.Workload("id", T=513, h=192, E=12, K=3, I=64, dtype="f32", score="softmax", capacity=100,
                           ep_size=3)
    ids, wts, lay = _layout_for(w, False)
    cfg = moe.config_from(w)
    x = device.fill_normal(torch.empty(w.T, w.h, device="cuda"), 0, synth.TID_X, 1.0)
    xp = torch.zeros(lay["rows"], w.h, device="cuda")
    moe.moe_permute(cfg, x, dev_of(lay["slot"]), None, xp)
    y = torch.empty_like(x)
    moe.moe_combine(cfg, xp, dev_of(lay["slot"]), dev_of(wts.astype(np.float32)), y)
    assert moe.moe_check() == 0
    assert lay["dropped"] > 0
    wk = np.where(lay["slot"] >= 0, wts.astype(np.float64), 0.0).sum(axis=1)
    np.testing.assert_allclose(np_of(y), wk[:, None] * np_of(x).astype(np.float64), rtol=1e-6, atol=1e-6)
