"""Back-to-back layer calls on one stream give bit-identical outputs.

Every kernel of the library is launched with programmatic stream
serialisation and waits for its predecessor before touching memory; a kernel
that read or wrote too early would show up here as a call whose output
differs from the others (the layer is deterministic: fixed reduction orders,
no atomics in any float sum)."""
import pytest
import torch

import expert_dispatch_bias_b300 as moe
from synth import device, workloads

pytestmark = pytest.mark.gpu

CASES = [
    workloads.DSV3.replace(name="dsv3_small", T=256, h=512, I=256),
    workloads.SWITCH.replace(name="switch_small", T=2048, h=256, I=256, capacity=16),
    workloads.DSV3.replace(name="dsv3_decode_T32_full_width", T=32),
    workloads.DSV3.replace(name="dsv3_small_block", T=256, h=512, I=256, shared_I=256),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_back_to_back_calls_are_bit_identical(w):
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    block = w.shared_I > 0
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_BLOCK if block else moe.MOE_OP_LAYER)
    n = 40
    ys = [torch.empty(w.T, w.h, dtype=inp["x"].dtype, device="cuda") for _ in range(n)]
    torch.cuda.synchronize()
    for y in ys:   # queued back to back, no synchronisation between the calls
        if block:
            moe.moe_block_forward(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                                  inp["w2"], inp["w13s"], inp["w2s"], y, moe.layer_out(), ws)
        else:
            moe.moe_layer_forward(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                                  inp["w2"], y, moe.layer_out(), ws)
    _same_outputs(ys)


def _same_outputs(ys):
    torch.cuda.synchronize()
    assert moe.moe_check() == 0
    assert torch.isfinite(ys[0].float()).all()
    differing = [i for i, y in enumerate(ys) if not torch.equal(y, ys[0])]
    assert not differing, f"calls {differing[:8]} differ from the first"


def test_back_to_back_fp8_layer_calls_are_bit_identical():
    from test_gpu_fp8 import _fp8_weights

    w = workloads.DSV3.replace(name="dsv3_fp8_small", T=256, h=512, I=256)
    inp = device.layer_inputs(w)
    q13, s13, q2, s2 = _fp8_weights(inp)
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYER_FP8)
    ys = [torch.empty(w.T, w.h, dtype=torch.bfloat16, device="cuda") for _ in range(40)]
    torch.cuda.synchronize()
    for y in ys:
        moe.moe_layer_forward_fp8(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], q13, s13, q2, s2,
                                  y, moe.layer_out(), ws)
    _same_outputs(ys)


def test_back_to_back_replica_layer_calls_are_bit_identical():
    import numpy as np

    import oracle
    from gpu_helpers import dev_of

    w = workloads.DSV3_EPLB.replace(name="dsv3_eplb_small", T=256, h=512, I=256)
    inp = device.layer_inputs(w)
    plan = oracle.eplb_plan(np.arange(1, w.E + 1, dtype=np.int64), w.ep_size, w.n_redundant)
    pd = {k: dev_of(plan[k]) for k in ("rep_offsets", "rep_phys", "phys_to_log")}
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYER)
    ys = [torch.empty(w.T, w.h, dtype=inp["x"].dtype, device="cuda") for _ in range(40)]
    torch.cuda.synchronize()
    for y in ys:
        moe.moe_layer_forward_eplb(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                                   inp["w2"], pd["rep_offsets"], pd["rep_phys"], pd["phys_to_log"], y,
                                   moe.layer_out(), ws)
    _same_outputs(ys)
