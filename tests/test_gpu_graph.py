"""A layer call captured into a CUDA graph and replayed gives the eager call's
output bit for bit (the library's launches, with programmatic stream
serialisation, are capturable; a first eager call sets the kernels' shared
memory limits and caches the device properties)."""
import pytest
import torch

import expert_dispatch_bias_b300 as moe
from synth import device, workloads

pytestmark = pytest.mark.gpu

CASES = [
    workloads.DSV3.replace(name="dsv3_small", T=256, h=512, I=256),
    workloads.SWITCH.replace(name="switch_small", T=2048, h=256, I=256, capacity=16),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_graph_replay_matches_eager(w):
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYER)

    def call(y):
        moe.moe_layer_forward(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                              inp["w2"], y, moe.layer_out(), ws)

    y_eager = torch.empty(w.T, w.h, dtype=inp["x"].dtype, device="cuda")
    call(y_eager)
    torch.cuda.synchronize()
    assert moe.moe_check() == 0

    y = torch.empty_like(y_eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # warm-up on a side stream, as graph capture expects
        call(y)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(y)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert moe.moe_check() == 0
    assert torch.equal(y, y_eager)
