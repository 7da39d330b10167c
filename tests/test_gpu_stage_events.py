"""Stage events of the layer call (moe_layer_out.stage_events): every stage
timed, or only some (NULL entries are skipped), with the layer's outputs
unchanged either way."""
import pytest
import torch

import expert_dispatch_bias_b300 as moe
from synth import device, workloads

pytestmark = pytest.mark.gpu


def _recorded(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:   # torch creates each CUDA event on its first record
        e.record()
    return evs


SMALL = [
    workloads.DSV3.replace(name="dsv3_small", T=256, h=512, I=256),
    workloads.SWITCH.replace(name="switch_small", T=2048, h=256, I=256, capacity=16),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_stage_events_all_and_partial(w):
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_LAYER)
    n_ev = len(moe.LAYER_STAGES) + 1
    i_ffn = list(moe.LAYER_STAGES).index("ffn")

    def call(out):
        y = torch.empty(w.T, w.h, dtype=inp["x"].dtype, device="cuda")
        moe.moe_layer_forward(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], inp["w13"],
                              inp["w2"], y, out, ws)
        torch.cuda.synchronize()
        assert moe.moe_check() == 0
        return y

    y_plain = call(moe.layer_out())

    # every stage: consecutive events, non-negative stage times that add up to the call
    evs = _recorded(n_ev)
    torch.cuda.synchronize()
    y_all = call(moe.layer_out(stage_events=evs))
    stage_ms = [evs[j].elapsed_time(evs[j + 1]) for j in range(n_ev - 1)]
    assert all(t >= 0.0 for t in stage_ms)
    assert stage_ms[i_ffn] > 0.0
    assert sum(stage_ms) == pytest.approx(evs[0].elapsed_time(evs[-1]), rel=1e-3, abs=1e-2)  # event resolution ~0.5 us each

    # only the FFN's two events (NULL elsewhere): recorded around the FFN alone
    a, b = _recorded(2)
    torch.cuda.synchronize()
    partial = [a if j == i_ffn else b if j == i_ffn + 1 else None for j in range(n_ev)]
    y_part = call(moe.layer_out(stage_events=partial))
    assert 0.0 < a.elapsed_time(b) <= stage_ms[i_ffn] * 4 + 1.0

    assert torch.equal(y_all, y_plain) and torch.equal(y_part, y_plain)
