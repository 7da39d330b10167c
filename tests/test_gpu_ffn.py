"""GPU grouped SwiGLU FFN against the oracle: whole small layers, and sampled
experts of the full-size ones in the launch configuration the layer uses."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import TOL, dev_of, expert_weights, np_of, rel_err

pytestmark = pytest.mark.gpu


def _run_ffn(w, lay, experts=None, rows_per_expert=None):
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    cfg = moe.config_from(w)
    R = lay["rows"]
    xp = device.fill_normal(torch.empty(R, w.h, dtype=dt, device="cuda"), 0, synth.TID_TEST + 11, 1.0)
    inp = device.layer_inputs(w)
    yp = torch.full((R, w.h), float("nan"), dtype=dt, device="cuda")
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_FFN)
    moe.moe_grouped_ffn(cfg, xp, dev_of(lay["offsets"]), dev_of(lay["kept"]), inp["w13"], inp["w2"], yp, ws)
    assert moe.moe_check() == 0
    xp_h, yp_h = np_of(xp), np_of(yp)
    if experts is None:
        get13 = lambda e: np_of(inp["w13"][e])  # noqa: E731
        get2 = lambda e: np_of(inp["w2"][e])  # noqa: E731
    else:
        get13 = lambda e: expert_weights(w, e)[0]  # noqa: E731
        get2 = lambda e: expert_weights(w, e)[1]  # noqa: E731
    rows = None
    if rows_per_expert is not None:
        rows = {}
        for e in experts:
            r0, n = int(lay["offsets"][e]), int(lay["kept"][e])
            rows[e] = np.unique(np.r_[r0:r0 + min(n, rows_per_expert), max(r0, r0 + n - 3):r0 + n])
    ref = oracle.grouped_ffn(xp_h, lay["offsets"], lay["kept"], get13, get2, w, experts=experts, rows=rows,
                             rounded=False)
    worst = 0.0
    for e, (idx, val) in ref.items():
        if len(idx):
            worst = max(worst, rel_err(yp_h[idx], val, w.dtype))
    return worst


def _small(name, **kw):
    return workloads.Workload(name, **kw)


SMALL = [
    _small("tiny_f32_full", T=256, h=256, E=8, K=2, I=512, dtype="f32", score="softmax", capacity=80),
    _small("bf16_ragged", T=300, h=512, E=8, K=2, I=384, dtype="bf16", score="softmax"),
    _small("bf16_many_experts", T=200, h=256, E=64, K=4, I=128, dtype="bf16", score="softmax"),
    _small("bf16_pad", T=250, h=256, E=16, K=2, I=256, dtype="bf16", score="softmax", capacity=40, pad=1),
    _small("bf16_empty_experts", T=40, h=768, E=32, K=1, I=256, dtype="bf16", score="softmax"),
    # widths that are multiples of 64 only: the last feature tile reaches past I
    # (or h) and the k-blocks (5) do not fill whole rounds of the 4-stage ring
    _small("bf16_odd_widths", T=300, h=320, E=8, K=2, I=320, dtype="bf16", score="softmax"),
    _small("bf16_odd_widths_tokens_as_m", T=2048, h=320, E=4, K=2, I=448, dtype="bf16", score="softmax"),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_ffn_small_full(w):
    ids = synth.uniform_topk_ids(5, synth.TID_TEST + 9, w.T, w.E, w.K)
    if w.name == "bf16_empty_experts":
        ids = (ids % 5).astype(np.int32)          # experts 5..31 receive nothing
    lay = oracle.dispatch_layout(ids, w)
    err = _run_ffn(w, lay)
    assert err <= TOL[w.dtype], err


@pytest.mark.parametrize("name", ["mixtral_8x7b", "deepseek_v3", "switch_base", "deepseek_v3_decode_T32"])
def test_ffn_full_size_sampled_experts(name):
    """Every row of three experts' segments at full h and I, in the launch
    configuration the layer uses (at Mixtral's shape: ~1024 rows per expert,
    every 128-row m-block of the tokens-as-M kernel)."""
    w = workloads.ALL[name]
    ids = synth.uniform_topk_ids(6, synth.TID_TEST + 10, w.T, w.E, w.K)
    lay = oracle.dispatch_layout(ids, w)
    nz = np.nonzero(lay["kept"])[0]
    experts = sorted({int(nz[0]), int(nz[len(nz) // 2]), int(nz[-1])})
    err = _run_ffn(w, lay, experts=experts)
    print(f"{name}: experts {experts}, {int(lay['kept'][experts].sum())} rows compared, err {err:.3e}")
    assert err <= TOL[w.dtype], err


# Expert row counts straddling every boundary of the token tiles (sub-blocks of
# at most 128 rows, MMA widths rounded to 16, tiles of 128, 160 or 256 rows
# chosen from the mean rows per expert, longer segments split evenly).
# "wide": more boundaries of the weights-as-M kernel (multiples of 32 and their
# neighbours, tiles split in two and three); the empty experts keep the mean
# rows per expert in the weights-as-M regime.
BOUNDARY_COUNTS = {
    "wide": [0, 1, 31, 32, 33, 63, 64, 65, 96, 97, 128, 129, 160, 192, 193, 224, 255, 256, 257, 320, 511, 512, 513,
             700] + [0] * 8,
    "tile128": [0, 1, 15, 16, 17, 33, 64, 127, 128, 129, 200],
    "tile160": [0, 1, 15, 16, 17, 127, 128, 129, 144, 160, 161, 255, 256, 257, 300, 511],
    "tile256": [0, 1, 16, 127, 128, 129, 160, 161, 255, 256, 257, 300, 511, 600, 700],
}


@pytest.mark.parametrize("regime", list(BOUNDARY_COUNTS))
def test_ffn_tile_boundaries(regime):
    counts = np.array(BOUNDARY_COUNTS[regime])
    E = len(counts)
    w = _small(f"bf16_{regime}", T=int(counts.sum()), h=256, E=E, K=1, I=384, dtype="bf16", score="softmax")
    rng = np.random.default_rng(11)
    ids = rng.permutation(np.repeat(np.arange(E, dtype=np.int32), counts)).reshape(-1, 1)
    lay = oracle.dispatch_layout(ids, w)
    assert np.array_equal(lay["kept"], counts)
    err = _run_ffn(w, lay)
    assert err <= TOL[w.dtype], err
