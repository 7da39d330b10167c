"""FP8 (E4M3) experts on the GPU against the oracle: codes and scales bit-exact
(quantisation and the fused quantise-permute), the FP8 FFN and the FP8 layer
within the bf16 tolerance of the oracle's FP8 computation on the same codes."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import TOL, dev_of, log_near_ties, np_of, rel_err
from test_gpu_layer import NEAR_TIE

pytestmark = pytest.mark.gpu


def quantize_dev(t):
    rows = t.shape[0]
    codes = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, dtype=torch.float32, device="cuda")
    moe.moe_quantize_fp8(t.reshape(rows, -1), codes, scales)
    return codes, scales


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 256), (1000, 7168), (4096, 2048)])
def test_quantize_bit_exact(rows, cols, dtype):
    rng = np.random.default_rng(rows + cols)
    v = (rng.normal(size=(rows, cols)) * np.exp(rng.normal(size=(rows, 1)) * 4)).astype(np.float32)
    v[0, :] = 0 if rows > 1 else v[0, :]
    v.reshape(-1)[rng.choice(v.size, size=min(50, v.size), replace=False)] *= 1e-6   # subnormal codes
    host = synth.f32_to_bf16_bits(v) if dtype == "bf16" else v
    codes, scales = quantize_dev(dev_of(host))
    assert moe.moe_check() == 0
    q, s = oracle.quantize_rows_e4m3(oracle.to_f64(host, dtype))
    assert np.array_equal(np_of(scales), s)
    assert np.array_equal(np_of(codes), q)


def test_permute_fp8_bit_exact():
    w = workloads.DSV3.replace(name="perm_fp8", T=300, h=512, I=256, capacity=12)
    inp = device.layer_inputs(w, weights=False)
    ids = synth.uniform_topk_ids(9, synth.TID_TEST + 50, w.T, w.E, w.K)
    lay = oracle.dispatch_layout(ids, w)
    xq = torch.zeros(lay["rows"], w.h, dtype=torch.uint8, device="cuda")
    sx = torch.zeros(lay["rows"], dtype=torch.float32, device="cuda")
    moe.moe_permute_fp8(moe.config_from(w), inp["x"], dev_of(lay["slot"]), xq, sx)
    assert moe.moe_check() == 0
    q, s = oracle.quantize_rows_e4m3(oracle.to_f64(np_of(inp["x"]), "bf16"))
    kept = lay["row_src"] >= 0
    src = lay["row_src"][kept]
    assert np.array_equal(np_of(xq)[kept], q[src])
    assert np.array_equal(np_of(sx)[kept], s[src])


def _fp8_weights(inp):
    E = inp["w13"].shape[0]
    q13, s13 = quantize_dev(inp["w13"].reshape(-1, inp["w13"].shape[-1]))
    q2, s2 = quantize_dev(inp["w2"].reshape(-1, inp["w2"].shape[-1]))
    return (q13.reshape(inp["w13"].shape), s13.reshape(E, -1), q2.reshape(inp["w2"].shape), s2.reshape(E, -1))


SMALL = [
    workloads.DSV3.replace(name="dsv3_fp8_small", T=256, h=512, I=256),
    workloads.SWITCH.replace(name="switch_fp8_small", T=2048, h=256, I=256, capacity=20),
    workloads.Workload("ragged_fp8", T=300, h=384, E=16, K=2, I=384, dtype="bf16", score="softmax", capacity=30),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_grouped_ffn_fp8(w):
    inp = device.layer_inputs(w)
    q13, s13, q2, s2 = _fp8_weights(inp)
    ids = synth.uniform_topk_ids(10, synth.TID_TEST + 51, w.T, w.E, w.K)
    lay = oracle.dispatch_layout(ids, w)
    cfg = moe.config_from(w)
    xq = torch.zeros(lay["rows"], w.h, dtype=torch.uint8, device="cuda")
    sx = torch.ones(lay["rows"], dtype=torch.float32, device="cuda")
    moe.moe_permute_fp8(cfg, inp["x"], dev_of(lay["slot"]), xq, sx)
    yp = torch.full((lay["rows"], w.h), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn_fp8(cfg, xq, sx, dev_of(lay["offsets"]), dev_of(lay["kept"]), q13, s13, q2, s2, yp,
                            moe.alloc_workspace(cfg, moe.MOE_OP_FFN_FP8))
    assert moe.moe_check() == 0
    xq_h, sx_h, y_h = np_of(xq), np_of(sx), np_of(yp)
    Q13, S13, Q2, S2 = np_of(q13), np_of(s13), np_of(q2), np_of(s2)
    worst = 0.0
    for e in range(w.E):
        r0, n = int(lay["offsets"][e]), int(lay["kept"][e])
        if n == 0:
            continue
        ref = oracle.expert_ffn_fp8(xq_h[r0:r0 + n], sx_h[r0:r0 + n], Q13[e], S13[e], Q2[e], S2[e], w.I,
                                    rounded=False)
        worst = max(worst, rel_err(y_h[r0:r0 + n], ref, "bf16"))
    assert worst <= TOL["bf16"], worst


def check_layer_fp8(w, sample=None, seed=0):
    inp = device.layer_inputs(w)
    q13, s13, q2, s2 = _fp8_weights(inp)
    cfg = moe.config_from(w)
    T, K = w.T, w.K
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(logits=torch.empty(T, w.E, device="cuda"), topk_ids=torch.empty(T, K, **i32),
             topk_w=torch.empty(T, K, device="cuda"), slot=torch.empty(T, K, **i32))
    y = torch.empty(T, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward_fp8(cfg, inp["x"], inp["w_r"], inp["logit_offset"], inp["sel_bias"], q13, s13, q2, s2, y,
                              moe.layer_out(**o), moe.alloc_workspace(cfg, moe.MOE_OP_LAYER_FP8))
    assert moe.moe_check() == 0
    h = {k: (np_of(v) if v is not None else None) for k, v in inp.items() if k in ("x", "w_r", "sel_bias",
                                                                                      "logit_offset")}
    L = oracle.router_logits(h["x"], h["w_r"], w.dtype, h["logit_offset"])
    ids, wts, keys, allowed = oracle.route(L, w, h["sel_bias"])
    gids = np_of(o["topk_ids"])
    bad = np.nonzero((gids != ids).any(axis=1))[0]
    margin = oracle.near_tie_margin(keys, allowed, w)
    assert np.all(margin[bad] < NEAR_TIE), f"routing differs away from a near-tie at tokens {bad[:8]}"
    lay = oracle.dispatch_layout(gids, w)
    assert np.array_equal(np_of(o["slot"]), lay["slot"])
    # weights from the GPU's float32 logits against the oracle's (see check_layer)
    same = np.setdiff1d(np.arange(T), bad)
    dL = float(np.abs(np_of(o["logits"]).astype(np.float64) - L).max())
    np.testing.assert_allclose(np_of(o["topk_w"])[same], wts[same], rtol=2.0 * dL + 2.0 ** -23)
    xq, sx = oracle.quantize_rows_e4m3(oracle.to_f64(h["x"], "bf16"))
    tokens = np.setdiff1d(np.arange(T), bad)
    if sample is not None:
        tokens = np.sort(np.random.default_rng(seed).choice(tokens, size=min(sample, len(tokens)), replace=False))
    # The experts' E4M3 weights of the reference come from the oracle's
    # quantiser.  At full size (about 5 s of oracle time per expert) the GPU's
    # codes are used instead, after two experts' codes matched the oracle's bit
    # for bit (every code is pinned by test_quantize_bit_exact as well).
    Q13, S13, Q2, S2 = np_of(q13), np_of(s13), np_of(q2), np_of(s2)
    full_size = w.h * w.I > 4 << 20
    qw = {}

    def weights(e):
        if e not in qw:
            w13h, w2h = workloads.host_w13(w, e), workloads.host_w2(w, e)
            if not full_size or len(qw) < 2:
                a, sa = oracle.quantize_rows_e4m3(oracle.to_f64(w13h, "bf16"))
                b, sb = oracle.quantize_rows_e4m3(oracle.to_f64(w2h, "bf16"))
                if full_size:
                    assert np.array_equal(a, Q13[e]) and np.array_equal(sa, S13[e])
                    assert np.array_equal(b, Q2[e]) and np.array_equal(sb, S2[e])
                qw[e] = (a, sa, b, sb)
            else:
                qw[e] = (Q13[e], S13[e], Q2[e], S2[e])
        return qw[e]

    ref = np.zeros((len(tokens), w.h))
    for i, t in enumerate(tokens):
        for k in range(K):
            if lay["slot"][t, k] < 0:
                continue
            e = int(gids[t, k])
            yk = oracle.expert_ffn_fp8(xq[t:t + 1], sx[t:t + 1], *weights(e), w.I)
            ref[i] += float(wts[t, k]) * oracle.to_f64(yk, "bf16")[0]
    err = rel_err(np_of(y)[tokens], ref, "bf16")
    log_near_ties(w.name, T, int((margin < NEAR_TIE).sum()), len(bad), len(tokens))
    assert err <= TOL["bf16"], err


@pytest.mark.parametrize("w", SMALL[:2], ids=[w.name for w in SMALL[:2]])
def test_layer_fp8_small(w):
    check_layer_fp8(w)


@pytest.mark.parametrize("name", ["deepseek_v3", "deepseek_v3_decode_T256"])
def test_layer_fp8_full_size_sampled(name):
    check_layer_fp8(workloads.ALL[name], sample=6)


def test_fp8_refuses_unsupported():
    w = workloads.MIXTRAL.replace(name="mixtral_fp8", T=4096)   # 1024 rows per expert: tokens-as-M layer
    cfg = moe.config_from(w)
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_grouped_ffn_fp8(cfg, z, z, z, z, z, z, z, z, z, torch.zeros(1 << 20, dtype=torch.uint8,
                                                                              device="cuda"))
