"""The shared expert and the whole DeepSeek-V3 MoE block on the GPU against the
oracle: the shared FFN alone, the combine with the shared term, and the block
through the C ABI (device and host buffers)."""
import numpy as np
import pytest
import torch

import expert_dispatch_bias_b300 as moe
import oracle
import synth
from synth import device, workloads

from gpu_helpers import TOL, np_of, rel_err
from test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu


def _shared_case(T, h, Is, dtype):
    w = workloads.Workload("shared_case", T=T, h=h, E=8, K=2, I=64, dtype=dtype, score="softmax", shared_I=Is)
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    ys = torch.full((T, h), float("nan"), dtype=inp["x"].dtype, device="cuda")
    ws = moe.alloc_workspace(cfg, moe.MOE_OP_SHARED)
    moe.moe_shared_ffn(cfg, inp["x"], inp["w13s"], inp["w2s"], ys, ws)
    assert moe.moe_check() == 0
    return w, inp, ys


@pytest.mark.parametrize("T,h,Is,dtype", [(1, 256, 128, "bf16"), (130, 256, 384, "bf16"), (300, 512, 256, "bf16"),
                                          (257, 256, 192, "f32"), (40, 768, 2048, "bf16")])
def test_shared_ffn(T, h, Is, dtype):
    w, inp, ys = _shared_case(T, h, Is, dtype)
    ref = oracle.shared_ffn(np_of(inp["x"]), np_of(inp["w13s"]), np_of(inp["w2s"]), w, rounded=False)
    assert rel_err(np_of(ys), ref, dtype) <= TOL[dtype]


def test_shared_ffn_full_size_sampled_rows():
    """The DeepSeek-V3 shared expert (h=7168, intermediate 2048) on 4096 tokens;
    the oracle evaluates a few rows across the m-blocks."""
    w, inp, ys = _shared_case(4096, 7168, 2048, "bf16")
    rows = np.array([0, 1, 127, 128, 2047, 3000, 4094, 4095])
    ref = oracle.shared_ffn(np_of(inp["x"])[rows], np_of(inp["w13s"]), np_of(inp["w2s"]), w, rounded=False)
    assert rel_err(np_of(ys)[rows], ref, "bf16") <= TOL["bf16"]


def test_combine_add():
    w = workloads.DSV3.replace(name="combine_add", T=300, h=512, I=256, shared_I=256)
    cfg = moe.config_from(w)
    rng = np.random.default_rng(3)
    ids = synth.uniform_topk_ids(3, synth.TID_TEST + 30, w.T, w.E, w.K)
    lay = oracle.dispatch_layout(ids, w)
    wts = rng.random((w.T, w.K)).astype(np.float32)
    yp = device.fill_normal(torch.empty(lay["rows"], w.h, dtype=torch.bfloat16, device="cuda"), 3,
                            synth.TID_TEST + 31, 1.0)
    ys = device.fill_normal(torch.empty(w.T, w.h, dtype=torch.bfloat16, device="cuda"), 3, synth.TID_TEST + 32, 1.0)
    y = torch.empty(w.T, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_combine_add(cfg, yp, torch.from_numpy(lay["slot"]).cuda(), torch.from_numpy(wts).cuda(), ys, y)
    assert moe.moe_check() == 0
    ref = oracle.combine_add(np_of(yp), lay["slot"], wts, np_of(ys), w, rounded=False)
    assert rel_err(np_of(y), ref, "bf16") <= TOL["bf16"]


BLOCKS = [
    workloads.DSV3_BLOCK.replace(name="dsv3_block_small", T=256, h=512, I=256, shared_I=256),
    workloads.TINY.replace(name="tiny_block_f32", shared_I=192),
]


@pytest.mark.parametrize("w", BLOCKS, ids=[w.name for w in BLOCKS])
def test_block_small_full_compare(w):
    check_layer(w)


def test_block_full_size_sampled():
    check_layer(workloads.DSV3_BLOCK, sample=6)


def test_block_host_buffers_match_device_call():
    w = BLOCKS[0]
    inp = device.layer_inputs(w)
    cfg = moe.config_from(w)
    y_dev = torch.empty(w.T, w.h, dtype=torch.bfloat16, device="cuda")
    moe.moe_block_forward(cfg, inp["x"], inp["w_r"], None, inp["sel_bias"], inp["w13"], inp["w2"], inp["w13s"],
                          inp["w2s"], y_dev, None, moe.alloc_workspace(cfg, moe.MOE_OP_BLOCK))
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    moe.moe_block_forward_host(cfg, x_host, inp["w_r"], None, inp["sel_bias"], inp["w13"], inp["w2"],
                               inp["w13s"], inp["w2s"], y_host, moe.alloc_workspace(cfg, moe.MOE_OP_BLOCK_HOST))
    assert moe.moe_check() == 0
    assert torch.equal(y_host, y_dev.cpu())
