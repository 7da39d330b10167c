"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import expert_dispatch_bias_b300 as moe
    declared = _declared_functions()
    assert len(declared) >= 14
    lib = ctypes.CDLL(moe.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(moe.EXPORTS) == declared


def test_no_oracle_or_cpu_fallback_in_product():
    pkg = os.path.join(ROOT, "expert_dispatch_bias_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def _cfg(**kw):
    import expert_dispatch_bias_b300 as moe
    base = dict(T=4096, h=7168, E=256, K=8, I=2048, dtype="bf16", score="sigmoid", renormalize=1, scale=2.5,
                n_groups=8, topk_groups=4, group_topn=2, capacity=0, pad=0, ep_size=64)
    base.update(kw)
    return moe.make_config(**base)


def test_rows_and_workspace_sizes():
    import expert_dispatch_bias_b300 as moe
    assert moe.moe_rows(_cfg()) == 4096 * 8
    assert moe.moe_rows(_cfg(capacity=100, pad=1)) == 256 * 100
    assert moe.moe_rows(_cfg(capacity=100, pad=0)) == 4096 * 8
    ffn = moe.moe_workspace_size(_cfg(), moe.MOE_OP_FFN)
    assert ffn >= 4096 * 8 * 2048 * 2
    layer = moe.moe_workspace_size(_cfg(), moe.MOE_OP_LAYER)
    assert layer >= ffn + 2 * 4096 * 8 * 7168 * 2
    host = moe.moe_workspace_size(_cfg(), moe.MOE_OP_LAYER_HOST)
    assert host >= layer + 2 * 4096 * 7168 * 2
    assert moe.moe_workspace_size(_cfg(T=0), moe.MOE_OP_LAYOUT) > 0
    # router logits: float32 partial sums of up to 8 slices of h, inside the layer's too
    logits = moe.moe_workspace_size(_cfg(), moe.MOE_OP_LOGITS)
    assert logits >= 8 * 4096 * 256 * 4
    assert layer >= logits + ffn + 2 * 4096 * 8 * 7168 * 2


@pytest.mark.parametrize("bad", [
    dict(h=100), dict(I=96), dict(E=0), dict(E=2048), dict(K=0), dict(K=17), dict(dtype=7), dict(score=5),
    dict(n_groups=7), dict(topk_groups=9), dict(group_topn=33), dict(topk_groups=1, K=64),
    dict(ep_size=3), dict(capacity=-1), dict(pad=1, capacity=0), dict(T=-1), dict(renormalize=2),
])
def test_invalid_configs_rejected(bad):
    import expert_dispatch_bias_b300 as moe
    cfg = _cfg(**bad)
    if "dtype" in bad:
        cfg.dtype = bad["dtype"]
    if "score" in bad:
        cfg.score = bad["score"]
    assert moe.moe_validate_config(cfg) == 1


def test_unsupported_group_topn():
    import expert_dispatch_bias_b300 as moe
    assert moe.moe_validate_config(_cfg(group_topn=9)) == 2


def test_argument_errors_before_any_launch():
    """Null and misaligned pointers are refused on the host (no CUDA call runs)."""
    import expert_dispatch_bias_b300 as moe
    lib = moe.lib
    cfg = _cfg()
    # moe_route with NULL logits
    st = lib.moe_route(ctypes.byref(cfg), None, None, 4096, 4096, None)
    assert st == 1
    # misaligned int32 output
    st = lib.moe_route(ctypes.byref(cfg), 4096, None, 4098, 4096, None)
    assert st == 3
    # layer with a misaligned activation pointer
    st = lib.moe_layer_forward(ctypes.byref(cfg), 4104, 4096, None, None, 4096, 4096, 4096, None, 4096,
                               1 << 40, None)
    assert st == 3
    # workspace too small
    st = lib.moe_grouped_ffn(ctypes.byref(cfg), 4096, 4096, 4096, 4096, 4096, 4096, 4096, 1024, None)
    assert st == 4
    assert lib.moe_status_string(6) == b"MOE_ERR_DEVICE_TIMEOUT"
    # bf16 router logits need their workspace (the partial sums of the h slices)
    need = moe.moe_workspace_size(cfg, moe.MOE_OP_LOGITS)
    st = lib.moe_router_logits(ctypes.byref(cfg), 4096, 4096, None, 4096, None, need, None)
    assert st == 1
    st = lib.moe_router_logits(ctypes.byref(cfg), 4096, 4096, None, 4096, 4096 + 128, need, None)
    assert st == 3
    st = lib.moe_router_logits(ctypes.byref(cfg), 4096, 4096, None, 4096, 4096, need - 1, None)
    assert st == 4


def test_launch_count_host_only():
    """The launch counter is host state: readable without a GPU, and no call
    refused on the host (no launch) moves it."""
    import expert_dispatch_bias_b300 as moe
    n0 = moe.moe_launch_count()
    assert n0 >= 0
    cfg = _cfg()
    assert moe.lib.moe_route(ctypes.byref(cfg), None, None, 4096, 4096, None) == 1
    assert moe.moe_launch_count() == n0
