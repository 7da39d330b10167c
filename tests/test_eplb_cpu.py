"""The library's host EPLB planner (moe_eplb_plan, no GPU needed) against the
oracle's plan: identical integer outputs for many count vectors."""
import numpy as np
import pytest

import expert_dispatch_bias_b300 as moe
import oracle
from synth import workloads


def _same(counts, n_ep, R):
    E = len(counts)
    got = moe.moe_eplb_plan(E, n_ep, R, counts)
    ref = oracle.eplb_plan(counts, n_ep, R)
    for k in ("rep_offsets", "rep_phys", "phys_to_log", "rank_load"):
        assert np.array_equal(got[k], ref[k]), (k, counts, n_ep, R)


@pytest.mark.parametrize("seed", range(40))
def test_plan_matches_oracle_random(seed):
    rng = np.random.default_rng(seed)
    n_ep = int(rng.choice([1, 2, 4, 8, 16]))
    E = n_ep * int(rng.integers(1, 9))
    R = n_ep * int(rng.integers(0, 4))
    counts = rng.integers(0, 5000, size=E) * (rng.random(E) < 0.8)
    if seed % 5 == 0:
        counts[:] = 7            # all equal: every tie rule decides
    _same(counts.tolist(), n_ep, R)


def test_plan_matches_oracle_skewed_workloads():
    """Zipf-skewed expert loads of the Switch-shaped layer (hottest expert ~29x
    the mean) and DeepSeek-V3-like uniform ones, with the replica budgets of the
    benchmark workloads."""
    p = np.arange(1, 129, dtype=np.float64) ** -1.1
    counts = np.floor(16384 * p / p.sum()).astype(np.int64)
    _same(counts.tolist(), 16, 16)
    rng = np.random.default_rng(1)
    _same(rng.binomial(32768, 1 / 256, size=256).tolist(), 64, 64)


def test_plan_rejects_bad_arguments():
    with pytest.raises(moe.MoeError):
        moe.moe_eplb_plan(8, 3, 0, [1] * 8)          # 8 physical experts on 3 ranks
    with pytest.raises(moe.MoeError):
        moe.moe_eplb_plan(8, 4, -4, [1] * 8)
