"""Pins of the oracle's near-tie margins (topk_margin, order_margin, group_margin).

The end-to-end GPU tests excuse a routing difference only at a token whose
margin is below 1e-4, so a margin that comes out too small would silently
excuse real routing errors.  Each margin is pinned three ways, none of which
re-types its formula:

* hand-worked values (golden ``margin_cases.txt``);
* brute force: the margin equals the smallest relative gap over the pairs of
  keys (or group scores) whose order the decision depends on -- a chosen and
  an unchosen key (group) with nothing strictly between them, or two of the
  top K+1 keys with nothing between them -- enumerated pair by pair instead of
  read off a sorted list;
* decision semantics through ``oracle.route``: pushing the critical pair of
  scores together by a bit more than half the oracle's margin changes the
  routing decision (so the margin is not too small), and an adversarial push
  of a quarter of it does not (so it is not too large).

A last test plants plausible mistakes (wrong pair, zero, top-1 group score)
and checks that the pins reject every one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from synth.workloads import Workload


def _cfg(**kw):
    base = dict(name="t", T=1, h=8, E=8, K=2, I=8, dtype="bf16", score="softmax")
    base.update(kw)
    return Workload(**base)


# --------------------------------------------------------------------------- hand-worked
def _cases(golden_dir):
    cases, cur = [], None
    for line in open(os.path.join(golden_dir, "margin_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, *rest = line.split()
        if head == "case":
            cur = {"name": rest[0]}
            cases.append(cur)
        elif head == "cfg":
            cur["cfg"] = {k: int(v) for k, v in (r.split("=") for r in rest)}
        else:
            cur[head] = rest
    return cases


def _close(got, want):
    if math.isinf(want):
        return math.isinf(got)
    return abs(got - want) <= 1e-6 * max(abs(want), 1e-7)


def test_margins_hand_worked(golden_dir):
    cases = _cases(golden_dir)
    assert len(cases) == 8
    for c in cases:
        keys = np.array([c["keys"]], dtype=np.float32)
        kw = c["cfg"]
        cfg = _cfg(E=keys.shape[1], **kw, score="sigmoid")
        allowed = oracle.allowed_experts(keys, cfg)
        assert np.nonzero(allowed[0])[0].tolist() == [int(v) for v in c["allowed"]], c["name"]
        got = {"topk": oracle.topk_margin(keys, allowed, cfg.K)[0],
               "order": oracle.order_margin(keys, allowed, cfg.K)[0],
               "group": oracle.group_margin(keys, cfg)[0]}
        for k, v in got.items():
            assert _close(float(v), float(c[k][0])), (c["name"], k, v, c[k][0])
        assert _close(float(oracle.near_tie_margin(keys, allowed, cfg)[0]),
                      min(float(c["order"][0]), float(c["group"][0])))


# --------------------------------------------------------------------------- brute force
def _rank(keys_row, members):
    """members sorted by key descending, ties to the lower id (the routing order)."""
    return sorted(members, key=lambda e: (-float(keys_row[e]), e))


def _rel(a, b):
    """|a - b| relative to the higher of the two scores compared."""
    hi, lo = (a, b) if float(a) >= float(b) else (b, a)
    return abs(float(hi) - float(lo)) / max(abs(float(hi)), 1e-30)


def _adjacent_gap(vals, side_a, side_b):
    """Smallest relative gap over pairs (i in side_a, j in side_b) with no value of
    `vals` strictly between vals[i] and vals[j]: the comparisons a ranking rests
    on, found pair by pair."""
    best = math.inf
    for i in side_a:
        for j in side_b:
            if i == j:
                continue
            lo, hi = sorted((float(vals[i]), float(vals[j])))
            if any(lo < float(vals[m]) < hi for m in range(len(vals))):
                continue
            best = min(best, _rel(vals[i], vals[j]))
    return best


def _topk_brute(keys_row, allowed_row, K):
    members = [e for e in range(len(keys_row)) if allowed_row[e]]
    chosen = _rank(keys_row, members)[:K]
    rest = [e for e in members if e not in chosen]
    sub = np.full(len(keys_row), np.nan)
    sub[members] = keys_row[members]      # only allowed keys can lie between
    return _adjacent_gap(np.where(np.isnan(sub), -np.inf, sub), chosen, rest)


def _order_brute(keys_row, allowed_row, K):
    members = [e for e in range(len(keys_row)) if allowed_row[e]]
    top = _rank(keys_row, members)[:K + 1]
    sub = np.full(len(keys_row), -np.inf)
    sub[top] = keys_row[top]              # only the top K+1 keys are ordered
    return _adjacent_gap(sub, top, top)


def _group_scores(keys_row, cfg):
    gs = cfg.E // cfg.n_groups
    return [sum(sorted(keys_row[g * gs:(g + 1) * gs].tolist(), reverse=True)[:cfg.group_topn])
            for g in range(cfg.n_groups)]


def _group_brute(keys_row, allowed_row, cfg):
    if cfg.n_groups <= 0 or cfg.topk_groups >= cfg.n_groups:
        return math.inf
    gs = cfg.E // cfg.n_groups
    sc = _group_scores(keys_row, cfg)
    kept = [g for g in range(cfg.n_groups) if allowed_row[g * gs]]
    assert len(kept) == cfg.topk_groups
    return _adjacent_gap(sc, kept, [g for g in range(cfg.n_groups) if g not in kept])


@pytest.mark.parametrize("seed", range(5))
def test_margins_brute_force(seed):
    """Quantised keys force exact ties; continuous keys give generic gaps."""
    rng = np.random.default_rng(100 + seed)
    for quant in (True, False):
        for E, K, G, M, n in ((8, 3, 0, 0, 0), (8, 2, 4, 2, 2), (12, 3, 4, 2, 1), (6, 5, 0, 0, 0)):
            T = 40
            keys = rng.normal(size=(T, E))
            keys = (np.round(keys * 4) / 4 if quant else keys).astype(np.float32)
            cfg = _cfg(T=T, E=E, K=K, n_groups=G, topk_groups=M, group_topn=n, score="sigmoid")
            allowed = oracle.allowed_experts(keys, cfg)
            tk = oracle.topk_margin(keys, allowed, K)
            om = oracle.order_margin(keys, allowed, K)
            gm = oracle.group_margin(keys, cfg)
            for t in range(T):
                assert _close(tk[t], _topk_brute(keys[t], allowed[t], K))
                assert _close(om[t], _order_brute(keys[t], allowed[t], K))
                assert _close(gm[t], _group_brute(keys[t], allowed[t], cfg))
                assert om[t] <= tk[t]


# --------------------------------------------------------------------------- decision semantics
# The checks below return the list of violations they find, so that the
# planted-mistake test can run them on wrong margin functions.
PUSH_OVER = 0.51    # x margin: pushes the critical pair past each other
PUSH_UNDER = 0.25   # x margin: must not change the decision


def _softmax_case(seed, T=60, E=8, K=3):
    """Logits in [1, 2] with every adjacent gap > 1e-3 (no near-ties to blur the
    checks); softmax without bias or groups ranks the logits themselves."""
    rng = np.random.default_rng(seed)
    rows = []
    while len(rows) < T:
        v = rng.uniform(1.0, 2.0, size=E)
        s = np.sort(v)
        if np.min(np.diff(s)) > 1e-3:
            rows.append(v)
    return np.array(rows, dtype=np.float32), _cfg(T=T, E=E, K=K, score="softmax")


def _push(L, hi, lo, d_hi, d_lo):
    """Lowers logit `hi` by d_hi and raises logit `lo` by d_lo (float32)."""
    P = L.astype(np.float64).copy()
    P[hi] -= d_hi
    P[lo] += d_lo
    return P.astype(np.float32)[None, :]


def check_topk(margin_fn, seed=0):
    L, cfg = _softmax_case(seed)
    allowed = np.ones(L.shape, dtype=bool)
    m = margin_fn(L, allowed, cfg.K)
    ids, _, _, _ = oracle.route(L, cfg)
    bad = []
    for t in range(L.shape[0]):
        r = _rank(L[t], range(cfg.E))
        a, b = r[cfg.K - 1], r[cfg.K]           # the pair the set decision compares
        over = _push(L[t], a, b, PUSH_OVER * m[t] * abs(L[t, a]), PUSH_OVER * m[t] * abs(L[t, a]))
        if set(oracle.route(over, cfg)[0][0].tolist()) == set(ids[t].tolist()):
            bad.append((t, "a push of 0.51 x margin left the set unchanged"))
        under = _push(L[t], a, b, PUSH_UNDER * m[t] * abs(L[t, a]), PUSH_UNDER * m[t] * abs(L[t, b]))
        if np.isfinite(m[t]) and set(oracle.route(under, cfg)[0][0].tolist()) != set(ids[t].tolist()):
            bad.append((t, "a push of 0.25 x margin changed the set"))
    return bad


def check_order(margin_fn, seed=0):
    L, cfg = _softmax_case(seed)
    allowed = np.ones(L.shape, dtype=bool)
    m = margin_fn(L, allowed, cfg.K)
    ids, _, _, _ = oracle.route(L, cfg)
    bad = []
    for t in range(L.shape[0]):
        r = _rank(L[t], range(cfg.E))[:cfg.K + 1]
        # the adjacent pair of the top K+1 that is closest, found by enumeration
        i = min(range(cfg.K), key=lambda i: _rel(L[t, r[i]], L[t, r[i + 1]]))
        a, b = r[i], r[i + 1]
        over = _push(L[t], a, b, PUSH_OVER * m[t] * abs(L[t, a]), PUSH_OVER * m[t] * abs(L[t, a]))
        if oracle.route(over, cfg)[0][0].tolist() == ids[t].tolist():
            bad.append((t, "a push of 0.51 x margin left the ordered ids unchanged"))
        # adversary: every adjacent pair of the top K+1 pushed together by 0.25 x margin
        P = L[t].astype(np.float64).copy()
        for j in range(cfg.K + 1):
            P[r[j]] += (-1.0 if j % 2 == 0 else 1.0) * PUSH_UNDER * m[t] * abs(L[t, r[j]])
        if oracle.route(P.astype(np.float32)[None, :], cfg)[0][0].tolist() != ids[t].tolist():
            bad.append((t, "pushes of 0.25 x margin changed the ordered ids"))
    return bad


def _group_case(seed, T=40, E=16, G=4, M=2, n=2):
    """Sigmoid keys plus a bias: shifting the bias of every expert of a group by d
    shifts that group's score by n*d (up to float32 rounding), so the bias
    steers the group decision directly."""
    rng = np.random.default_rng(seed)
    cfg = _cfg(T=1, E=E, K=2, n_groups=G, topk_groups=M, group_topn=n, score="sigmoid")
    out = []
    while len(out) < T:
        L = rng.normal(size=(1, E)).astype(np.float32)
        bias = rng.uniform(0.5, 0.6, size=E).astype(np.float32)
        keys = oracle.selection_keys(L, cfg, bias)
        sc = sorted(_group_scores(keys[0], cfg), reverse=True)
        if min(_rel(a, b) for a, b in zip(sc, sc[1:])) > 1e-3:
            out.append((L, bias))
    return out, cfg


def check_group(margin_fn, seed=0):
    cases, cfg = _group_case(seed)
    gs = cfg.E // cfg.n_groups
    bad = []
    for t, (L, bias) in enumerate(cases):
        keys = oracle.selection_keys(L, cfg, bias)
        allowed = oracle.allowed_experts(keys, cfg)
        m = float(margin_fn(keys, cfg)[0])
        sc = _group_scores(keys[0], cfg)
        order = sorted(range(cfg.n_groups), key=lambda g: (-sc[g], g))
        a, b = order[cfg.topk_groups - 1], order[cfg.topk_groups]   # last kept, first dropped
        for frac, should_change in ((PUSH_OVER, True), (PUSH_UNDER, False)):
            d = frac * m * abs(sc[a]) / cfg.group_topn
            bb = bias.astype(np.float64).copy()
            bb[a * gs:(a + 1) * gs] -= d
            bb[b * gs:(b + 1) * gs] += d if should_change else frac * m * abs(sc[b]) / cfg.group_topn
            k2 = oracle.selection_keys(L, cfg, bb.astype(np.float32))
            changed = not np.array_equal(oracle.allowed_experts(k2, cfg), allowed)
            if changed != should_change:
                bad.append((t, f"a push of {frac} x margin {'kept' if should_change else 'changed'} the groups"))
    return bad


@pytest.mark.parametrize("seed", range(3))
def test_topk_margin_is_the_set_decision_boundary(seed):
    assert check_topk(oracle.topk_margin, seed) == []


@pytest.mark.parametrize("seed", range(3))
def test_order_margin_is_the_order_decision_boundary(seed):
    assert check_order(oracle.order_margin, seed) == []


@pytest.mark.parametrize("seed", range(3))
def test_group_margin_is_the_group_decision_boundary(seed):
    assert check_group(oracle.group_margin, seed) == []


# --------------------------------------------------------------------------- planted mistakes
def _wrong_pair_topk(keys, allowed, K):
    """(K-1)-th against K-th: the gap inside the chosen set."""
    out = np.full(keys.shape[0], np.inf)
    for t in range(keys.shape[0]):
        v = sorted(keys[t][allowed[t]].astype(np.float64).tolist(), reverse=True)
        if len(v) > K and K >= 2:
            out[t] = abs(v[K - 2] - v[K - 1]) / abs(v[K - 2])
    return out


def _zero_topk(keys, allowed, K):
    return np.zeros(keys.shape[0])


def _set_only_order(keys, allowed, K):
    """Forgets that two chosen experts may swap places."""
    return oracle.topk_margin(keys, allowed, K)


def _top1_group(keys, cfg):
    return oracle.group_margin(keys, cfg.replace(group_topn=1))


def _wrong_pair_group(keys, cfg):
    return oracle.group_margin(keys, cfg.replace(topk_groups=cfg.topk_groups - 1))


def _zero_group(keys, cfg):
    return np.zeros(keys.shape[0])


@pytest.mark.parametrize("check,fn", [
    (check_topk, _wrong_pair_topk), (check_topk, _zero_topk), (check_order, _set_only_order),
    (check_order, _zero_topk), (check_group, _top1_group), (check_group, _wrong_pair_group),
    (check_group, _zero_group)],
    ids=["topk-wrong-pair", "topk-zero", "order-set-only", "order-zero", "group-top1", "group-wrong-pair",
         "group-zero"])
def test_planted_mistakes_fail_the_pins(check, fn):
    assert len(check(fn)) > 0
