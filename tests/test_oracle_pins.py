"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test ties an oracle function to something other than itself: numbers the
pages print, closed forms under uniform routing, hand-worked cases, brute-force
enumeration on tiny inputs, or a library routine.  A plausible slip in the
oracle (a dropped bias or offset, reversed order or tie rule, wrong group
score, biased combine weights, transposed n_ij, swapped gate/up, an
inclusive scan) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth
from synth.workloads import Workload


def _cfg(**kw):
    base = dict(name="t", T=4, h=8, E=4, K=2, I=8, dtype="bf16", score="softmax")
    base.update(kw)
    return Workload(**base)


# --------------------------------------------------------------------------- volumes
def _parse_bytes(tok):
    for unit, mul in (("MB", 1e6), ("KB", 1e3)):
        if tok.endswith(unit):
            return tok[:-len(unit)], mul
    raise ValueError(tok)


def _truncates_to(value_bytes, printed):
    digits, mul = _parse_bytes(printed)
    dec = len(digits.split(".")[1]) if "." in digits else 0
    q = 10 ** dec
    return math.floor(value_bytes / mul * q) / q == float(digits)


def test_ep_volume_table(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "ep_volume_table.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for model, B, K, h, N, chip, pair, flag in rows:
        v = oracle.ep_volumes(int(B), int(K), int(h), 2, int(N))
        assert v["total"] == int(B) * int(K) * int(h) * 2
        assert _truncates_to(v["per_chip"], chip), (model, N, v["per_chip"], chip)
        if flag == "ok":
            assert _truncates_to(v["pair"], pair), (model, N, v["pair"], pair)
        else:
            # The page's own formula gives 114688 B; the printed cell is off.
            assert v["pair"] == 114688
            assert not _truncates_to(v["pair"], pair)


def _uniform_layout(seed, T, E, K, N, h=7168):
    ids = synth.uniform_topk_ids(seed, synth.TID_TEST, T, E, K)
    cfg = _cfg(T=T, E=E, K=K, h=h, ep_size=N)
    return ids, oracle.dispatch_layout(ids, cfg)


def test_dispatch_volume_formulas_exact():
    """Dropless: sum_ij C[i][j] = B*K*h*dtype and every chip sends (B*K/N_EP)*h*dtype,
    so the pair mean is m_pair (eqs. par-ep-comm-total / per-chip / pair)."""
    T, E, K, N, h = 4096, 256, 8, 64, 7168
    ids, lay = _uniform_layout(3, T, E, K, N, h)
    v = oracle.ep_volumes(T, K, h, 2, N)
    C = lay["n_ij"] * h * 2
    assert C.sum() == v["total"]
    assert np.all(lay["sent_bytes"] == v["per_chip"])
    assert C.mean() == v["pair"]
    assert lay["dropped"] == 0 and lay["counts"].sum() == T * K


def test_uniform_routing_sparsity_closed_form(golden_dir):
    """EP=64, 512 tokens, top-8 of 256: ~36% empty chip pairs, ~30-50 targets."""
    g = dict(l.split() for l in open(os.path.join(golden_dir, "ep_uniform_sparsity.txt"))
             if l.strip() and not l.startswith("#"))
    N, B, K, E, epr = int(g["EP"]), int(g["B"]), int(g["K"]), int(g["E"]), int(g["experts_per_chip"])
    p_empty = (math.comb(E - epr, K) / math.comb(E, K)) ** (B // N)
    targets = N * (1 - p_empty)
    assert abs(p_empty - float(g["printed_empty_pair_fraction"])) < 0.005
    assert float(g["printed_target_chips_low"]) <= targets <= float(g["printed_target_chips_high"])
    empties, tg = [], []
    for seed in range(60):
        _, lay = _uniform_layout(seed, B, E, K, N)
        nz = lay["n_ij"] > 0
        empties.append(1.0 - nz.mean())
        tg.append(nz.sum(axis=1).mean())
    assert abs(np.mean(empties) - p_empty) < 0.005
    assert abs(np.mean(tg) - targets) < 0.3


def test_pair_volume_expectation_uniform():
    """Every chip pair receives m_pair in expectation under uniform routing."""
    T, E, K, N = 4096, 256, 8, 64
    acc = np.zeros((N, N))
    trials = 12
    for seed in range(trials):
        _, lay = _uniform_layout(100 + seed, T, E, K, N)
        acc += lay["n_ij"]
    mean = acc / trials
    expect = (T / N) * K / N
    # per-token hits on one chip: hypergeometric(E, epr, K); 64 tokens per pair
    var = (T / N) * K * (4 / E) * (1 - 4 / E) * (E - K) / (E - 1)
    assert abs(mean.mean() - expect) < 1e-9
    assert np.abs(mean - expect).max() < 6 * math.sqrt(var / trials)


@pytest.mark.parametrize("T", [32, 256])
def test_active_experts_balls_into_bins(T):
    """Experts touched per chip vs the balls-into-bins estimate (eq. par-ep-active-experts).
    The estimate treats each of the T*K picks as independent; the exact expectation
    for K distinct experts per token is E/P * (1 - (1 - K/E)**T)."""
    E, K, P = 256, 8, 64
    exact = (E / P) * (1 - (1 - K / E) ** T)
    page = oracle.active_experts_per_chip(E, P, T, K)
    assert abs(page - exact) / exact < 0.01
    touched = [(_uniform_layout(seed, T, E, K, P)[1]["experts_touched"]) / P for seed in range(150)]
    assert abs(np.mean(touched) - exact) < 0.05


# --------------------------------------------------------------------------- routing
def _route_cases(golden_dir):
    cases, cur = [], None
    for line in open(os.path.join(golden_dir, "route_cases.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, *rest = line.split()
        if head == "case":
            cur = {"name": rest[0]}
            cases.append(cur)
        elif head == "cfg":
            cur["cfg"] = {k: v for k, v in (r.split("=") for r in rest)}
        else:
            cur[head] = rest
    return cases


def test_route_hand_worked(golden_dir):
    cases = _route_cases(golden_dir)
    assert len(cases) == 7
    for c in cases:
        L = np.array([c["logits"]], dtype=np.float32)
        E = L.shape[1]
        kw = c["cfg"]
        cfg = _cfg(E=E, K=int(kw["K"]), score=kw["score"], renormalize=int(kw["renormalize"]),
                   scale=float(kw["scale"]), n_groups=int(kw["n_groups"]),
                   topk_groups=int(kw["topk_groups"]), group_topn=int(kw["group_topn"]))
        bias = np.array(c["bias"], dtype=np.float32) if "bias" in c else None
        ids, w, _, _ = oracle.route(L, cfg, bias)
        assert ids[0].tolist() == [int(v) for v in c["ids"]], c["name"]
        np.testing.assert_allclose(w[0], np.array(c["weights"], dtype=np.float64), rtol=2e-7,
                                   err_msg=c["name"])


def _beats(ka, a, kb, b):
    return ka > kb or (ka == kb and a < b)


@pytest.mark.parametrize("seed", range(6))
def test_route_brute_force(seed):
    """Enumerate every group subset and every expert subset on tiny inputs: exactly one
    subset dominates its complement, and it is the oracle's choice, in order."""
    rng = np.random.default_rng(seed)
    E, G = 8, 4
    for score, groups in (("softmax", 0), ("sigmoid", 0), ("sigmoid", G)):
        T, K = 12, 3
        # quantised logits force exact ties
        L = (rng.integers(-4, 5, size=(T, E)) / 4.0).astype(np.float32)
        bias = (rng.integers(-2, 3, size=E) / 16.0).astype(np.float32) if score == "sigmoid" else None
        cfg = _cfg(T=T, E=E, K=K, score=score, n_groups=groups, topk_groups=2 if groups else 0,
                   group_topn=2 if groups else 0)
        ids, _, keys, _ = oracle.route(L, cfg, bias)
        for t in range(T):
            if score == "sigmoid":
                s = 1.0 / (1.0 + np.exp(-L[t].astype(np.float64)))
                k = (s + (bias.astype(np.float64) if bias is not None else 0.0)).astype(np.float32)
            else:
                k = L[t]
            allowed = list(range(E))
            if groups:
                gs = E // G
                gsc = []
                for g in range(G):
                    a, b = sorted(k[g * gs:(g + 1) * gs].tolist(), reverse=True)[:2]
                    gsc.append(np.float32(np.float32(a) + np.float32(b)))
                winners = [S for S in itertools.combinations(range(G), 2)
                           if all(_beats(gsc[x], x, gsc[y], y) for x in S for y in range(G) if y not in S)]
                assert len(winners) == 1
                allowed = [e for e in range(E) if e // gs in winners[0]]
            winners = [S for S in itertools.combinations(allowed, K)
                       if all(_beats(k[x], x, k[y], y) for x in S for y in allowed if y not in S)]
            assert len(winners) == 1
            assert sorted(ids[t].tolist()) == sorted(winners[0])
            for i in range(K - 1):
                assert _beats(k[ids[t, i]], ids[t, i], k[ids[t, i + 1]], ids[t, i + 1])


def test_route_weights_library():
    """With K = E every expert is chosen: renormalised softmax weights are the full
    softmax; renormalised sigmoid weights are expit / sum(expit)."""
    rng = np.random.default_rng(7)
    L = rng.normal(size=(16, 8)).astype(np.float32)
    _, w, _, _ = oracle.route(L, _cfg(E=8, K=8, score="softmax"))
    ids, _, _, _ = oracle.route(L, _cfg(E=8, K=8, score="softmax"))
    ref = scipy.special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids.astype(np.int64), 1), rtol=1e-6)
    cfg = _cfg(E=8, K=8, score="sigmoid", scale=2.5)
    ids, w, _, _ = oracle.route(L, cfg)
    s = scipy.special.expit(L.astype(np.float64))
    ref = 2.5 * s / s.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids.astype(np.int64), 1), rtol=1e-6)
    # without renormalisation the softmax weight is the probability itself
    ids, w, _, _ = oracle.route(L, _cfg(E=8, K=2, score="softmax", renormalize=0))
    ref = scipy.special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(ref, ids.astype(np.int64), 1), rtol=1e-6)


def test_router_logits_library():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 24)).astype(np.float32)
    wr = rng.normal(size=(6, 24)).astype(np.float32)
    o = rng.normal(size=6).astype(np.float32)
    L = oracle.router_logits(x, wr, "f32", o)
    ref = torch.nn.functional.linear(torch.from_numpy(x).double(), torch.from_numpy(wr).double(),
                                     torch.from_numpy(o).double()).numpy()
    np.testing.assert_allclose(L, ref, rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------- layout
def _layout_blocks(golden_dir):
    head, blocks, cur = {}, [], None
    for line in open(os.path.join(golden_dir, "layout_case.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        k, *v = line.split()
        if k == "mode":
            cur = {"mode": dict(x.split("=") for x in v)}
        elif k == "end":
            blocks.append(cur)
            cur = None
        elif cur is None:
            head[k] = v
        else:
            cur[k] = v
    return head, blocks


def test_layout_hand_worked(golden_dir):
    head, blocks = _layout_blocks(golden_dir)
    T, K, E = int(head["T"][0]), int(head["K"][0]), int(head["E"][0])
    ids = np.array([int(v) for v in head["ids"]]).reshape(T, K)
    assert len(blocks) == 3
    for b in blocks:
        cfg = _cfg(T=T, K=K, E=E, h=int(head["h"][0]), ep_size=int(head["ep"][0]),
                   capacity=int(b["mode"]["capacity"]), pad=int(b["mode"]["pad"]))
        lay = oracle.dispatch_layout(ids, cfg)
        for key in ("counts", "kept", "offsets", "row_src", "sent_bytes", "recv_bytes"):
            assert lay[key].tolist() == [int(v) for v in b[key]], (b["mode"], key)
        assert lay["slot"].reshape(-1).tolist() == [int(v) for v in b["slot"]]
        assert lay["n_ij"].reshape(-1).tolist() == [int(v) for v in b["n_ij"]]
        assert lay["dropped"] == int(b["dropped"][0])
        assert lay["balancedness"] == np.float32(float(b["balancedness"][0]))


@pytest.mark.parametrize("cap,pad", [(0, 0), (7, 0), (7, 1), (1, 0)])
def test_layout_invariants(cap, pad):
    rng = np.random.default_rng(cap * 10 + pad)
    T, E, K, N = 96, 16, 3, 4
    # skewed routing: expert popularity ~ Zipf
    p = 1.0 / np.arange(1, E + 1)
    ids = np.stack([rng.choice(E, size=K, replace=False, p=p / p.sum()) for _ in range(T)]).astype(np.int32)
    cfg = _cfg(T=T, E=E, K=K, ep_size=N, capacity=cap, pad=pad)
    lay = oracle.dispatch_layout(ids, cfg)
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert lay["counts"].tolist() == counts.tolist()
    assert counts.sum() == T * K
    if cap > 0:
        assert np.all(lay["kept"] <= cap)
    slot = lay["slot"]
    used = slot[slot >= 0]
    assert len(np.unique(used)) == len(used)                       # injective
    R = lay["rows"]
    assert R == (E * cap if (pad and cap) else T * K)
    assert np.all((used >= 0) & (used < R))
    for r in range(R):                                             # row_src inverts slot
        t = lay["row_src"][r]
        if t >= 0:
            assert r in slot[t].tolist()
    for e in range(E):                                             # drops in token order
        toks = [t for t in range(T) if e in ids[t].tolist()]
        kept_toks = [t for t in toks if slot[t, ids[t].tolist().index(e)] >= 0]
        assert kept_toks == toks[:len(kept_toks)]
        assert len(kept_toks) == (min(len(toks), cap) if cap > 0 else len(toks))
        rows = sorted(slot[t, ids[t].tolist().index(e)] for t in kept_toks)
        lo = lay["offsets"][e]
        assert rows == list(range(lo, lo + len(rows)))             # contiguous segment
    assert lay["n_ij"].sum() == T * K - lay["dropped"]
    if cap <= 0:
        assert np.all(lay["n_ij"].sum(axis=1) == (T // N) * K)


# --------------------------------------------------------------------------- permute/ffn/combine
def test_identity_experts_combine():
    """With identity experts the combine returns (sum of kept weights) * x."""
    T, h, E, K = 40, 16, 6, 3
    cfg = _cfg(T=T, h=h, E=E, K=K, dtype="f32", capacity=17, ep_size=2)
    rng = np.random.default_rng(5)
    x = rng.normal(size=(T, h)).astype(np.float32)
    L = rng.normal(size=(T, E)).astype(np.float32)
    ids, w, _, _ = oracle.route(L, cfg)
    lay = oracle.dispatch_layout(ids, cfg)
    assert lay["dropped"] > 0
    xp = oracle.permute(x, lay["row_src"])
    y = oracle.combine(xp, lay["slot"], w, cfg)
    wk = np.where(lay["slot"] >= 0, w.astype(np.float64), 0.0).sum(axis=1)
    np.testing.assert_allclose(y, wk[:, None] * x.astype(np.float64), rtol=1e-6, atol=1e-7)


def test_expert_ffn_library_and_brute_force():
    h, I, n = 24, 40, 7
    rng = np.random.default_rng(11)
    x = rng.normal(size=(n, h)).astype(np.float32)
    w13 = rng.normal(size=(2 * I, h)).astype(np.float32) / 4
    w2 = rng.normal(size=(h, I)).astype(np.float32) / 4
    y = oracle.expert_ffn(x, w13, w2, "f32", I)
    tx, t13, t2 = (torch.from_numpy(a).double() for a in (x, w13, w2))
    F = torch.nn.functional
    ref = F.linear(F.silu(F.linear(tx, t13[:I])) * F.linear(tx, t13[I:]), t2).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-5, atol=1e-6)
    # element (1, 3) by explicit sums
    r, j = 1, 3
    g = [math.fsum(float(x[r, c]) * float(w13[i, c]) for c in range(h)) for i in range(I)]
    u = [math.fsum(float(x[r, c]) * float(w13[I + i, c]) for c in range(h)) for i in range(I)]
    a = [float(np.float32(gi / (1 + math.exp(-gi)) * ui)) for gi, ui in zip(g, u)]
    assert abs(math.fsum(a[i] * float(w2[j, i]) for i in range(I)) - float(y[r, j])) < 1e-5


def test_layer_matches_per_token_sum():
    """Whole layer vs a per-token evaluation that bypasses the permutation:
    y[t] = sum_k w[t,k] * FFN_{ids[t,k]}(x[t]) over kept (t, k)."""
    cfg = _cfg(T=24, h=16, E=4, K=2, I=12, dtype="f32", capacity=10, ep_size=2)
    rng = np.random.default_rng(2)
    x = rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)
    wr = rng.normal(size=(cfg.E, cfg.h)).astype(np.float32)
    W13 = [rng.normal(size=(2 * cfg.I, cfg.h)).astype(np.float32) for _ in range(cfg.E)]
    W2 = [rng.normal(size=(cfg.h, cfg.I)).astype(np.float32) for _ in range(cfg.E)]
    out = oracle.layer_forward(x, wr, lambda e: W13[e], lambda e: W2[e], cfg)
    F = torch.nn.functional
    for t in range(cfg.T):
        ref = np.zeros(cfg.h)
        for k in range(cfg.K):
            if out["layout"]["slot"][t, k] < 0:
                continue
            e = out["ids"][t, k]
            xt = torch.from_numpy(x[t:t + 1]).double()
            w13 = torch.from_numpy(W13[e]).double()
            a = (F.silu(F.linear(xt, w13[:cfg.I])) * F.linear(xt, w13[cfg.I:])).float().double()
            ref += float(out["w"][t, k]) * F.linear(a, torch.from_numpy(W2[e]).double()).float().double().numpy()[0]
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-5, atol=1e-5)


def test_bf16_rounding(golden_dir):
    vals, bits = [], []
    for line in open(os.path.join(golden_dir, "bf16_rounding.txt")):
        line = line.split("#")[0].strip()
        if line:
            v, b = line.split()
            vals.append(float(v))
            bits.append(int(b, 16))
    v = np.array(vals, dtype=np.float64)
    assert oracle.round_to_bf16_bits(v).tolist() == bits
    assert synth.f32_to_bf16_bits(v.astype(np.float32)).tolist() == bits


# --------------------------------------------------------------------------- shared expert
def _block_case(dtype, seed=4):
    cfg = _cfg(T=20, h=16, E=4, K=2, I=12, dtype=dtype, score="sigmoid", scale=2.5, ep_size=2, shared_I=12)
    rng = np.random.default_rng(seed)
    mk = (lambda shape, s: synth.f32_to_bf16_bits((rng.normal(size=shape) * s).astype(np.float32))) \
        if dtype == "bf16" else (lambda shape, s: (rng.normal(size=shape) * s).astype(np.float32))
    x = mk((cfg.T, cfg.h), 1.0)
    wr = mk((cfg.E, cfg.h), 0.3)
    W13 = [mk((2 * cfg.I, cfg.h), 0.3) for _ in range(cfg.E)]
    W2 = [mk((cfg.h, cfg.I), 0.3) for _ in range(cfg.E)]
    w13s, w2s = mk((2 * cfg.shared_I, cfg.h), 0.3), mk((cfg.h, cfg.shared_I), 0.3)
    return cfg, x, wr, W13, W2, w13s, w2s


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_is_routed_layer_plus_an_always_chosen_expert(dtype):
    """The shared expert is an expert that every token uses outside the routing:
    the block must equal a routed layer with one more expert, forced into every
    token's choice with weight 1 (computed through the layout, permutation,
    grouped FFN and combine of the routed path)."""
    cfg, x, wr, W13, W2, w13s, w2s = _block_case(dtype)
    blk = oracle.block_forward(x, wr, lambda e: W13[e], lambda e: W2[e], w13s, w2s, cfg)
    aug = cfg.replace(E=cfg.E + 1, K=cfg.K + 1, ep_size=1)
    ids = np.concatenate([blk["ids"], np.full((cfg.T, 1), cfg.E, dtype=np.int32)], axis=1)
    w = np.concatenate([blk["w"], np.ones((cfg.T, 1), dtype=np.float32)], axis=1)
    lay = oracle.dispatch_layout(ids, aug)
    xp = oracle.permute(x, lay["row_src"])
    W13a, W2a = W13 + [w13s], W2 + [w2s]
    parts = oracle.grouped_ffn(xp, lay["offsets"], lay["kept"], lambda e: W13a[e], lambda e: W2a[e], aug)
    yp = np.zeros_like(xp)
    for e, (idx, rows) in parts.items():
        yp[idx] = rows
    y_aug = oracle.combine(yp, lay["slot"], w, aug, rounded=False)
    np.testing.assert_allclose(blk["y_exact"], y_aug, rtol=1e-12, atol=1e-12)


def test_block_without_shared_weights_is_the_layer():
    """Zero shared-expert weights leave exactly the routed layer; doubling the
    down weight (an exact scaling in bf16) doubles the shared expert's output."""
    cfg, x, wr, W13, W2, w13s, w2s = _block_case("bf16", seed=5)
    lay = oracle.layer_forward(x, wr, lambda e: W13[e], lambda e: W2[e], cfg)
    zero = np.zeros_like(w13s)
    blk = oracle.block_forward(x, wr, lambda e: W13[e], lambda e: W2[e], zero, np.zeros_like(w2s), cfg)
    assert np.array_equal(blk["y"], lay["y"])
    ys1 = oracle.to_f64(oracle.shared_ffn(x, w13s, w2s, cfg), "bf16")
    w2x2 = synth.f32_to_bf16_bits((oracle.to_f64(w2s, "bf16") * 2).astype(np.float32))
    ys2 = oracle.to_f64(oracle.shared_ffn(x, w13s, w2x2, cfg), "bf16")
    assert np.array_equal(ys2, 2 * ys1)


def test_shared_ffn_library_other_width():
    """A shared expert narrower than the routed ones (shared_I != I) against
    torch's linear and silu in float64, intermediate rounded to bf16."""
    cfg, x, wr, W13, W2, _, _ = _block_case("bf16", seed=6)
    cfg = cfg.replace(shared_I=8)
    rng = np.random.default_rng(7)
    w13s = synth.f32_to_bf16_bits((rng.normal(size=(16, cfg.h)) * 0.3).astype(np.float32))
    w2s = synth.f32_to_bf16_bits((rng.normal(size=(cfg.h, 8)) * 0.3).astype(np.float32))
    F = torch.nn.functional
    X = torch.from_numpy(oracle.to_f64(x, "bf16"))
    A = torch.from_numpy(oracle.to_f64(w13s, "bf16"))
    a = F.silu(F.linear(X, A[:8])) * F.linear(X, A[8:])
    a = torch.from_numpy(oracle.to_f64(oracle.round_to_bf16_bits(a.numpy()), "bf16"))
    ref = F.linear(a, torch.from_numpy(oracle.to_f64(w2s, "bf16"))).numpy()
    got = oracle.shared_ffn(x, w13s, w2s, cfg, rounded=False)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- EPLB
def test_eplb_hand_worked(golden_dir):
    g = {}
    for line in open(os.path.join(golden_dir, "eplb_case.txt")):
        line = line.split("#")[0].split()
        if line:
            g[line[0]] = [int(v) for v in line[1:]]
    p = oracle.eplb_plan(g["counts"], g["n_ep"][0], g["n_redundant"][0])
    for k in ("n_rep", "rep_offsets", "rep_phys", "phys_to_log", "rank_load"):
        assert p[k].tolist() == g[k], k


@pytest.mark.parametrize("seed", range(6))
def test_eplb_replication_minimises_the_largest_replica_load(seed):
    """Brute force over every way to hand out R redundant replicas: the plan's
    largest load per replica (count / replicas) is the smallest possible."""
    from fractions import Fraction
    rng = np.random.default_rng(seed)
    E, R = int(rng.integers(2, 5)), int(rng.integers(1, 5))
    counts = rng.integers(0, 40, size=E).tolist()
    p = oracle.eplb_plan(counts, 1, R)
    worst = max(Fraction(c, n) for c, n in zip(counts, p["n_rep"].tolist()))
    best = min(max(Fraction(c, n) for c, n in zip(counts, reps))
               for reps in itertools.product(range(1, R + 2), repeat=E) if sum(reps) == E + R)
    assert worst == best
    assert p["n_rep"].sum() == E + R and p["n_rep"].min() >= 1


@pytest.mark.parametrize("seed", range(6))
def test_eplb_placement(seed):
    """Every replica on exactly one slot, every rank full, loads adding up; the
    most loaded rank within one replica's load of the best possible placement
    (brute force over all placements with equal slot counts)."""
    rng = np.random.default_rng(100 + seed)
    n_ep = int(rng.integers(2, 4))
    E = n_ep * int(rng.integers(1, 3))
    R = n_ep * int(rng.integers(0, 2))
    counts = rng.integers(0, 30, size=E).tolist()
    p = oracle.eplb_plan(counts, n_ep, R)
    P, slots = E + R, (E + R) // n_ep
    assert sorted(p["rep_phys"].tolist()) == list(range(P))
    assert p["rank_load"].sum() == sum(counts)
    loads = []
    for e in range(E):
        n = int(p["n_rep"][e])
        q, m = divmod(counts[e], n)
        loads += [q + (1 if r < m else 0) for r in range(n)]
    best = min(max(sum(loads[i] for i in range(P) if assign[i] == j) for j in range(n_ep))
               for assign in itertools.product(range(n_ep), repeat=P)
               if all(assign.count(j) == slots for j in range(n_ep)))
    assert p["rank_load"].max() <= best + max(loads)


def test_eplb_map_round_robin_and_layer_unchanged():
    """Tokens of a logical expert go to its replicas by t mod n_rep; relabelling
    experts into replicas leaves a dropless layer's output bit for bit as it
    was, while the per-rank load becomes more even."""
    cfg = _cfg(T=48, h=16, E=8, K=1, I=8, dtype="f32", score="softmax", ep_size=4, n_redundant=4)
    rng = np.random.default_rng(9)
    x = rng.normal(size=(cfg.T, cfg.h)).astype(np.float32)
    wr = rng.normal(size=(cfg.E, cfg.h)).astype(np.float32) * 0.2
    off = np.zeros(cfg.E, dtype=np.float32)
    off[0] = 2.0                                     # expert 0 takes most tokens
    W13 = [rng.normal(size=(2 * cfg.I, cfg.h)).astype(np.float32) for _ in range(cfg.E)]
    W2 = [rng.normal(size=(cfg.h, cfg.I)).astype(np.float32) for _ in range(cfg.E)]
    base = oracle.layer_forward(x, wr, lambda e: W13[e], lambda e: W2[e], cfg.replace(n_redundant=0),
                                logit_offset=off)
    plan = oracle.eplb_plan(base["layout"]["counts"], cfg.ep_size, cfg.n_redundant)
    r = oracle.layer_forward_eplb(x, wr, lambda e: W13[e], lambda e: W2[e], cfg, plan, logit_offset=off)
    assert base["layout"]["counts"][0] > cfg.T // 2
    assert np.array_equal(r["ids"], base["ids"])
    for t in range(cfg.T):
        for k in range(cfg.K):
            e = base["ids"][t, k]
            reps = plan["rep_phys"][plan["rep_offsets"][e]:plan["rep_offsets"][e + 1]]
            assert r["phys_ids"][t, k] == reps[t % len(reps)]
    assert np.array_equal(r["y"], base["y"])
    assert r["layout"]["balancedness"] > base["layout"]["balancedness"] + 0.2


# --------------------------------------------------------------------------- FP8 experts
def test_e4m3_rounding_matches_torch():
    """Round-to-nearest-even E4M3 with saturation against torch's float8_e4m3fn
    cast: random values over the whole range, subnormals, every tie between two
    neighbouring codes, signed zeros, the largest finite value."""
    rng = np.random.default_rng(0)
    mags = oracle.moe_oracle._E4M3
    mid = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.normal(size=20000) * 10, rng.normal(size=5000) * 1e-3, rng.uniform(-448, 448, 5000),
                        mid, -mid, [0.0, -0.0, 448.0, -448.0, 1e-12, -1e-12]]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.round_to_e4m3(v), ref)
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    assert np.array_equal(oracle.e4m3_decode(codes),
                          torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy())


def test_quantize_rows_definition():
    """The largest magnitude of a row maps to 448 times its scale; an all-zero
    row has scale 1 and zero codes; every value comes back within half a step
    of E4M3 (1/16 relative in the normal range, half the smallest subnormal
    step below it)."""
    rng = np.random.default_rng(1)
    v = (rng.normal(size=(50, 300)) * np.exp(rng.normal(size=(50, 1)) * 3)).astype(np.float32)
    v[7] = 0
    q, s = oracle.quantize_rows_e4m3(v)
    assert s[7] == 1.0 and not q[7].any()
    dec = oracle.e4m3_decode(q)
    for r in range(50):
        if r == 7:
            continue
        j = np.argmax(np.abs(v[r]))
        assert abs(dec[r, j]) == 448.0
        assert s[r] == np.float32(np.abs(v[r]).max() / np.float32(448))
        err = np.abs(dec[r] * float(s[r]) - v[r].astype(np.float64))
        bound = np.maximum(np.abs(v[r]) / 16 * (1 + 1e-6), float(s[r]) * 2.0 ** -10)
        assert np.all(err <= bound)


def test_fp8_expert_ffn_against_torch_float8():
    """One FP8 expert against a path built from torch: float8_e4m3fn casts of
    the scaled rows, float64 F.linear and F.silu, the intermediate rounded to
    bf16 and re-quantised by the same torch casts."""
    rng = np.random.default_rng(2)
    h, I, n = 64, 32, 9
    F = torch.nn.functional

    def tq(a):  # torch-side row quantisation: float32 scale, float8 cast
        a32 = torch.from_numpy(np.asarray(a, dtype=np.float32))
        s = a32.abs().amax(dim=1) / 448.0
        s = torch.where(s > 0, s, torch.ones_like(s))
        return (a32 / s[:, None]).to(torch.float8_e4m3fn), s

    bf = lambda a: oracle.to_f64(synth.f32_to_bf16_bits(np.asarray(a, np.float32)), "bf16")  # noqa: E731
    x, w13, w2 = bf(rng.normal(size=(n, h))), bf(rng.normal(size=(2 * I, h)) / 8), bf(rng.normal(size=(h, I)) / 6)
    (xt, sxt), (wt, swt), (w2t, sw2t) = tq(x), tq(w13), tq(w2)
    g = F.linear(xt.double(), wt.double()[:I]) * sxt.double()[:, None] * swt.double()[None, :I]
    u = F.linear(xt.double(), wt.double()[I:]) * sxt.double()[:, None] * swt.double()[None, I:]
    a = bf((F.silu(g) * u).numpy())
    at, sat = tq(a)
    ref = (F.linear(at.double(), w2t.double()) * sat.double()[:, None] * sw2t.double()[None, :]).numpy()
    u8 = lambda t: t.view(torch.uint8).numpy()  # noqa: E731
    got = oracle.expert_ffn_fp8(u8(xt), sxt.numpy(), u8(wt), swt.numpy(), u8(w2t), sw2t.numpy(), I, rounded=False)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    xq, sx = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(xq, u8(xt)) and np.array_equal(sx, sxt.numpy())


def test_fp8_layer_routes_like_the_bf16_layer():
    """FP8 experts leave routing and layout untouched, and the output stays
    close to the bf16 layer's (E4M3 carries 3 mantissa bits)."""
    cfg, x, wr, W13, W2, _, _ = _block_case("bf16", seed=8)
    cfg = cfg.replace(shared_I=0)
    Q13 = [oracle.quantize_rows_e4m3(oracle.to_f64(w, "bf16")) for w in W13]
    Q2 = [oracle.quantize_rows_e4m3(oracle.to_f64(w, "bf16")) for w in W2]
    a = oracle.layer_forward(x, wr, lambda e: W13[e], lambda e: W2[e], cfg)
    b = oracle.layer_forward_fp8(x, wr, lambda e: Q13[e], lambda e: Q2[e], cfg)
    assert np.array_equal(a["ids"], b["ids"]) and np.array_equal(a["layout"]["slot"], b["layout"]["slot"])
    ya, yb = oracle.to_f64(a["y"], "bf16"), oracle.to_f64(b["y"], "bf16")
    # E4M3 steps are at most 1/16 relative: a few quantised stages stay within
    # a few percent of the output's RMS
    assert np.sqrt(np.mean((ya - yb) ** 2)) <= 0.1 * np.sqrt(np.mean(ya ** 2))
