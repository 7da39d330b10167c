"""CPU oracle for the forward pass of a Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library never
calls it and shares no code with it.

Plain and slow on purpose: float64 arithmetic, a library matrix product or sort
where one is a step of the definition, plain loops elsewhere, and no blocking,
fusion or reordering beyond what the definition states.

Pages followed (cited by title and section):
  [overview]  "专家并行 / 总览" (t6page.pages.dev): the glossary table
              (tbl-ep-overview-glossary), "MoE 路由机制是什么", "Dispatch 通信矩阵"
              (eq. par-ep-dispatch-matrix), "通信量公式" (eqs. par-ep-comm-total,
              par-ep-comm-per-chip, par-ep-comm-pair, table tbl-ep-02), "如何在不跑
              模型时估算 EP 负载" (eq. par-ep-active-experts).
  [notes]     "专家并行与 MoE" (note.yj-dis.top): "MoE 结构回顾" (router, capacity
              factor, token drop), "负载均衡" (aux-loss-free bias, drop/pad).
  [compass]   "專家並行（Expert Parallelism, EP）" (compassingai.com): "技術原理"
              (the four steps route / dispatch / expert compute / weighted combine),
              "關鍵引數與考量" (capacity factor).
  [serving]   "MoE 服務的專家並行性" (aiunderstanding.org): "技術洞察" (capacity,
              drop or pad so that expert GEMMs have uniform shapes).

Readings of points the pages leave open are marked READING below.

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
what the pages or mathematics fix (tests/test_oracle_pins.py): printed volumes,
closed forms of uniform routing, hand-worked cases, brute-force enumeration and
library routines.  No function is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

# ----------------------------------------------------------------- precision helpers


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64, exactly."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 (nearest-even) -> bfloat16 (nearest-even) bit patterns."""
    f = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored tensor (float32 values or bf16 bits) to float64."""
    return bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a, dtype=np.float64)


def store(v: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float64 result to the storage type (float32 values or bf16 bits)."""
    return round_to_bf16_bits(v) if dtype == "bf16" else np.asarray(v, dtype=np.float64).astype(np.float32)


# ----------------------------------------------------------------- step 1: router logits


def router_logits(x: np.ndarray, w_r: np.ndarray, dtype: str,
                  logit_offset: Optional[np.ndarray] = None) -> np.ndarray:
    """L[t, e] = sum_j x[t, j] * W_r[e, j] (+ o[e]), float64 sums stored as float32.

    The router is the light network that scores every expert for every token
    ([overview] glossary "Router"; [notes] "MoE 结构回顾" Router/Gating Network).
    ``w_r`` is [E, h].  ``logit_offset`` is an optional per-expert additive
    term of the logits (used to impose a skewed expert popularity).
    """
    L = to_f64(x, dtype) @ to_f64(w_r, dtype).T
    if logit_offset is not None:
        L = L + np.asarray(logit_offset, dtype=np.float64)[None, :]
    return L.astype(np.float32)


# ----------------------------------------------------------------- step 2: routing


def scores_f64(L: np.ndarray, score: str) -> np.ndarray:
    """Router scores in float64: softmax over experts, or the elementwise sigmoid.

    READING: the pages speak of per-expert "weights/probabilities" ([compass]
    "技術原理" step 1) without naming the function; the layer's configuration
    names softmax or sigmoid.
    """
    L = np.asarray(L, dtype=np.float64)
    if score == "softmax":
        z = np.exp(L - L.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if score == "sigmoid":
        return 1.0 / (1.0 + np.exp(-L))
    raise ValueError(score)


def selection_keys(L: np.ndarray, cfg, bias: Optional[np.ndarray]) -> np.ndarray:
    """float32 keys on which experts are ranked.

    Aux-loss-free balancing adds a per-expert bias to the score used for
    selection only ([notes] "负载均衡", aux-loss-free row: the bias of each
    expert is adjusted instead of adding a loss term).

    READING (pages silent; needed so that two implementations agree bit for
    bit): the key is ``fl32(s + b)``, the float64 score plus the bias rounded
    once to float32.  For softmax with neither bias nor group limit the key is
    the logit itself: softmax is strictly increasing in the logit, so ranking
    logits ranks the exact probabilities and no exponential is rounded.
    """
    if cfg.score == "softmax" and bias is None and cfg.n_groups <= 0:
        return np.asarray(L, dtype=np.float32).copy()
    s = scores_f64(L, cfg.score)
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return s.astype(np.float32)


def _rank_order(keys_row: np.ndarray, allowed: np.ndarray) -> list:
    """Allowed expert ids ordered by key descending, ties to the lower id."""
    ids = [e for e in range(len(keys_row)) if allowed[e]]
    return sorted(ids, key=lambda e: (-float(keys_row[e]), e))


def allowed_experts(keys: np.ndarray, cfg) -> np.ndarray:
    """Group-limited routing mask [T, E] (all True without a group limit).

    DeepSeek-V3's group-limited routing lets a token use experts of its top-M
    groups only ([overview] glossary "Expert group"; node-limited routing with
    M=4 in "EP AllToAll 为什么不同于普通 AllToAll?").  Experts are split into
    ``n_groups`` contiguous groups of E/n_groups; a group's score is the sum
    of its ``group_topn`` largest keys, added in descending key order in
    float32; the ``topk_groups`` best groups are kept (ties to the lower group id).
    """
    T, E = keys.shape
    if cfg.n_groups <= 0:
        return np.ones((T, E), dtype=bool)
    G, gs = cfg.n_groups, E // cfg.n_groups
    mask = np.zeros((T, E), dtype=bool)
    for t in range(T):
        gscore = []
        for g in range(G):
            members = keys[t, g * gs:(g + 1) * gs]
            top = sorted(members.tolist(), reverse=True)[:cfg.group_topn]
            acc = np.float32(0.0)
            for v in top:
                acc = np.float32(acc + np.float32(v))
            gscore.append(acc)
        chosen = sorted(range(G), key=lambda g: (-float(gscore[g]), g))[:cfg.topk_groups]
        for g in chosen:
            mask[t, g * gs:(g + 1) * gs] = True
    return mask


def route(L: np.ndarray, cfg, bias: Optional[np.ndarray] = None):
    """Top-K expert ids and combine weights for every token.

    Each token keeps its K best experts ([overview] glossary "top-K", "MoE 路由
    机制是什么"; [notes] "MoE 结构回顾").  Ids are listed by key descending, ties
    to the lower expert id (READING: the tiny layer's configuration states this
    tie rule; it is used everywhere).

    Weights: the chosen experts' scores, taken WITHOUT the selection bias
    ([notes] "负载均衡": the bias only steers selection); with
    ``renormalize`` they are divided by their sum; then multiplied by
    ``scale``.  Computed in float64 and stored as float32.

    Returns (ids int32 [T,K], w float32 [T,K], keys float32 [T,E], allowed bool [T,E]).
    """
    L = np.asarray(L, dtype=np.float32)
    T, E = L.shape
    K = cfg.K
    keys = selection_keys(L, cfg, bias)
    allowed = allowed_experts(keys, cfg)
    ids = np.zeros((T, K), dtype=np.int32)
    for t in range(T):
        order = _rank_order(keys[t], allowed[t])
        ids[t] = order[:K]
    s = scores_f64(L, cfg.score)
    chosen = np.take_along_axis(s, ids.astype(np.int64), axis=1)
    if cfg.renormalize:
        chosen = chosen / chosen.sum(axis=1, keepdims=True)
    w = (chosen * float(cfg.scale)).astype(np.float32)
    return ids, w, keys, allowed


# Near-ties.  Two implementations whose logits differ in the last bits (float32
# against float64 sums) may route a token differently only where the decision
# rests on keys that nearly tie.  The margins below measure, per token, how far
# the decision is from a tie: the relative gap between the two scores the
# decision compares.  READING (the parity rule for routing; [overview]
# glossary "top-K"): a top-K difference is excused only where such a gap is
# < 1e-4.


def group_margin(keys: np.ndarray, cfg) -> np.ndarray:
    """Relative gap between the last kept and the first dropped group score of every
    token: (g_M - g_{M+1}) / |g_M| with the group scores sorted descending and M
    = topk_groups (inf without a group limit or when every group is kept).  A
    group's score is the sum of its ``group_topn`` largest keys, as in
    allowed_experts."""
    T, E = keys.shape
    out = np.full(T, np.inf)
    if cfg.n_groups <= 0 or cfg.topk_groups >= cfg.n_groups:
        return out
    gs = E // cfg.n_groups
    for t in range(T):
        sc = []
        for g in range(cfg.n_groups):
            top = sorted(keys[t, g * gs:(g + 1) * gs].tolist(), reverse=True)[:cfg.group_topn]
            sc.append(sum(top))
        sc.sort(reverse=True)
        a, b = sc[cfg.topk_groups - 1], sc[cfg.topk_groups]
        out[t] = abs(a - b) / max(abs(a), 1e-30)
    return out


def topk_margin(keys: np.ndarray, allowed: np.ndarray, K: int) -> np.ndarray:
    """Relative gap between the K-th and (K+1)-th allowed key of every token,
    (k_K - k_{K+1}) / |k_K| (inf when fewer than K+1 experts are allowed): how
    far the choice of the K-expert SET is from a tie."""
    T, E = keys.shape
    out = np.full(T, np.inf)
    for t in range(T):
        v = sorted(keys[t][allowed[t]].astype(np.float64).tolist(), reverse=True)
        if len(v) > K:
            out[t] = abs(v[K - 1] - v[K]) / max(abs(v[K - 1]), 1e-30)
    return out


def order_margin(keys: np.ndarray, allowed: np.ndarray, K: int) -> np.ndarray:
    """Smallest relative gap (k_i - k_{i+1}) / |k_i| between adjacent keys among a
    token's K+1 largest allowed keys (inf when at most one key is allowed).

    The ids are listed in descending key order, so two chosen experts whose keys
    nearly tie may swap places, just as the K-th and (K+1)-th may swap in and
    out of the set; this margin covers both (it is <= topk_margin)."""
    T, E = keys.shape
    out = np.full(T, np.inf)
    for t in range(T):
        v = sorted(keys[t][allowed[t]].astype(np.float64).tolist(), reverse=True)[:K + 1]
        for a, b in zip(v, v[1:]):
            out[t] = min(out[t], abs(a - b) / max(abs(a), 1e-30))
    return out


def near_tie_margin(keys: np.ndarray, allowed: np.ndarray, cfg) -> np.ndarray:
    """Per token, the smaller of order_margin and group_margin: the relative gap of
    the closest comparison the routing decision (groups, set and order) rests on."""
    return np.minimum(order_margin(keys, allowed, cfg.K), group_margin(keys, cfg))


# ----------------------------------------------------------------- step 3: dispatch layout


def dispatch_layout(ids: np.ndarray, cfg) -> dict:
    """Per-expert histogram, capacity drop/pad, permutation and the dispatch matrix.

    * counts[e]: assignments (t, k) routed to e; their sum is T*K since every
      token goes to K experts ([overview] "通信量公式": total volume B*K*h*dtype).
    * rank of (t, k) inside expert e: the number of earlier tokens routed to e
      (token order; a token never picks one expert twice).
    * capacity ([compass] "關鍵引數與考量"; [notes] "MoE 结构回顾": tokens over
      an expert's cap are dropped; [serving] "技術洞察": drop or pad so expert
      GEMMs are uniform): with capacity > 0 an assignment is kept iff its rank
      < capacity, so overflow is dropped in token order; kept[e] = min(counts,
      capacity).  With pad, expert e owns rows [e*cap, (e+1)*cap) and unused
      rows are pad rows.
    * offsets: exclusive prefix sum of kept (pad: e*cap); offsets[E] = rows used.
    * slot[t, k] = offsets[e] + rank, or -1 if dropped; row_src is its inverse
      (the token of every permuted row, -1 for pad/unused rows).
    * n_ij ([overview] "Dispatch 通信矩阵", eq. par-ep-dispatch-matrix): the
      number of kept assignments that chip i sends to chip j of a virtual EP
      group; C[i][j] = n_ij * h * dtype_size.  Expert e lives on chip
      e // (E / N_EP) ([overview] "Dispatch 通信矩阵": expert_id / 4 = chip_id with
      4 experts per chip; glossary "EP 组": consecutive chip ids).
      READING: chip i holds the contiguous token block t*N_EP // T == i (each
      chip holds B/N_EP tokens in the page's worked example).
    * Balancedness ([overview] glossary: mean over GPUs of MoE time / max).
      READING: the per-chip time is represented by the rows it receives,
      recv_j = sum_i n_ij; balancedness = sum_j recv_j / (N_EP * max_j recv_j),
      1.0 when nothing is received.  Evaluated in float64, stored float32.
    """
    ids = np.asarray(ids, dtype=np.int64)
    T, K = ids.shape
    E, cap, N = cfg.E, int(cfg.capacity), int(cfg.ep_size)
    pad = bool(cfg.pad) and cap > 0
    flat = ids.reshape(-1)

    counts = np.zeros(E, dtype=np.int64)
    rank = np.zeros(T * K, dtype=np.int64)
    for a in range(T * K):            # token order: a = t*K + k
        e = flat[a]
        rank[a] = counts[e]
        counts[e] += 1

    keep = (rank < cap) if cap > 0 else np.ones(T * K, dtype=bool)
    kept = np.minimum(counts, cap) if cap > 0 else counts.copy()
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + (cap if pad else kept[e])
    slot = np.where(keep, offsets[flat] + rank, -1)
    R = E * cap if pad else T * K
    row_src = np.full(R, -1, dtype=np.int64)
    for a in range(T * K):
        if keep[a]:
            row_src[slot[a]] = a // K

    epr = E // N
    n_ij = np.zeros((N, N), dtype=np.int64)
    for a in range(T * K):
        if keep[a]:
            t = a // K
            n_ij[(t * N) // T, flat[a] // epr] += 1
    ds = 4 if cfg.dtype == "f32" else 2
    sent = n_ij.sum(axis=1)
    recv = n_ij.sum(axis=0)
    mx = int(recv.max()) if N > 0 else 0
    bal = np.float32(1.0) if mx == 0 else np.float32(float(recv.sum()) / float(N * mx))
    kept_total = int(keep.sum())
    return {
        "counts": counts.astype(np.int32),
        "kept": kept.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "slot": slot.reshape(T, K).astype(np.int32),
        "row_src": row_src.astype(np.int32),
        "n_ij": n_ij,
        "sent_bytes": sent * cfg.h * ds,
        "recv_bytes": recv * cfg.h * ds,
        "kept_total": kept_total,
        "dropped": T * K - kept_total,
        "offdiag_rows": int(n_ij.sum() - np.trace(n_ij)),
        "experts_touched": int((kept > 0).sum()),
        "balancedness": bal,
        "rows": R,
    }


# ----------------------------------------------------------------- step 4: permute


def permute(x: np.ndarray, row_src: np.ndarray) -> np.ndarray:
    """The on-device stand-in for the dispatch All-to-All ([overview] glossary
    "Dispatch"; [compass] "技術原理" step 2): permuted row r is a copy of token
    row_src[r]'s hidden vector; pad/unused rows are zero.  Exact copy."""
    R = len(row_src)
    out = np.zeros((R,) + x.shape[1:], dtype=x.dtype)
    for r in range(R):
        if row_src[r] >= 0:
            out[r] = x[row_src[r]]
    return out


# ----------------------------------------------------------------- step 5: expert FFN


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def expert_ffn(xrows: np.ndarray, w13: np.ndarray, w2: np.ndarray, dtype: str, I: int,
               rounded: bool = True) -> np.ndarray:
    """One expert's SwiGLU FFN on a block of rows ([compass] "技術原理" step 3:
    every expert is an independent FFN; SwiGLU per the layer's configuration).

    g = X Wg^T, u = X Wu^T (Wg = w13[:I], Wu = w13[I:]); a = silu(g) * u,
    stored in the data type (READING: the intermediate activation is a stored
    tensor of the layer's data type); y = a Wd^T with Wd = w2 [h, I], stored in
    the data type.  float64 sums.  With ``rounded=False`` the output is returned
    in float64 before its final rounding (the intermediate is still rounded).
    """
    X = to_f64(xrows, dtype)
    W = to_f64(w13, dtype)
    g = X @ W[:I].T
    u = X @ W[I:].T
    a = to_f64(store(silu(g) * u, dtype), dtype)
    y = a @ to_f64(w2, dtype).T
    return store(y, dtype) if rounded else y


def grouped_ffn(xp: np.ndarray, offsets: np.ndarray, kept: np.ndarray, get_w13, get_w2,
                cfg, experts=None, rows=None, rounded: bool = True) -> dict:
    """Runs expert_ffn on every expert's rows [offsets[e], offsets[e] + kept[e]).

    ``get_w13(e)`` / ``get_w2(e)`` return an expert's weights (so a caller can
    stream them); ``experts`` restricts the work to a subset and ``rows`` (a
    dict e -> absolute row indices inside e's segment) to some of its rows.
    Returns {e: (row indices, yp rows)}.
    """
    out = {}
    for e in (range(cfg.E) if experts is None else experts):
        n = int(kept[e])
        r0 = int(offsets[e])
        idx = np.arange(r0, r0 + n) if rows is None else np.asarray(rows[e], dtype=np.int64)
        assert np.all((idx >= r0) & (idx < r0 + n))
        if len(idx) == 0:
            out[e] = (idx, np.zeros((0, cfg.h)))
            continue
        out[e] = (idx, expert_ffn(xp[idx], get_w13(e), get_w2(e), cfg.dtype, cfg.I, rounded))
    return out


# ----------------------------------------------------------------- step 6: combine


def combine(yp: np.ndarray, slot: np.ndarray, w: np.ndarray, cfg, tokens=None, rounded: bool = True) -> np.ndarray:
    """Weighted combine back into token order ([compass] "技術原理" step 4: results
    return to the token's device and are summed with the routing weights;
    [overview] glossary "Combine").

    y[t] = sum over k = 0..K-1 with slot[t,k] >= 0 of w[t,k] * yp[slot[t,k]],
    float64, stored in the data type.  Dropped assignments contribute nothing
    and the remaining weights are not renormalised (READING).  ``yp`` may be
    float64 (unrounded rows); ``rounded=False`` returns float64.
    """
    T = slot.shape[0]
    tok = range(T) if tokens is None else tokens
    Y = yp if yp.dtype == np.float64 else to_f64(yp, cfg.dtype)
    out = np.zeros((len(tok), cfg.h), dtype=np.float64)
    for i, t in enumerate(tok):
        for k in range(cfg.K):
            s = int(slot[t, k])
            if s >= 0:
                out[i] += float(w[t, k]) * Y[s]
    return store(out, cfg.dtype) if rounded else out


# ----------------------------------------------------------------- whole layer


def layer_forward(x, w_r, get_w13, get_w2, cfg, sel_bias=None, logit_offset=None) -> dict:
    """route -> layout -> permute -> expert FFN -> combine ([overview] "MoE 路由机制
    是什么": Router -> Dispatch -> Expert Compute -> Combine)."""
    L = router_logits(x, w_r, cfg.dtype, logit_offset)
    ids, w, keys, allowed = route(L, cfg, sel_bias)
    lay = dispatch_layout(ids, cfg)
    xp = permute(x, lay["row_src"])
    parts = grouped_ffn(xp, lay["offsets"], lay["kept"], get_w13, get_w2, cfg, rounded=False)
    yp_exact = np.zeros(xp.shape, dtype=np.float64)
    for e, (idx, rows) in parts.items():
        yp_exact[idx] = rows
    yp = store(yp_exact, cfg.dtype)
    y = combine(yp, lay["slot"], w, cfg)
    y_exact = combine(yp, lay["slot"], w, cfg, rounded=False)
    return {"logits": L, "ids": ids, "w": w, "keys": keys, "allowed": allowed,
            "layout": lay, "xp": xp, "yp": yp, "y": y, "y_exact": y_exact}


# ----------------------------------------------------------------- shared expert, whole block


def shared_ffn(x: np.ndarray, w13s: np.ndarray, w2s: np.ndarray, cfg, rounded: bool = True) -> np.ndarray:
    """The shared expert: an expert that every token passes through, outside the
    routing ([overview] glossary "Expert" and "MoE 路由机制是什么": DeepSeek-V3
    has 256 routed experts plus 1 shared expert per layer).  The same SwiGLU
    FFN as a routed expert (expert_ffn) on all T rows of x, with intermediate
    size ``cfg.shared_I``; output stored in the data type (READING: like a
    routed expert's output rows)."""
    return expert_ffn(x, w13s, w2s, cfg.dtype, cfg.shared_I, rounded)


def combine_add(yp: np.ndarray, slot: np.ndarray, w: np.ndarray, ys: np.ndarray, cfg, tokens=None,
                rounded: bool = True) -> np.ndarray:
    """y[t] = ys[t] + the routed combine of token t (float64, stored in the data
    type): the block's output is the shared expert's plus the routed experts'
    weighted sum."""
    tok = list(range(slot.shape[0])) if tokens is None else list(tokens)
    Ys = ys if ys.dtype == np.float64 else to_f64(ys, cfg.dtype)
    out = combine(yp, slot, w, cfg, tokens=tok, rounded=False) + Ys[tok]
    return store(out, cfg.dtype) if rounded else out


def block_forward(x, w_r, get_w13, get_w2, w13s, w2s, cfg, sel_bias=None, logit_offset=None) -> dict:
    """The DeepSeek-V3 MoE block: the routed layer (layer_forward) plus the shared
    expert, y = shared(x) + sum_k w_k expert_k(x)."""
    r = layer_forward(x, w_r, get_w13, get_w2, cfg, sel_bias, logit_offset)
    ys = shared_ffn(x, w13s, w2s, cfg)
    r["ys"] = ys
    r["y"] = combine_add(r["yp"], r["layout"]["slot"], r["w"], ys, cfg)
    r["y_exact"] = combine_add(r["yp"], r["layout"]["slot"], r["w"], ys, cfg, rounded=False)
    return r


# ----------------------------------------------------------------- EPLB: logical and physical experts


def eplb_plan(counts, n_ep: int, n_redundant: int) -> dict:
    """Replica plan of expert-parallel load balancing ([overview] glossary
    "Logical expert", "Physical expert / Replica", "Redundant expert": a placement
    algorithm copies hot logical experts so that E + R physical experts, a
    multiple of the number of GPUs, flatten the load; e.g. 256 logical + 32
    redundant = 288 physical).

    READINGS (the pages define the terms and the goal, not the algorithm):
    * replication: each of the R redundant replicas goes, one at a time, to the
      logical expert with the largest load per replica counts[e] / n_rep[e]
      (exact integer comparison; ties to the lower id);
    * a logical expert's load is split over its replicas as evenly as possible:
      replica r gets counts // n + (1 if r < counts % n else 0);
    * placement: replicas in order of load descending (ties: lower logical id,
      then lower replica index) each go to the rank with the least load among
      ranks with a free slot (ties to the lower rank); every rank has
      (E + R) / N_EP slots, and physical ids are rank-major in placement order.
    Returns n_rep [E], rep_offsets [E+1], rep_phys [E+R] (physical ids of the
    replicas of e at rep_offsets[e]..), phys_to_log [E+R], rank_load [N_EP]."""
    counts = [int(c) for c in counts]
    E = len(counts)
    P = E + n_redundant
    assert P % n_ep == 0
    n_rep = [1] * E
    for _ in range(n_redundant):
        best = 0
        for e in range(1, E):
            if counts[e] * n_rep[best] > counts[best] * n_rep[e]:
                best = e
        n_rep[best] += 1
    reps = []
    for e in range(E):
        q, m = divmod(counts[e], n_rep[e])
        for r in range(n_rep[e]):
            reps.append((q + (1 if r < m else 0), e, r))
    reps.sort(key=lambda x: (-x[0], x[1], x[2]))
    slots = P // n_ep
    load, fill = [0] * n_ep, [0] * n_ep
    phys = {}
    for ld, e, r in reps:
        j = min((j for j in range(n_ep) if fill[j] < slots), key=lambda j: (load[j], j))
        phys[(e, r)] = j * slots + fill[j]
        fill[j] += 1
        load[j] += ld
    rep_offsets = np.zeros(E + 1, dtype=np.int32)
    rep_offsets[1:] = np.cumsum(n_rep)
    rep_phys = np.zeros(P, dtype=np.int32)
    phys_to_log = np.zeros(P, dtype=np.int32)
    for e in range(E):
        for r in range(n_rep[e]):
            rep_phys[rep_offsets[e] + r] = phys[(e, r)]
            phys_to_log[phys[(e, r)]] = e
    return {"n_rep": np.array(n_rep, dtype=np.int32), "rep_offsets": rep_offsets, "rep_phys": rep_phys,
            "phys_to_log": phys_to_log, "rank_load": np.array(load, dtype=np.int64)}


def eplb_map(ids: np.ndarray, rep_offsets: np.ndarray, rep_phys: np.ndarray) -> np.ndarray:
    """Physical expert of every routed (t, k): replica t mod n_rep(e) of its
    logical expert e (READING: the pages leave the choice among replicas open;
    token order round robin keeps it a function of (t, e) alone)."""
    T, K = ids.shape
    out = np.zeros_like(ids)
    for t in range(T):
        for k in range(K):
            e = int(ids[t, k])
            n = int(rep_offsets[e + 1] - rep_offsets[e])
            out[t, k] = rep_phys[rep_offsets[e] + t % n]
    return out


def layer_forward_eplb(x, w_r, get_w13, get_w2, cfg, plan: dict, sel_bias=None, logit_offset=None) -> dict:
    """The routed layer with replicas: route over the E logical experts, map each
    choice to a physical replica, then layout (capacity, n_ij and Balancedness
    over the E + R physical experts on their ranks), permutation, the FFN of
    each replica with its logical expert's weights, and combine."""
    L = router_logits(x, w_r, cfg.dtype, logit_offset)
    ids, w, keys, allowed = route(L, cfg, sel_bias)
    pids = eplb_map(ids, plan["rep_offsets"], plan["rep_phys"])
    pcfg = cfg.replace(E=cfg.E + cfg.n_redundant, n_groups=0, topk_groups=0, group_topn=0)
    lay = dispatch_layout(pids, pcfg)
    xp = permute(x, lay["row_src"])
    p2l = plan["phys_to_log"]
    parts = grouped_ffn(xp, lay["offsets"], lay["kept"], lambda p: get_w13(int(p2l[p])),
                        lambda p: get_w2(int(p2l[p])), pcfg, rounded=False)
    yp_exact = np.zeros(xp.shape, dtype=np.float64)
    for e, (idx, rows) in parts.items():
        yp_exact[idx] = rows
    yp = store(yp_exact, cfg.dtype)
    return {"logits": L, "ids": ids, "phys_ids": pids, "w": w, "keys": keys, "allowed": allowed, "layout": lay,
            "yp": yp, "y": combine(yp, lay["slot"], w, pcfg), "y_exact": combine(yp, lay["slot"], w, pcfg,
                                                                                   rounded=False)}


# ----------------------------------------------------------------- FP8 experts


def _e4m3_magnitudes() -> np.ndarray:
    """Magnitudes of the non-negative E4M3 codes 0x00..0x7E (OCP FP8 E4M3: 1 sign,
    4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal,
    m/8 * 2^-6; 0x7F is NaN and there is no infinity; largest finite 448).
    Increasing with the code."""
    out = np.zeros(0x7F, dtype=np.float64)
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_E4M3 = _e4m3_magnitudes()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) to float64 values (codes 0x7F/0xFF never occur here)."""
    c = np.asarray(codes, dtype=np.uint8)
    v = _E4M3[np.minimum(c & 0x7F, 0x7E)]
    return np.where(c & 0x80, -v, v)


def round_to_e4m3(v: np.ndarray) -> np.ndarray:
    """float32 values to E4M3 codes: round to nearest, ties to the even code
    (the one whose mantissa ends in 0), magnitudes above 448 saturate to 448;
    the sign is kept (negative values that round to zero give 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), _E4M3[-1])
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _E4M3[lo], _E4M3[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_rows_e4m3(v: np.ndarray):
    """Row-wise FP8 quantisation (READING: the pages name FP8 MoE without a
    format; E4M3 with one float32 scale per row is used).  Per row: amax =
    max |v|, scale = fl32(amax / 448) (1 for an all-zero row), codes =
    round_to_e4m3(fl32(v / scale)); both divisions in float32, correctly
    rounded.  v holds float32-representable values (bf16 or float32 data).
    Returns (codes uint8 [rows, cols], scales float32 [rows])."""
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    amax = np.abs(v32).max(axis=1) if v32.shape[1] else np.zeros(v32.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (v32 / scale[:, None]).astype(np.float32)
    return round_to_e4m3(q), scale


def expert_ffn_fp8(xq, sx, w13q, s13, w2q, s2, I: int, rounded: bool = True) -> np.ndarray:
    """One expert's SwiGLU FFN with FP8 operands: g = (Xq Wq_gate^T) * sx[row] *
    s13[unit] in float64 from the decoded codes (and u likewise); a =
    silu(g) * u stored in bf16 (the intermediate buffer), then quantised per
    row like the inputs; y = (Aq W2q^T) * sa[row] * s2[feature], stored in
    bf16 (READING: FP8 is the storage of weights and expert inputs; the
    intermediate keeps the layer's bf16 and is re-quantised for the down
    projection)."""
    X, W = e4m3_decode(xq), e4m3_decode(w13q)
    sx = np.asarray(sx, dtype=np.float64)[:, None]
    s13 = np.asarray(s13, dtype=np.float64)[None, :]
    g = (X @ W[:I].T) * sx * s13[:, :I]
    u = (X @ W[I:].T) * sx * s13[:, I:]
    a = to_f64(store(silu(g) * u, "bf16"), "bf16")
    aq, sa = quantize_rows_e4m3(a)
    y = (e4m3_decode(aq) @ e4m3_decode(w2q).T) * sa.astype(np.float64)[:, None] * \
        np.asarray(s2, dtype=np.float64)[None, :]
    return store(y, "bf16") if rounded else y


def layer_forward_fp8(x, w_r, get_w13q, get_w2q, cfg, sel_bias=None, logit_offset=None) -> dict:
    """The routed layer with FP8 experts: routing and layout as layer_forward (bf16
    router); x quantised per token (quantize_rows_e4m3) and permuted with its
    scale; each expert's FFN by expert_ffn_fp8 with its quantised weights
    get_w13q(e) = (codes [2I, h], scales [2I]) and get_w2q(e) = (codes [h, I],
    scales [h]); combine as before."""
    L = router_logits(x, w_r, cfg.dtype, logit_offset)
    ids, w, keys, allowed = route(L, cfg, sel_bias)
    lay = dispatch_layout(ids, cfg)
    xq, sx = quantize_rows_e4m3(to_f64(x, cfg.dtype))
    R = lay["rows"]
    yp = np.zeros((R, cfg.h), dtype=np.float64)
    for e in range(cfg.E):
        r0, n = int(lay["offsets"][e]), int(lay["kept"][e])
        if n == 0:
            continue
        src = lay["row_src"][r0:r0 + n]
        (w13q, s13), (w2q, s2) = get_w13q(e), get_w2q(e)
        yp[r0:r0 + n] = expert_ffn_fp8(xq[src], sx[src], w13q, s13, w2q, s2, cfg.I, rounded=False)
    yp = store(yp, "bf16")
    return {"logits": L, "ids": ids, "w": w, "keys": keys, "allowed": allowed, "layout": lay, "xq": xq, "sx": sx,
            "yp": yp, "y": combine(yp, lay["slot"], w, cfg), "y_exact": combine(yp, lay["slot"], w, cfg,
                                                                              rounded=False)}


# ----------------------------------------------------------------- page formulas


def ep_volumes(B: int, K: int, h: int, dtype_size: int, n_ep: int) -> dict:
    """Dispatch volumes of one EP All-to-All ([overview] "通信量公式"):
    M_total = B*K*h*dtype (eq. par-ep-comm-total); M_per_chip = (B*K/N_EP)*h*dtype
    (eq. par-ep-comm-per-chip); m_pair = B*K*h*dtype/N_EP**2 under uniform
    routing (eq. par-ep-comm-pair).  Bytes."""
    total = B * K * h * dtype_size
    return {"total": total, "per_chip": total / n_ep, "pair": total / n_ep ** 2}


def active_experts_per_chip(E: int, P: int, T: int, K: int) -> float:
    """Balls-into-bins estimate of experts hit at least once per chip
    ([overview] "如何在不跑模型时估算 EP 负载", eq. par-ep-active-experts):
    (E/P) * (1 - exp(-T*K/E))."""
    return (E / P) * (1.0 - math.exp(-T * K / E))
