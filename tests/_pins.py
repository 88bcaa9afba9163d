"""Checks that tie the CPU oracle to the pages and to mathematics.

Each ``pin_*`` function runs the oracle (optionally a rebuilt copy, ``lib``)
and returns a list of failure messages (empty = the pin holds).  The regular
tests assert that every pin holds for the committed oracle; the mutation test
plants plausible mistakes in a copy of the oracle source and asserts that some
pin catches each of them.

None of these checks re-types the oracle's formulas: they use closed forms,
exact enumeration of the method's branch probabilities against the
equivalence theorem, library routines (scipy softmax, numpy argmax and
searchsorted), brute force over tree chains, and the worked examples printed
on the pages.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
from scipy.special import softmax as sp_softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _softmax_T(x, T):
    return sp_softmax(np.asarray(x, dtype=np.float64) / np.float64(np.float32(T)))


# --------------------------------------------------------------------------- softmax
def pin_softmax(lib=None) -> list[str]:
    """Closed forms and the scipy special case of softmax(x / T)."""
    errs = []
    # uniform logits -> 1/V
    p = oracle.softmax(np.full(7, 3.25, np.float32), 0.7, lib=lib)
    if np.max(np.abs(p - 1.0 / 7)) > 1e-15:
        errs.append("uniform logits do not give 1/V")
    # two tokens [a, 0] -> logistic(a / T)
    for a, T in [(1.5, 1.0), (-2.0, 0.5), (4.0, 0.8)]:
        p = oracle.softmax(np.array([a, 0.0], np.float32), T, lib=lib)
        want = 1.0 / (1.0 + np.exp(-a / np.float64(np.float32(T))))
        if abs(p[0] - want) > 1e-14 or abs(p.sum() - 1.0) > 1e-15:
            errs.append(f"two-token closed form fails at a={a} T={T}")
    # large logits: the closed form holds far beyond exp's range (the
    # maximum is taken out before exponentiating)
    p = oracle.softmax(np.array([1000.0, 999.0], np.float32), 1.0, lib=lib)
    if not np.all(np.isfinite(p)) or abs(p[0] - 1.0 / (1.0 + np.exp(-1.0))) > 1e-14:
        errs.append("softmax of [1000, 999] is not logistic(1)")
    # bf16 widening: 1.0 (0x3F80) and -2.0 (0xC000) -> logistic(3)
    p = oracle.softmax(np.array([0x3F80, 0xC000], np.uint16), 1.0, dtype="bf16", lib=lib)
    if abs(p[0] - 1.0 / (1.0 + np.exp(-3.0))) > 1e-14:
        errs.append("bf16 widening wrong")
    # library special case: scipy softmax of x / T in float64
    rng = np.random.default_rng(5)
    for T in (1.0, 0.7, 2.5):
        x = (rng.standard_normal(513) * 4).astype(np.float32)
        p = oracle.softmax(x, T, lib=lib)
        if np.max(np.abs(p - _softmax_T(x, T))) > 1e-14 or abs(p.sum() - 1) > 1e-12:
            errs.append(f"disagrees with scipy softmax at T={T}")
    return errs


# --------------------------------------------------------------------------- inverse CDF
def _window_tie(c, target, Z, t, tol=1e-6):
    """Whether u*Z (``target``) lies within tol*Z of C(t) or C(t-1), from
    numpy's cumulative sums ``c``."""
    lo = c[t - 1] if t > 0 else 0.0
    return abs(c[t] - target) <= tol * Z or abs(lo - target) <= tol * Z


def pin_inverse_cdf(lib=None) -> list[str]:
    """numpy searchsorted(side='right') special case; zero weights never drawn;
    the near-tie flag is set exactly when u*Z lies within 1e-6*Z of the drawn
    token's CDF interval ends (checked on random draws and on draws placed
    next to a boundary)."""
    errs = []
    rng = np.random.default_rng(11)
    for trial in range(400):
        V = int(rng.integers(1, 40))
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[int(rng.integers(0, V))] = 0.5
        c = np.cumsum(w)
        Z = c[-1]
        if trial % 2:  # half the draws sit within +-3e-6 of a CDF boundary
            edge = c[int(rng.integers(0, V))] / Z
            u = float(np.clip(edge + rng.uniform(-3e-6, 3e-6), 0.0, np.nextafter(1.0, 0.0)))
        else:
            u = float(rng.random())
        t, tie = oracle.inverse_cdf(w, u, lib=lib)
        want = int(np.searchsorted(c, u * Z, side="right"))
        if want >= V:  # rounding past the end: the last positive weight
            want = int(np.flatnonzero(w > 0)[-1])
        if t != want:
            errs.append(f"searchsorted mismatch V={V} u={u}: {t} vs {want}")
            break
        if w[t] <= 0:
            errs.append("zero-weight token drawn")
            break
        if tie != _window_tie(c, u * Z, Z, t):
            errs.append(f"near-tie flag {tie} wrong for u={u} (V={V})")
            break
    w = np.array([0.0, 0.0, 0.3, 0.0, 0.7, 0.0])
    if oracle.inverse_cdf(w, 0.0, lib=lib)[0] != 2:
        errs.append("u=0 must draw the first positive-weight token")
    if oracle.inverse_cdf(w, np.nextafter(1.0, 0.0), lib=lib)[0] != 4:
        errs.append("u->1 must draw the last positive-weight token")
    if oracle.inverse_cdf(np.zeros(4), 0.3, lib=lib)[0] != -1:
        errs.append("Z == 0 must return -1")
    return errs


def pin_near_ties(lib=None) -> list[str]:
    """The near-tie windows (an accept test with |r - p/q| < 1e-5, a final
    draw whose u*Z lies within 1e-6*Z of a CDF boundary), on closed-form
    cases: a two-token chain whose p/q is a ratio of logistic functions, and
    weights [1/4, 1/4, 1/2] whose first boundary sits at exactly Z/4.  A flag
    must be set inside each window and clear just outside it."""
    errs = []
    # Final draw: boundary C(0) = Z/4 (u*Z at 0.5e-6*Z is inside, 2e-6*Z outside).
    w = np.array([0.25, 0.25, 0.5])
    for d, want_tok, want_tie in [(0.5e-6, 1, True), (-0.5e-6, 0, True),
                                  (2e-6, 1, False), (-2e-6, 0, False)]:
        t, tie = oracle.inverse_cdf(w, 0.25 + d, lib=lib)
        if t != want_tok or tie != want_tie:
            errs.append(f"draw at Z/4 {d:+g}*Z: token {t} flag {tie}, want {want_tok} {want_tie}")
    # Accept test: k = 1, V = 2, T = 1; target row [a, 0], draft row [b, 0]
    # and x_0 = 0, so p/q = logistic(a) / logistic(b).
    a, b = np.float32(0.3), np.float32(0.9)
    ratio = (1.0 / (1.0 + np.exp(-np.float64(a)))) / (1.0 / (1.0 + np.exp(-np.float64(b))))
    target = np.array([[[a, 0.0], [0.5, -0.25]]], np.float32)
    draft = np.array([[[b, 0.0]]], np.float32)
    x = np.zeros((1, 1), np.int32)
    for d, want_n, want_tie in [(5e-6, 0, True), (-5e-6, 1, True),
                                (2e-5, 0, False), (-2e-5, 1, False)]:
        r = np.array([[ratio + d, 0.3]], np.float32)
        res = oracle.verify_chain(target, draft, x, r, 1.0, lib=lib)
        if res["num_accepted"][0] != want_n or bool(res["flags"][0, 0]) != want_tie:
            errs.append(f"accept test at p/q {d:+g}: n={res['num_accepted'][0]} "
                        f"flag={res['flags'][0, 0]}, want {want_n} {want_tie}")
    # The final draw's flag reaches the chain's column k: identical rows
    # accept every draft, and the bonus row [0, 0, ln 4] has its first CDF
    # boundary at 1/(2 + 4) of Z.
    c4 = np.float32(np.log(4.0))
    z4 = 2.0 + np.exp(np.float64(c4))
    target = np.array([[[0.1, -0.2, 0.4], [0.0, 0.0, c4]]], np.float32)
    x = np.zeros((1, 1), np.int32)
    for d, want_tok, want_tie in [(0.5e-6, 1, True), (2e-6, 1, False), (-0.5e-6, 0, True),
                                  (-2e-6, 0, False)]:
        r = np.array([[0.5, 1.0 / z4 + d]], np.float32)
        res = oracle.verify_chain(target, target[:, :1].copy(), x, r, 1.0, lib=lib)
        if res["tokens"][0, 1] != want_tok or bool(res["flags"][0, 1]) != want_tie:
            errs.append(f"bonus draw at C(0) {d:+g}*Z: token {res['tokens'][0, 1]} "
                        f"flag {res['flags'][0, 1]}, want {want_tok} {want_tie}")
    # Random chains whose uniforms sit near p/q and near the final draw's CDF
    # boundaries: every flag equals the window test computed from scipy's
    # softmax and numpy's cumulative sums; positions past the first
    # rejection are never flagged.
    rng = np.random.default_rng(31)
    B, k, V, T = 300, 3, 7, 0.8
    target = (rng.standard_normal((B, k + 1, V)) * 1.5).astype(np.float32)
    draft = (target[:, :k] + rng.standard_normal((B, k, V)) * 0.6).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    r = np.empty((B, k + 1), np.float32)
    plan = []
    for bb in range(B):
        p = [_softmax_T(target[bb, i], T) for i in range(k + 1)]
        q = [_softmax_T(draft[bb, i], T) for i in range(k)]
        ratio = [p[i][x[bb, i]] / q[i][x[bb, i]] for i in range(k)]
        for i in range(k):
            r[bb, i] = np.float32(min(ratio[i] + rng.uniform(-3e-5, 3e-5), 0.999))
        j = next((i for i in range(k) if not (np.float64(r[bb, i]) < ratio[i])), k)
        wts = np.maximum(p[j] - q[j], 0.0) if j < k else p[k]
        c = np.cumsum(wts)
        u = np.float32(np.clip(c[int(rng.integers(0, V))] / c[-1] + rng.uniform(-3e-6, 3e-6), 0.0,
                               np.nextafter(np.float32(1.0), np.float32(0.0))))
        r[bb, k] = u
        plan.append((ratio, j, wts, c))
    res = oracle.verify_chain(target, draft, x, r, T, lib=lib)
    for bb in range(B):
        ratio, j, wts, c = plan[bb]
        if res["num_accepted"][bb] != j:
            errs.append(f"request {bb}: n_acc {res['num_accepted'][bb]} want {j}")
            break
        want = [abs(np.float64(r[bb, i]) - ratio[i]) < 1e-5 if i <= min(j, k - 1) else False
                for i in range(k)]
        t = int(res["tokens"][bb, j])
        want.append(_window_tie(c, np.float64(r[bb, k]) * c[-1], c[-1], t))
        if [bool(f) for f in res["flags"][bb]] != want:
            errs.append(f"request {bb}: flags {res['flags'][bb].tolist()} want {want}")
            break
    return errs


# --------------------------------------------------------------------------- exact distribution
def _topk_softmax_T(x, T, top_k):
    """softmax(x / T) over the top_k logits (numpy's stable argsort of -x:
    larger logit first, lower index first among equals), 0 elsewhere."""
    x = np.asarray(x, dtype=np.float64)
    keep = np.argsort(-x, kind="stable")[:top_k]
    p = np.zeros(x.shape[0])
    p[keep] = _softmax_T(x[keep], T)
    return p


def _filter_np(x, T, top_k=0, top_p=1.0, min_p=0.0):
    """Reading F5/F6 written with numpy's sort and cumulative sums: the top_k
    tokens by (logit descending, index ascending; 0 = all), then the shortest
    prefix whose mass over that set reaches top_p, then the tokens with
    exp(z - z_max) >= min_p; softmax of x / T over what is left."""
    x = np.asarray(x, dtype=np.float64)
    z = x / np.float64(np.float32(T))
    order = np.lexsort((np.arange(x.size), -x))
    keep = order[: x.size if top_k <= 0 else min(top_k, x.size)]
    e = np.exp(z[keep] - z[order[0]])
    if top_p < 1.0:
        m = int(np.searchsorted(np.cumsum(e / e.sum()), top_p, side="left")) + 1
        keep, e = keep[:m], e[:m]
    if min_p > 0.0:
        keep, e = keep[e >= min_p], e[e >= min_p]
    p = np.zeros(x.size)
    p[keep] = e / e.sum()
    return p


def enumerate_chain(target, draft, T, lib=None, top_k=None, filt=None):
    """Drive the oracle through every branch of the chain verify for one small problem.

    For every draft tuple x in [V]^k (weight prod q_i(x_i)), every stopping
    position j, and every final token t with positive weight, build uniforms
    that take that branch: r_i = min(1,a_i)/2 accepts (weight min(1,a_i)),
    r_j = (1+a_j)/2 rejects (weight 1-a_j), and u at the midpoint of t's CDF
    interval (weight w_t/Z).  Returns (weights, expected rows, oracle result).
    With top_k, p and q are the top-k filtered distributions of both sides and
    the oracle's filtered verify runs.
    """
    k1, V = target.shape
    k = k1 - 1
    if filt is not None:
        p = [_filter_np(target[i], T, *filt) for i in range(k + 1)]
        q = [_filter_np(draft[i], T, *filt) for i in range(k)]
    elif top_k is None:
        p = [_softmax_T(target[i], T) for i in range(k + 1)]
        q = [_softmax_T(draft[i], T) for i in range(k)]
    else:
        p = [_topk_softmax_T(target[i], T, top_k) for i in range(k + 1)]
        q = [_topk_softmax_T(draft[i], T, top_k) for i in range(k)]
    reqs_x, reqs_r, weights, expect = [], [], [], []
    for x in itertools.product(range(V), repeat=k):
        wx = np.prod([q[i][x[i]] for i in range(k)])
        if wx == 0:  # a draft the draft side never proposes
            continue
        a = [p[i][x[i]] / q[i][x[i]] for i in range(k)]
        for j in range(k + 1):
            wb = wx
            r = np.full(k + 1, 0.5)
            for i in range(j):
                wb *= min(1.0, a[i])
                r[i] = min(1.0, a[i]) / 2
            if j < k:
                if a[j] >= 1.0:
                    continue
                wb *= 1.0 - a[j]
                r[j] = (1.0 + a[j]) / 2
                wts = np.maximum(p[j] - q[j], 0.0)
            else:
                wts = p[k]
            if wb == 0:  # an accept of weight min(1, 0): a draft outside the target's kept set
                continue
            Z = wts.sum()
            c = np.concatenate([[0.0], np.cumsum(wts)])
            for t in range(V):
                if wts[t] <= 0:
                    continue
                rr = r.copy()
                rr[k] = (c[t] + c[t + 1]) / (2 * Z)
                reqs_x.append(x)
                reqs_r.append(rr)
                weights.append(wb * wts[t] / Z)
                expect.append((j, list(x[:j]) + [t] + [-1] * (k - j)))
    Bn = len(weights)
    tgt = np.broadcast_to(target, (Bn, k + 1, V)).astype(np.float32)
    drf = np.broadcast_to(draft, (Bn, k, V)).astype(np.float32)
    xs = np.array(reqs_x, np.int32).reshape(Bn, k)
    rs = np.array(reqs_r, np.float32)
    if filt is not None:
        res = oracle.verify_chain_filtered(tgt, drf, xs, rs, T, filt[0], filt[1], lib=lib, min_p=filt[2])
    elif top_k is None:
        res = oracle.verify_chain(tgt, drf, xs, rs, T, lib=lib)
    else:
        res = oracle.verify_chain_filtered(tgt, drf, xs, rs, T, top_k, lib=lib)
    return np.array(weights), expect, res, p


def pin_exact_distribution(lib=None) -> list[str]:
    """The equivalence theorem on enumerated branches (vLLM anatomy page,
    "Why this works"; vLLM learning book, section 2 and question 2):
    P(y_i = t | n_acc >= i) = p_i(t) and P(n_acc >= i+1 | n_acc >= i) =
    sum_t min(p_i, q_i), to 1e-12, plus the exact branch outcome per request."""
    errs = []
    rng = np.random.default_rng(2024)
    for (k, V, T) in [(1, 5, 1.0), (2, 4, 0.7), (3, 3, 1.3), (2, 6, 1.0), (3, 5, 0.9)]:
        target = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
        draft = (target[:k] + rng.standard_normal((k, V)) * 0.8).astype(np.float32)
        wts, expect, res, p = enumerate_chain(target, draft, T, lib=lib)
        for e, (j, row) in enumerate(expect):
            if res["num_accepted"][e] != j or list(res["tokens"][e]) != row:
                errs.append(f"k={k} V={V}: branch {e} gave {res['tokens'][e]} want {row}")
                break
        n_acc = res["num_accepted"]
        toks = res["tokens"]
        if abs(wts.sum() - 1.0) > 1e-12:
            errs.append(f"k={k} V={V}: branch weights sum to {wts.sum()}")
        q = [_softmax_T(draft[i], T) for i in range(k)]
        for i in range(k + 1):
            reach = n_acc >= i
            pr = wts[reach].sum()
            dist = np.array([wts[reach & (toks[:, i] == t)].sum() for t in range(V)]) / pr
            if np.max(np.abs(dist - p[i])) > 1e-12:
                errs.append(f"k={k} V={V}: emitted token at {i} is not distributed as p_{i}")
            if i < k:
                beta = np.minimum(p[i], q[i]).sum()
                if abs(wts[n_acc >= i + 1].sum() / pr - beta) > 1e-12:
                    errs.append(f"k={k} V={V}: acceptance at {i} is not sum min(p,q)")
    return errs


# --------------------------------------------------------------------------- invariants
def pin_invariants(lib=None) -> list[str]:
    """q == p accepts all k; r == 0 accepts all k; output-row structure."""
    errs = []
    rng = np.random.default_rng(7)
    B, k, V = 64, 4, 50
    target = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    draft = (target[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    r = rng.random((B, k + 1)).astype(np.float32)
    same = oracle.verify_chain(target, target[:, :k].copy(), x, r, 0.9, lib=lib)
    if not np.all(same["num_accepted"] == k):
        errs.append("identical draft and target must accept every draft")
    zero = r.copy()
    zero[:, :k] = 0.0
    if not np.all(oracle.verify_chain(target, draft, x, zero, 0.9, lib=lib)["num_accepted"] == k):
        errs.append("uniforms of 0 must accept every draft")
    res = oracle.verify_chain(target, draft, x, r, 0.9, lib=lib)
    for b in range(B):
        n = res["num_accepted"][b]
        row = res["tokens"][b]
        if not (0 <= n <= k):
            errs.append("n_acc outside [0, k]")
            break
        if np.count_nonzero(row >= 0) != n + 1 or np.any(row[: n + 1] < 0):
            errs.append("row must hold exactly n_acc+1 tokens then -1")
            break
        if list(row[:n]) != list(x[b, :n]):
            errs.append("the first n_acc tokens must be the drafts")
            break
    bad = x.copy()
    bad[3, 1] = V
    res = oracle.verify_chain(target, draft, bad, r, 0.9, lib=lib)
    if res["rc"] != oracle.EBADINDEX or res["num_accepted"][3] != -1 or np.any(res["tokens"][3] != -1):
        errs.append("an out-of-range draft token must fail that request closed")
    return errs


# --------------------------------------------------------------------------- greedy
def pin_greedy(lib=None) -> list[str]:
    """argmax = numpy argmax (first occurrence); greedy verify emits the argmax chain."""
    errs = []
    rng = np.random.default_rng(3)
    for dtype in ("f32", "bf16"):
        for _ in range(50):
            V = int(rng.integers(2, 300))
            vals = rng.integers(-4, 5, V).astype(np.float32)  # many exact ties
            raw = vals if dtype == "f32" else (vals.view(np.uint32) >> 16).astype(np.uint16)
            if oracle.argmax(raw, dtype, lib=lib) != int(np.argmax(vals)):
                errs.append(f"argmax tie-break differs from numpy ({dtype})")
                break
    B, k, V = 40, 5, 64
    target = rng.integers(-3, 4, (B, k + 1, V)).astype(np.float32)
    g = np.argmax(target, axis=2)
    d = g[:, :k].copy()
    cut = rng.integers(0, k + 1, B)
    for b in range(B):
        if cut[b] < k:
            d[b, cut[b]] = (g[b, cut[b]] + 1) % V
    res = oracle.verify_greedy(target, d, lib=lib)
    for b in range(B):
        want = list(g[b, : cut[b] + 1]) + [-1] * (k - cut[b])
        if res["num_accepted"][b] != cut[b] or list(res["tokens"][b]) != want:
            errs.append("greedy verify does not emit the target's argmax chain")
            break
    return errs


# --------------------------------------------------------------------------- tree
def _random_tree(rng, N, V, accept_bias):
    parent = np.full(N, -1)
    for n in range(1, N):
        parent[n] = int(rng.integers(0, n))
    target = rng.integers(-3, 4, (N, V)).astype(np.float32)
    g = np.argmax(target, axis=1)
    tokens = np.zeros(N, np.int32)
    tokens[0] = int(rng.integers(0, V))
    for n in range(1, N):
        sib_used = {int(tokens[m]) for m in range(1, n) if parent[m] == parent[n]}
        want = int(g[parent[n]])
        if rng.random() < accept_bias and want not in sib_used:
            tokens[n] = want
        else:
            choices = [t for t in range(V) if t not in sib_used]
            tokens[n] = choices[int(rng.integers(0, len(choices)))]
    return parent, target, tokens


def _paths_from_parents(parent, L, P):
    N = len(parent)
    kids = {n: [] for n in range(N)}
    for n in range(1, N):
        kids[int(parent[n])].append(n)
    paths = np.full((P, L), -1, np.int32)
    leaves = [n for n in range(N) if not kids[n]]
    for i, leaf in enumerate(leaves):
        chain = [leaf]
        while chain[-1] != 0:
            chain.append(int(parent[chain[-1]]))
        chain = chain[::-1][:L]
        paths[i, : len(chain)] = chain
    return paths


def _depth(parent, n):
    d = 0
    while n != 0:
        n = int(parent[n])
        d += 1
    return d


def pin_tree(lib=None) -> list[str]:
    """Brute force over root-to-node chains; a one-chain tree equals chain greedy."""
    errs = []
    rng = np.random.default_rng(17)
    for trial in range(60):
        N = int(rng.integers(2, 14))
        V = int(rng.integers(N + 2, N + 12))
        parent, target, tokens = _random_tree(rng, N, V, accept_bias=0.6)
        depth = max(_depth(parent, n) for n in range(N))
        L = depth + 1
        paths = _paths_from_parents(parent, L, N)
        g = np.argmax(target, axis=1)
        # brute force: a node is reachable when every edge on its root chain is accepted
        ok = [True] + [False] * (N - 1)
        for n in range(1, N):  # parents have lower ids
            ok[n] = ok[int(parent[n])] and tokens[n] == g[int(parent[n])]
        best_depth = max(_depth(parent, n) for n in range(N) if ok[n])
        res = oracle.verify_tree(target[None], tokens[None], paths[None], lib=lib)
        n_acc = int(res["num_accepted"][0])
        if n_acc != best_depth:
            errs.append(f"tree n_acc {n_acc} != brute-force depth {best_depth}")
            break
        nodes = [int(v) for v in res["accepted_nodes"][0] if v >= 0]
        if nodes[0] != 0 or len(nodes) != n_acc + 1 or any(
                parent[nodes[i + 1]] != nodes[i] or not ok[nodes[i + 1]] for i in range(n_acc)):
            errs.append("accepted nodes are not an accepted root chain")
            break
        row = res["tokens"][0]
        want = [int(tokens[n]) for n in nodes[1:]] + [int(g[nodes[-1]])]
        if list(row[: n_acc + 1]) != want or np.any(row[n_acc + 1:] != -1):
            errs.append("tree output row wrong")
            break
        # the kept path: the most accepted steps, ties to the lowest path
        # index (numpy's first-occurrence argmax over the paths' step counts)
        steps = []
        for pth in paths:
            a = 0
            while a + 1 < L and pth[a + 1] >= 0 and ok[int(pth[a + 1])]:
                a += 1
            steps.append(a if pth[0] >= 0 else -1)
        if int(res["best_path"][0]) != int(np.argmax(steps)):
            errs.append(f"tree kept path {res['best_path'][0]}, want {int(np.argmax(steps))} (lowest index of the longest)")
            break
    # one-chain tree == chain greedy
    B, k, V = 16, 4, 20
    target = rng.integers(-3, 4, (B, k + 1, V)).astype(np.float32)
    g = np.argmax(target, axis=2)
    d = np.where(rng.random((B, k)) < 0.7, g[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    tree_tokens = np.concatenate([np.zeros((B, 1), np.int32), d], axis=1)
    paths = np.tile(np.arange(k + 1, dtype=np.int32), (B, 1, 1))
    t = oracle.verify_tree(target, tree_tokens, paths, lib=lib)
    c = oracle.verify_greedy(target, d, lib=lib)
    if not (np.array_equal(t["tokens"], c["tokens"]) and np.array_equal(t["num_accepted"], c["num_accepted"])):
        errs.append("one-chain tree differs from chain greedy")
    return errs


# --------------------------------------------------------------------------- rollback
def pin_rollback(lib=None) -> list[str]:
    """Closed form and the boundaries of the TensorRT-LLM walkthrough (update_requests:
    all accepted -> rewind 0; all rejected -> rewind = whole window)."""
    errs = []
    rng = np.random.default_rng(1)
    k = 7
    old = rng.integers(0, 100000, 500).astype(np.int32)
    n = rng.integers(0, k + 1, 500).astype(np.int32)
    res = oracle.rollback(old, n, k, lib=lib)
    for b in range(500):
        if res["new_lens"][b] != old[b] + n[b] + 1 or res["rewind_lens"][b] != k - n[b]:
            errs.append("rollback closed form fails")
            break
    edge = oracle.rollback(np.array([10, 10], np.int32), np.array([k, 0], np.int32), k, lib=lib)
    if list(edge["rewind_lens"]) != [0, k] or list(edge["new_lens"]) != [10 + k + 1, 11]:
        errs.append("rewind boundaries wrong")
    # a count outside [0, k] (a failed request's -1, or a corrupt k + 1)
    # keeps the length and reads rewind -1
    bad = oracle.rollback(np.array([10, 20, 30], np.int32), np.array([-1, k + 1, 2], np.int32), k,
                          lib=lib)
    if bad["rc"] != oracle.EBADINDEX or list(bad["new_lens"]) != [10, 20, 33] or \
            list(bad["rewind_lens"]) != [-1, -1, k - 2]:
        errs.append(f"bad rollback entries: {bad['new_lens']} / {bad['rewind_lens']}")
    return errs


# --------------------------------------------------------------------------- worked example
def pin_worked_example(lib=None) -> list[str]:
    """The FGH example of the TensorRT-LLM walkthrough (MTP section, generation
    phase 1): drafts F G H, target samples F G X (Y discarded) -> accepted F G X,
    H's KV row invalid (rewind 1), two drafts accepted."""
    errs = []
    with open(os.path.join(GOLDEN, "fgh_worked_example.json")) as f:
        ex = json.load(f)
    tok = ex["tokens"]
    target = np.array(ex["target_logits"], np.float32)[None]
    draft = np.array(ex["draft_logits"], np.float32)[None]
    drafts = np.array([[tok["F"], tok["G"], tok["H"]]], np.int32)
    r = np.array([ex["uniforms"]], np.float32)
    want = [tok[c] if c != "-" else -1 for c in ex["expect"]["tokens"]]
    for name, res in (("stochastic", oracle.verify_chain(target, draft, drafts, r, ex["temperature"], lib=lib)),
                      ("greedy", oracle.verify_greedy(target, drafts, lib=lib))):
        if list(res["tokens"][0]) != want or res["num_accepted"][0] != ex["expect"]["num_accepted"]:
            errs.append(f"{name} verify of the FGH example gave {res['tokens'][0]}")
    rb = oracle.rollback(np.array([ex["old_len"]], np.int32),
                         np.array([ex["expect"]["num_accepted"]], np.int32), 3, lib=lib)
    if rb["rewind_lens"][0] != ex["expect"]["rewind"] or rb["new_lens"][0] != ex["expect"]["new_len"]:
        errs.append("FGH rollback wrong")
    return errs


# --------------------------------------------------------------------------- filtered
def pin_filtered(lib=None) -> list[str]:
    """Symmetric top-k / top-p filtering (TensorRT-LLM walkthrough, rejection-
    sampling section): hand examples with closed-form values, the library
    special cases (top_k >= V is scipy's softmax, top_k = 1 numpy's argmax),
    identical filtered sides accept everything, and the equivalence theorem
    on enumerated branches with both sides top-k filtered."""
    errs = []
    fs = lambda x, T, kk, pp=1.0: oracle.filtered_softmax(np.asarray(x, np.float32), T, kk, pp, lib=lib)[0]
    x = [3.0, 1.0, 2.0, 2.0, 0.0]
    e1 = np.exp(-1.0)
    cases = [  # (T, top_k, top_p, expected p)
        (1.0, 3, 1.0, np.array([1.0, 0.0, e1, e1, 0.0]) / (1.0 + 2.0 * e1)),
        (1.0, 3, 0.5, np.array([1.0, 0.0, 0.0, 0.0, 0.0])),
        # 1 / (1 + 2/e) = 0.576 reaches 0.55 alone (mass over the top 3, not the vocabulary)
        (1.0, 3, 0.55, np.array([1.0, 0.0, 0.0, 0.0, 0.0])),
        # two tokens; the tie at logit 2 keeps the lower index
        (1.0, 3, 0.6, np.array([1.0, 0.0, e1, 0.0, 0.0]) / (1.0 + e1)),
        # temperature before the cut: at T = 2 the top token has 0.452 < 0.5
        (2.0, 3, 0.5, np.array([1.0, 0.0, np.exp(-0.5), 0.0, 0.0]) / (1.0 + np.exp(-0.5))),
        # a cut exactly at top_p keeps the shorter prefix
        (1.0, 2, 0.5, None),
    ]
    for T, kk, pp, want in cases:
        if want is None:
            got = fs([1.0, 1.0, 0.0], T, kk, pp)
            want = np.array([1.0, 0.0, 0.0])
        else:
            got = fs(x, T, kk, pp)
        if np.max(np.abs(got - want)) > 1e-12:
            errs.append(f"filtered softmax T={T} top_k={kk} top_p={pp}: {got} want {want}")
    rng = np.random.default_rng(11)
    row = (rng.standard_normal(40) * 2).astype(np.float32)
    if np.max(np.abs(fs(row, 0.8, 40) - _softmax_T(row, 0.8))) > 1e-12:
        errs.append("top_k = V is not the plain softmax")
    tie = np.array([1.0, 5.0, 5.0, 2.0], np.float32)
    if fs(tie, 1.0, 1).tolist() != [0.0, 1.0, 0.0, 0.0] or int(np.argmax(tie)) != 1:
        errs.append("top_k = 1 is not one-hot at the first argmax")
    # The residual after a rejection uses the filtered draft row: p = 1/3 on
    # tokens 0..2, the draft keeps {0, 3, 4} at 1/3 each (token 1, at 4.9, is
    # fourth), draft token 3 (p = 0) is rejected, max(0, p - q) is 1/3 on
    # tokens 1 and 2, and u = 0.1 draws token 1.  (Against the unfiltered
    # draft softmax the residual would be 0.078, 0.102, 0.333 on tokens 0..2
    # and u = 0.1 would draw token 0.)
    tgt = np.array([[[0, 0, 0, -20, -20, -20], [0, 0, 0, 0, 0, 0]]], np.float32)
    drf = np.array([[[5, 4.9, -20, 5, 5, -20]]], np.float32)
    res = oracle.verify_chain_filtered(tgt, drf, np.array([[3]], np.int32),
                                       np.array([[0.5, 0.1]], np.float32), 1.0, 3, lib=lib)
    if res["num_accepted"][0] != 0 or res["tokens"][0].tolist() != [1, -1]:
        errs.append(f"filtered residual example gave {res['tokens'][0]} want [1, -1]")
    B, k, V = 16, 3, 30
    target = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    xs = rng.integers(0, V, (B, k)).astype(np.int32)
    r = rng.random((B, k + 1)).astype(np.float32)
    same = oracle.verify_chain_filtered(target, target[:, :k].copy(), xs, r, 0.9, 5, 0.8, lib=lib)
    kept = same["probs"][:, :, 1] > 0  # drafts inside the draft's kept set
    if not np.all(same["num_accepted"][kept.all(axis=1)] == k):
        errs.append("identically filtered sides must accept every kept draft")
    for (k2, V2, T2, kk) in [(1, 6, 1.0, 3), (2, 5, 0.8, 2), (2, 4, 1.2, 3)]:
        tg = (rng.standard_normal((k2 + 1, V2)) * 1.5).astype(np.float32)
        dr = (tg[:k2] + rng.standard_normal((k2, V2)) * 0.8).astype(np.float32)
        wts, expect, res, p = enumerate_chain(tg, dr, T2, lib=lib, top_k=kk)
        for e, (j, rowe) in enumerate(expect):
            if res["num_accepted"][e] != j or list(res["tokens"][e]) != rowe:
                errs.append(f"filtered k={k2} V={V2}: branch {e} gave {res['tokens'][e]} want {rowe}")
                break
        n_acc, toks = res["num_accepted"], res["tokens"]
        for i in range(k2 + 1):
            reach = n_acc >= i
            dist = np.array([wts[reach & (toks[:, i] == t)].sum() for t in range(V2)]) / wts[reach].sum()
            if np.max(np.abs(dist - p[i])) > 1e-12:
                errs.append(f"filtered k={k2} V={V2}: token {i} is not distributed as filtered p_{i}")
    return errs


# --------------------------------------------------------------------------- Philox, ragged, paged
def pin_philox(lib=None) -> list[str]:
    """Philox4x32-10 against its published known-answer vectors (Salmon et
    al., SC'11, Random123), and the uniforms' stated counter, word and 24-bit
    mapping on top of it."""
    errs = []
    kat = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    h = lambda xs: [int(x, 16) for x in xs]  # noqa: E731
    for v in kat["vectors"]:
        if oracle.philox4x32_10(h(v["ctr"]), h(v["key"]), lib=lib).tolist() != h(v["out"]):
            errs.append(f"Philox known answer {v['ctr']} / {v['key']}")
    seeds = np.array([0x0123456789ABCDEF, 7], dtype=np.uint64)
    offsets = np.array([0xFEDCBA9876543210, 0], dtype=np.uint64)
    u = oracle.philox_uniforms(seeds, offsets, 9, lib=lib)
    for b in range(2):
        key = [int(seeds[b]) & 0xFFFFFFFF, int(seeds[b]) >> 32]
        for i in range(9):
            ctr = [int(offsets[b]) & 0xFFFFFFFF, int(offsets[b]) >> 32, i // 4, 0]
            word = int(oracle.philox4x32_10(ctr, key, lib=lib)[i % 4])
            if u[b, i] != np.float32((word >> 8) / 2.0**24):
                errs.append(f"uniform {i} of stream {b} is not word {i % 4} of counter block {i // 4}")
                return errs
    return errs


def pin_rollback_paged(lib=None) -> list[str]:
    """Closed forms of the paged rollback (TensorRT-LLM walkthrough,
    update_requests and rewind_cache: rewind k_b - n, keep ceil(len / block)
    blocks, return the whole surplus)."""
    errs = []
    res = oracle.rollback_paged([10, 10, 7, 0], [2, 0, 3, 0], k=4, tokens_per_block=4,
                                draft_lens=[3, 0, 3, 2], blocks_held=[5, 3, 2, 1], lib=lib)
    if res["new_lens"].tolist() != [13, 11, 11, 1] or res["rewind_lens"].tolist() != [1, 0, 0, 2]:
        errs.append(f"paged rollback lengths {res['new_lens']} / {res['rewind_lens']}")
    if res["free_blocks"].tolist() != [1, 0, 0, 0]:  # ceil(13/4)=4 of 5; ceil(11/4)=3 of 3; 3 > 2; 1 of 1
        errs.append(f"paged rollback free blocks {res['free_blocks']}")
    bad = oracle.rollback_paged([5, 5], [3, 1], k=4, tokens_per_block=4, draft_lens=[2, 9],
                                blocks_held=[9, 9], lib=lib)
    if bad["rc"] != oracle.EBADINDEX or bad["new_lens"].tolist() != [5, 5] or \
            bad["free_blocks"].tolist() != [0, 0] or bad["rewind_lens"].tolist() != [-1, -1]:
        errs.append("paged rollback must refuse n > k_b and k_b > k entry by entry")
    return errs


def pin_ragged(lib=None) -> list[str]:
    """Ragged draft lengths: each request equals the plain verify of its
    truncated chain (its own k_b drafts, target rows 0..k_b, uniforms r_0..r_{k_b});
    full lengths equal the plain call; a length outside [0, k] fails closed."""
    errs = []
    rng = np.random.default_rng(4)
    B, k, V, T = 6, 5, 60, 0.9
    target = rng.normal(0, 2, size=(B, k + 1, V)).astype(np.float32)
    draft = (target[:, :k] + rng.normal(0, 0.6, size=(B, k, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    r = rng.random((B, k + 1), dtype=np.float32)
    r[:, :k] *= 0.5  # longer accepted prefixes
    lens = np.array([1, 2, 3, 0, 5, 3], np.int32)
    got = oracle.verify_chain(target, draft, x, r, T, draft_lens=lens, lib=lib)
    for b in range(B):
        kb = int(lens[b])
        if kb == 0:
            p = _softmax_T(target[b, 0], T)
            want_tok = int(np.searchsorted(np.cumsum(p), float(r[b, 0]) * p.sum(), side="right"))
            if got["num_accepted"][b] != 0 or got["tokens"][b, 0] != want_tok:
                errs.append("zero drafts must be one draw from target row 0 at r_0")
            continue
        rr = np.concatenate([r[b, :kb], r[b, kb:kb + 1]])[None]
        want = oracle.verify_chain(target[b:b + 1, :kb + 1], draft[b:b + 1, :kb], x[b:b + 1, :kb], rr, T,
                                   lib=lib)
        if got["num_accepted"][b] != want["num_accepted"][0] or \
                not np.array_equal(got["tokens"][b, :kb + 1], want["tokens"][0]) or \
                np.any(got["tokens"][b, kb + 1:] != -1):
            errs.append(f"request {b} (k_b={kb}) is not its truncated chain")
    full = oracle.verify_chain(target, draft, x, r, T, draft_lens=np.full(B, k, np.int32), lib=lib)
    plain = oracle.verify_chain(target, draft, x, r, T, lib=lib)
    if not np.array_equal(full["tokens"], plain["tokens"]):
        errs.append("full lengths must equal the plain call")
    badl = lens.copy()
    badl[2] = k + 1
    bad = oracle.verify_chain(target, draft, x, r, T, draft_lens=badl, lib=lib)
    if bad["rc"] != oracle.EBADINDEX or bad["num_accepted"][2] != -1 or np.any(bad["tokens"][2] != -1):
        errs.append("a draft length above k must fail that request closed")
    # Greedy: every draft, padding included, is numpy's argmax of its target
    # row, so each request accepts exactly its k_b drafts and emits the argmax
    # of row k_b; nothing past k_b is read.
    g = np.argmax(target, axis=-1)
    glens = np.array([0, 1, 2, 5, 4, 3], np.int32)
    got = oracle.verify_greedy(target, g[:, :k].astype(np.int32), draft_lens=glens, lib=lib)
    for b in range(B):
        kb = int(glens[b])
        want = list(g[b, :kb + 1]) + [-1] * (k - kb)
        if got["num_accepted"][b] != kb or got["tokens"][b].tolist() != want:
            errs.append(f"greedy request {b} (k_b={kb}) read past its length")
            break
    return errs


# --------------------------------------------------------------------------- stochastic tree
def _children(paths, prefix):
    """Distinct next nodes (increasing id) of the used paths that start with ``prefix``."""
    d = len(prefix) - 1
    out = set()
    for row in paths:
        if row[0] != 0 or d + 1 >= len(row):
            continue
        if list(row[: d + 1]) == list(prefix) and row[d + 1] >= 0:
            out.add(int(row[d + 1]))
    return sorted(out)


def enumerate_tree_sampled(target, tokens, paths, T):
    """Every branch of the stochastic tree walk for one small tree: for each
    state (accepted prefix), each candidate accepted after the earlier ones
    were rejected, or the final draw of each token with positive residual
    weight.  Uniforms take each branch (reject: (1 + p')/2, accept: p'/2,
    final draw: the midpoint of the token's CDF interval).  Returns
    (weights, expected (n_acc, tokens), uniforms [n, N], reach) where reach
    lists (branch mask of reaching node n, p_n)."""
    N, V = target.shape
    L = paths.shape[1]
    p_of = [_softmax_T(target[n], T) for n in range(N)]
    branches = []  # (weight, n_acc, tokens, uniforms, visited nodes)

    def walk(prefix, weight, u, emitted):
        node = prefix[-1]
        p = p_of[node].copy()
        removed = 0.0
        for c in _children(paths, prefix):
            pc = p[tokens[c]]
            ratio = pc / (1.0 - removed) if 1.0 - removed > 0 else 0.0
            if ratio > 0:
                u2 = u.copy()
                u2[c] = ratio / 2
                walk(prefix + [c], weight * ratio, u2, emitted + [int(tokens[c])])
            if ratio >= 1.0:
                return
            u[c] = (1.0 + ratio) / 2
            weight *= 1.0 - ratio
            removed += pc
            p[tokens[c]] = 0.0
        Z = p.sum()
        cdf = np.concatenate([[0.0], np.cumsum(p)])
        for t in range(V):
            if p[t] > 0:
                u2 = u.copy()
                u2[0] = (cdf[t] + cdf[t + 1]) / (2 * Z)
                toks = emitted + [t]
                branches.append((weight * p[t] / Z, len(emitted), toks + [-1] * (L - len(toks)),
                                 u2, list(prefix)))

    walk([0], 1.0, np.full(N, 0.5), [])
    return branches, p_of


def _random_small_tree(rng, N, V, L):
    parent = np.zeros(N, int)
    depth = np.zeros(N, int)
    for n in range(1, N):
        cands = [m for m in range(n) if depth[m] < L - 1]
        parent[n] = cands[int(rng.integers(0, len(cands)))]
        depth[n] = depth[parent[n]] + 1
    tokens = np.zeros(N, np.int32)
    tokens[0] = int(rng.integers(0, V))
    for n in range(1, N):
        used = {int(tokens[m]) for m in range(1, n) if parent[m] == parent[n]}
        free = [t for t in range(V) if t not in used]
        tokens[n] = free[int(rng.integers(0, len(free)))]
    return parent, tokens, _paths_from_parents(parent, L, N)


def pin_tree_sampled(lib=None) -> list[str]:
    """Stochastic tree verify (reading T5: chosen children are point-mass
    proposals).  Exact enumeration of every branch on small trees: each
    branch's outcome, and the theorem that at every reached node the next
    emitted token is distributed as that node's target row, to 1e-12.  A
    one-chain tree equals the chain verify with one-hot draft rows; one-hot
    target rows equal the greedy tree verify; the near-tie windows on closed
    forms; fail-closed inputs."""
    errs = []
    rng = np.random.default_rng(41)
    for trial, (N, V, L, T) in enumerate([(4, 5, 3, 1.0), (6, 4, 4, 0.7), (7, 6, 3, 1.3), (5, 3, 5, 0.9)]):
        parent, tokens, paths = _random_small_tree(rng, N, V, L)
        target = (rng.standard_normal((N, V)) * 1.5).astype(np.float32)
        # make the drafted children likely under their parent's row
        for n in range(1, N):
            target[parent[n], tokens[n]] += 1.0
        branches, p_of = enumerate_tree_sampled(target, tokens, paths, T)
        wts = np.array([b[0] for b in branches])
        if abs(wts.sum() - 1.0) > 1e-12:
            errs.append(f"tree {trial}: branch weights sum to {wts.sum()}")
        n = len(branches)
        res = oracle.verify_tree_sampled(np.broadcast_to(target, (n, N, V)).copy(),
                                         np.broadcast_to(tokens, (n, N)).copy(),
                                         np.broadcast_to(paths, (n,) + paths.shape).copy(),
                                         np.array([b[3] for b in branches], np.float32), T, lib=lib)
        for e, (_, nacc, toks, _, _) in enumerate(branches):
            if res["num_accepted"][e] != nacc or list(res["tokens"][e]) != toks:
                errs.append(f"tree {trial}: branch {e} gave {res['tokens'][e]} (n={res['num_accepted'][e]}), "
                            f"want {toks} (n={nacc})")
                break
        # theorem: at each reached node, the next emitted token ~ p_node
        for node in range(N):
            reach = np.array([node in b[4] for b in branches])
            pos = [b[4].index(node) if node in b[4] else -1 for b in branches]
            if not reach.any():
                continue
            pr = wts[reach].sum()
            dist = np.zeros(V)
            for e in np.flatnonzero(reach):
                dist[branches[e][2][pos[e]]] += wts[e]
            if np.max(np.abs(dist / pr - p_of[node])) > 1e-12:
                errs.append(f"tree {trial}: token after node {node} is not distributed as its row")
                break
    # one-chain tree == chain verify with one-hot draft rows (q = point mass)
    k, V, T = 3, 9, 0.8
    target = (rng.standard_normal((20, k + 1, V)) * 2).astype(np.float32)
    x = rng.integers(0, V, (20, k)).astype(np.int32)
    u = rng.random((20, k + 1)).astype(np.float32)
    draft = np.full((20, k, V), -np.inf, np.float32)
    for b in range(20):
        draft[b, np.arange(k), x[b]] = 0.0
    chain = oracle.verify_chain(target, draft, x, u, T, lib=lib)
    toks = np.concatenate([np.zeros((20, 1), np.int32), x], axis=1)
    paths = np.tile(np.arange(k + 1, dtype=np.int32), (20, 1, 1))
    tu = np.concatenate([u[:, k:], u[:, :k]], axis=1)
    tree = oracle.verify_tree_sampled(target, toks, paths, tu, T, lib=lib)
    if not (np.array_equal(tree["tokens"], chain["tokens"]) and
            np.array_equal(tree["num_accepted"], chain["num_accepted"])):
        errs.append("a one-chain tree differs from the chain verify with one-hot draft rows")
    # one-hot target rows: the stochastic walk is the greedy tree verify
    for trial in range(30):
        N, V, L = int(rng.integers(2, 12)), int(rng.integers(12, 20)), int(rng.integers(2, 5))
        parent, tokens, paths = _random_small_tree(rng, N, V, L)
        g = rng.integers(0, V, N)
        for n in range(1, N):
            if rng.random() < 0.6:
                g[parent[n]] = tokens[n]
        target = np.full((N, V), -np.inf, np.float32)
        target[np.arange(N), g] = 1.0
        u = rng.random((1, N)).astype(np.float32)
        a = oracle.verify_tree_sampled(target[None], tokens[None], paths[None], u, 1.0, lib=lib)
        gr = oracle.verify_tree(target[None], tokens[None], paths[None], lib=lib)
        if not (np.array_equal(a["tokens"], gr["tokens"]) and
                np.array_equal(a["accepted_nodes"], gr["accepted_nodes"])):
            errs.append(f"one-hot rows: stochastic walk {a['tokens']} differs from greedy {gr['tokens']}")
            break
    # near-tie windows: root with children 1, 2 (tokens 0, 1) over V = 3,
    # target row 0 = [a, b, 0] at T = 1; child 2's test divides by 1 - p(0)
    a_, b_ = np.float32(0.4), np.float32(-0.3)
    z = np.array([a_, b_, 0.0], np.float64)
    p0 = np.exp(z) / np.exp(z).sum()
    target = np.zeros((1, 3, 3), np.float32)
    target[0, 0] = [a_, b_, 0.0]
    toks = np.array([[2, 0, 1]], np.int32)
    paths = np.array([[[0, 1], [0, 2]]], np.int32)
    for d, want_n, want_flag in [(5e-6, 0, True), (-5e-6, 1, True), (2e-5, 0, False), (-2e-5, 1, False)]:
        u = np.array([[0.5, p0[0] + d, 0.99]], np.float32)
        r = oracle.verify_tree_sampled(target, toks, paths, u, 1.0, lib=lib)
        if r["num_accepted"][0] != want_n or bool(r["flags"][0, 1]) != want_flag:
            errs.append(f"tree accept window at p {d:+g}: n={r['num_accepted'][0]} flag={r['flags'][0, 1]}")
    r2 = p0[1] / (1 - p0[0])
    win = 1e-5 / (1 - p0[0])
    # (0.8 of the scaled window is beyond the unscaled 1e-5: p(0) is about 0.46)
    for d, want_tok, want_flag in [(0.8 * win, 2, True), (-0.8 * win, 1, True), (2 * win, 2, False),
                                   (-2 * win, 1, False)]:
        u = np.array([[0.5, 0.999, r2 + d]], np.float32)
        r = oracle.verify_tree_sampled(target, toks, paths, u, 1.0, lib=lib)
        got_n = r["num_accepted"][0]
        if (got_n == 1) != (want_tok == 1) or bool(r["flags"][0, 2]) != want_flag:
            errs.append(f"second child's window at {d:+g}: n={got_n} flag={r['flags'][0, 2]}")
    # fail closed
    target = rng.standard_normal((2, 3, 5)).astype(np.float32)
    toks = np.array([[0, 1, 5], [0, 1, 2]], np.int32)
    paths = np.array([[[0, 1, 2]], [[0, 3, -1]]], np.int32)
    r = oracle.verify_tree_sampled(target, toks, paths, np.full((2, 3), 0.5, np.float32), 1.0, lib=lib)
    if r["rc"] != oracle.EBADINDEX or list(r["num_accepted"]) != [-1, -1] or np.any(r["tokens"] != -1):
        errs.append("bad tree tokens or node ids must fail closed")
    # no used path: one draw from the root row at u[0], best path -1
    paths = np.full((1, 2, 3), -1, np.int32)
    u = np.array([[0.37, 0.1, 0.2]], np.float32)
    r = oracle.verify_tree_sampled(target[:1], np.array([[0, 1, 2]], np.int32), paths, u, 1.0, lib=lib)
    want, _ = oracle.inverse_cdf(_softmax_T(target[0, 0], 1.0), 0.37)
    if r["num_accepted"][0] != 0 or r["tokens"][0, 0] != want or r["best_path"][0] != -1:
        errs.append("a tree without used paths must draw once from the root row")
    return errs


def pin_filter_min_p_and_wide_top_p(lib=None) -> list[str]:
    """min_p and top-p over the whole vocabulary (reading F6: temperature, then
    top-k, top-p and min_p in the walkthrough's order; top_k = 0 keeps every
    token).  Closed-form hand examples, a min_p tie kept and flagged, 300
    random rows against numpy's sort and cumulative sums, and the equivalence
    theorem on enumerated branches with both sides filtered by top-p and
    min_p alone."""
    errs = []
    fr = lambda x, T, kk, pp, mp: oracle.filtered_softmax(np.asarray(x, np.float32), T, kk, pp, lib=lib,
                                                          min_p=mp)
    x = [3.0, 1.0, 2.0, 2.0, 0.0]
    e1, e2, e3 = np.exp(-1.0), np.exp(-2.0), np.exp(-3.0)
    cases = [  # (T, top_k, top_p, min_p, expected p)
        # min_p = e^-1.5 keeps the logits within 1.5 of the maximum
        (1.0, 0, 1.0, np.exp(-1.5), np.array([1.0, 0.0, e1, e1, 0.0]) / (1.0 + 2 * e1)),
        # min_p = 1/2 keeps the maximum alone
        (1.0, 0, 1.0, 0.5, np.array([1.0, 0.0, 0.0, 0.0, 0.0])),
        # top-p over the whole vocabulary: p(0) = 1/(1 + e^-2 + 2e^-1 + e^-3) = 0.521 < 0.55,
        # so token 2 joins (over the top 3 alone 0.576 would reach it)
        (1.0, 0, 0.55, 0.0, np.array([1.0, 0.0, e1, 0.0, 0.0]) / (1.0 + e1)),
        # min_p after top-p: top-p 0.9 keeps {0, 2, 3, 1}, min_p e^-1.2 then drops token 1
        (1.0, 0, 0.9, np.exp(-1.2), np.array([1.0, 0.0, e1, e1, 0.0]) / (1.0 + 2 * e1)),
        # top-k, then min_p: top_k = 2 keeps {0, 2}; min_p e^-1.5 keeps both
        (1.0, 2, 1.0, np.exp(-1.5), np.array([1.0, 0.0, e1, 0.0, 0.0]) / (1.0 + e1)),
        # temperature applies before min_p: at T = 2, exp((2 - 3)/2) = 0.607 >= 0.6
        (2.0, 0, 1.0, 0.6, np.array([1.0, 0.0, np.exp(-0.5), np.exp(-0.5), 0.0]) / (1.0 + 2 * np.exp(-0.5))),
    ]
    for T, kk, pp, mp, want in cases:
        got, _ = fr(x, T, kk, pp, mp)
        if np.max(np.abs(got - want)) > 1e-12:
            errs.append(f"filter T={T} top_k={kk} top_p={pp} min_p={mp:.4f}: {got} want {want}")
    # a token exactly at min_p is kept, and the row is flagged as a near tie
    got, tie = fr(x, 1.0, 0, 1.0, e1)
    if np.max(np.abs(got - np.array([1.0, 0.0, e1, e1, 0.0]) / (1.0 + 2 * e1))) > 1e-12 or not tie:
        errs.append(f"a token exactly at min_p must be kept and flagged: {got} {tie}")
    # min_p decides an accept test: target row [0, 0, -0.5, -3] with min_p =
    # e^-1 keeps tokens 0..2, p(0) = 1 / (2 + e^-0.5) = 0.3861 (unfiltered it
    # would be 0.3693); the draft row is one-hot at token 0, so r = 0.378
    # accepts token 0 only under the filtered target row.
    tgt = np.array([[[0.0, 0.0, -0.5, -3.0], [0.0, -1.0, 0.5, 0.0]]], np.float32)
    drf = np.array([[[0.0, -np.inf, -np.inf, -np.inf]]], np.float32)
    res = oracle.verify_chain_filtered(tgt, drf, np.array([[0]], np.int32),
                                       np.array([[0.378, 0.2]], np.float32), 1.0, 0, 1.0, lib=lib, min_p=e1)
    if res["num_accepted"][0] != 1 or abs(res["probs"][0, 0, 0] - 1.0 / (2.0 + np.exp(-0.5))) > 1e-12:
        errs.append(f"min_p accept example: n={res['num_accepted'][0]} p={res['probs'][0, 0, 0]}")
    # min_p = 1 keeps the tied maxima; no filter at all is scipy's softmax
    got, _ = fr([5.0, 1.0, 5.0, 2.0], 1.0, 0, 1.0, 1.0)
    if got.tolist() != [0.5, 0.0, 0.5, 0.0]:
        errs.append(f"min_p = 1 must keep the tied maxima: {got}")
    rng = np.random.default_rng(19)
    row = (rng.standard_normal(50) * 2).astype(np.float32)
    if np.max(np.abs(fr(row, 0.7, 0, 1.0, 0.0)[0] - _softmax_T(row, 0.7))) > 1e-12:
        errs.append("no filter is not the plain softmax")
    for trial in range(300):
        V = int(rng.integers(2, 60))
        xr = (rng.integers(-6, 7, size=V) * 0.5).astype(np.float32)
        T = float(rng.choice([0.5, 1.0, 1.6]))
        kk = int(rng.choice([0, 0, 1, 3, V + 2]))
        pp = float(np.float32(rng.choice([0.3, 0.6, 0.9, 1.0])))
        mp = float(rng.choice([0.0, 0.01, 0.1, 0.5]))
        got, tie = fr(xr, T, kk, pp, mp)
        if tie:
            continue
        want = _filter_np(xr, T, kk, pp, mp)
        if np.max(np.abs(got - want)) > 1e-12:
            errs.append(f"filter row {trial} (top_k={kk}, top_p={pp}, min_p={mp}) differs from numpy")
            break
    # kept sets of hundreds to thousands of tokens (top_k above 256, top-p and
    # min_p over wide rows), logits on a coarse grid so that the cuts fall
    # inside runs of equal values
    for trial in range(24):
        V = int(rng.integers(300, 3000))
        xr = (np.round(rng.standard_normal(V) * 24) / 8).astype(np.float32)
        T = float(rng.choice([0.7, 1.0, 2.0]))
        kk = int(rng.choice([0, 0, 257, 1000, V - 1]))
        pp = float(np.float32(rng.choice([0.5, 0.9, 0.99, 1.0])))
        mp = float(rng.choice([0.0, 0.0, 1e-4, 0.01]))
        got, tie = fr(xr, T, kk, pp, mp)
        if tie:
            continue
        want = _filter_np(xr, T, kk, pp, mp)
        if np.max(np.abs(got - want)) > 1e-12 or not np.array_equal(got > 0, want > 0):
            errs.append(f"wide filter row {trial} (V={V}, top_k={kk}, top_p={pp}, min_p={mp}) differs from numpy")
            break
    for (k2, V2, T2, filt) in [(1, 6, 1.0, (0, 0.8, 0.0)), (2, 5, 0.8, (0, 1.0, 0.2)),
                               (2, 4, 1.2, (0, 0.7, 0.1)), (2, 5, 1.0, (3, 0.9, 0.3))]:
        tg = (rng.standard_normal((k2 + 1, V2)) * 1.5).astype(np.float32)
        dr = (tg[:k2] + rng.standard_normal((k2, V2)) * 0.8).astype(np.float32)
        wts, expect, res, p = enumerate_chain(tg, dr, T2, lib=lib, filt=filt)
        for e, (j, rowe) in enumerate(expect):
            if res["num_accepted"][e] != j or list(res["tokens"][e]) != rowe:
                errs.append(f"filter {filt} k={k2}: branch {e} gave {res['tokens'][e]} want {rowe}")
                break
        n_acc, toks = res["num_accepted"], res["tokens"]
        for i in range(k2 + 1):
            reach = n_acc >= i
            dist = np.array([wts[reach & (toks[:, i] == t)].sum() for t in range(V2)]) / wts[reach].sum()
            if np.max(np.abs(dist - p[i])) > 1e-12:
                errs.append(f"filter {filt} k={k2}: token {i} is not distributed as filtered p_{i}")
    return errs


ALL_PINS = {
    "softmax": pin_softmax,
    "inverse_cdf": pin_inverse_cdf,
    "near_ties": pin_near_ties,
    "exact_distribution": pin_exact_distribution,
    "invariants": pin_invariants,
    "greedy": pin_greedy,
    "tree": pin_tree,
    "rollback": pin_rollback,
    "worked_example": pin_worked_example,
    "filtered": pin_filtered,
    "philox": pin_philox,
    "rollback_paged": pin_rollback_paged,
    "ragged": pin_ragged,
    "tree_sampled": pin_tree_sampled,
    "filter_min_p_wide_top_p": pin_filter_min_p_and_wide_top_p,
}
