"""Monte-Carlo chi-square check of the oracle's chain verify at V=16, k=3.

The equivalence theorem (vLLM anatomy page, "Why this works"; vLLM learning
book, section 2) says the emitted token at position i, given that position i
was reached, follows the target row p_i, and that position i+1 is reached with
probability sum_t min(p_i(t), q_i(t)).  Draft tokens are drawn from q with
numpy's own sampler and the uniforms from numpy's generator.
"""
import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chisquare

import oracle


def _chisq(counts, probs, min_expected=5.0):
    n = counts.sum()
    exp = probs * n
    big = exp >= min_expected
    obs = np.append(counts[big], counts[~big].sum())
    ex = np.append(exp[big], exp[~big].sum())
    if ex[-1] == 0:
        obs, ex = obs[:-1], ex[:-1]
    ex = ex * obs.sum() / ex.sum()
    return chisquare(obs, ex).pvalue


@pytest.mark.parametrize("seed", [0, 1])
def test_chain_chisquare(seed):
    rng = np.random.default_rng(100 + seed)
    k, V, T, n = 3, 16, 0.9, 200_000
    target = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    draft = (target[:k] + rng.standard_normal((k, V))).astype(np.float32)
    Tf = np.float64(np.float32(T))
    p = [softmax(target[i].astype(np.float64) / Tf) for i in range(k + 1)]
    q = [softmax(draft[i].astype(np.float64) / Tf) for i in range(k)]
    x = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(k)], axis=1).astype(np.int32)
    u = rng.random((n, k + 1), dtype=np.float32)
    res = oracle.verify_chain(np.broadcast_to(target, (n, k + 1, V)),
                              np.broadcast_to(draft, (n, k, V)), x, u, T)
    n_acc, toks = res["num_accepted"], res["tokens"]
    pvals = []
    for i in range(k + 1):
        reach = n_acc >= i
        counts = np.bincount(toks[reach, i], minlength=V).astype(np.float64)
        pvals.append(_chisq(counts, p[i]))
    beta = [np.minimum(p[i], q[i]).sum() for i in range(k)]
    law = np.array([np.prod(beta[:j]) * (1 - beta[j]) for j in range(k)] + [np.prod(beta)])
    pvals.append(_chisq(np.bincount(n_acc, minlength=k + 1).astype(np.float64), law))
    assert min(pvals) > 1e-3, pvals


@pytest.mark.parametrize("top_k,top_p", [(6, 1.0), (6, 0.8)])
def test_filtered_chain_chisquare(top_k, top_p):
    # The same theorem on filtered rows: with draft tokens drawn from the
    # filtered draft rows, the emitted token at a reached position follows the
    # filtered target row (TensorRT-LLM walkthrough, rejection-sampling
    # section: both sides filtered alike), and position i+1 is reached with
    # probability sum_t min(p_i(t), q_i(t)) of the filtered rows.
    rng = np.random.default_rng(300 + top_k + int(10 * top_p))
    k, V, T, n = 3, 16, 0.9, 200_000
    target = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    draft = (target[:k] + rng.standard_normal((k, V))).astype(np.float32)
    tp = float(np.float32(top_p))
    p = [oracle.filtered_softmax(target[i], T, top_k, tp)[0] for i in range(k + 1)]
    q = [oracle.filtered_softmax(draft[i], T, top_k, tp)[0] for i in range(k)]
    x = np.stack([rng.choice(V, size=n, p=q[i] / q[i].sum()) for i in range(k)],
                 axis=1).astype(np.int32)
    u = rng.random((n, k + 1), dtype=np.float32)
    res = oracle.verify_chain_filtered(np.broadcast_to(target, (n, k + 1, V)),
                                       np.broadcast_to(draft, (n, k, V)), x, u, T, top_k, tp)
    n_acc, toks = res["num_accepted"], res["tokens"]
    pvals = []
    for i in range(k + 1):
        reach = n_acc >= i
        counts = np.bincount(toks[reach, i], minlength=V).astype(np.float64)
        assert counts[p[i] == 0].sum() == 0  # nothing outside the kept set
        pvals.append(_chisq(counts, p[i]))
    beta = [np.minimum(p[i], q[i]).sum() for i in range(k)]
    law = np.array([np.prod(beta[:j]) * (1 - beta[j]) for j in range(k)] + [np.prod(beta)])
    pvals.append(_chisq(np.bincount(n_acc, minlength=k + 1).astype(np.float64), law))
    assert min(pvals) > 1e-3, pvals


def test_tree_sampled_chisquare():
    # A tree of 8 nodes over V = 16 with children chosen as the top tokens of
    # their parent's row (as a top-K drafter does): 200 000 walks with
    # numpy's uniforms.  At the root and at each accepted child, the next
    # emitted token must follow that node's target row.
    rng = np.random.default_rng(211)
    V, T, n = 16, 0.8, 200_000
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 4])
    N = parent.size
    target = (rng.standard_normal((N, V)) * 1.5).astype(np.float32)
    tokens = np.zeros(N, np.int32)
    for par in range(N):
        kids = np.flatnonzero(parent == par)
        top = np.argsort(-(target[par] + rng.standard_normal(V) * 0.3), kind="stable")
        tokens[kids] = top[: kids.size]
    paths = np.array([[0, 1, 4, 7], [0, 1, 5, -1], [0, 2, 6, -1], [0, 3, -1, -1]], np.int32)
    u = rng.random((n, N), dtype=np.float32)
    res = oracle.verify_tree_sampled(np.broadcast_to(target, (n, N, V)), np.broadcast_to(tokens, (n, N)),
                                     np.broadcast_to(paths, (n,) + paths.shape), u, T)
    Tf = np.float64(np.float32(T))
    nodes, toks = res["accepted_nodes"], res["tokens"]
    pvals = []
    for node in range(N):
        for d in range(paths.shape[1]):
            reach = nodes[:, d] == node
            if reach.sum() < 2000:
                continue
            p = softmax(target[node].astype(np.float64) / Tf)
            counts = np.bincount(toks[reach, d], minlength=V).astype(np.float64)
            pvals.append(_chisq(counts, p))
    assert len(pvals) >= 3
    assert min(pvals) > 1e-3, pvals


def test_q_based_tree_rule_is_biased_for_chosen_children():
    # Why the stochastic tree verify treats chosen children as point-mass
    # proposals: the rule that tests each child against the draft row q
    # (accept with min(1, p/q), continue from max(0, p - q) normalised) keeps
    # the target distribution only when the children are independent draws
    # from q.  With the two top tokens of q as children it does not: the
    # first emitted token's law, computed exactly here, differs from p.
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.1, 0.6, 0.3])
    kids = [1, 2]  # the top-2 tokens of q, in order
    law = np.zeros(3)
    stay, resid = 1.0, p.copy()
    for c in kids:
        a = min(1.0, resid[c] / q[c])
        law[c] += stay * a
        stay *= 1.0 - a
        resid = np.maximum(resid - q, 0.0)
        resid /= resid.sum()
    law += stay * resid
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.max(np.abs(law - p)) > 0.05
    # the point-mass rule on the same children gives p exactly
    law2 = np.zeros(3)
    stay, resid = 1.0, p.copy()
    for c in kids:
        a = resid[c] / resid.sum()
        law2[c] += stay * a
        stay *= 1.0 - a
        resid[c] = 0.0
    law2 += stay * resid / resid.sum()
    assert np.max(np.abs(law2 - p)) < 1e-12
