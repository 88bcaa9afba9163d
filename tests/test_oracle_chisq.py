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
