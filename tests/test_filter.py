"""Symmetric top-k / top-p filtering before verify (TensorRT-LLM walkthrough,
rejection-sampling section: the target must be filtered exactly as the draft
was, or acceptance goes silently wrong).  Oracle pins on the CPU; the CUDA
path against the oracle on the GPU."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads


def test_filtered_softmax_hand_example():
    x = np.array([3.0, 1.0, 2.0, 2.0, 0.0], np.float32)
    # top-3 by (logit desc, index asc): tokens 0, 2, 3
    p, tie = oracle.filtered_softmax(x, 1.0, top_k=3)
    e = np.exp(np.array([0.0, -1.0, -1.0]))
    want = np.zeros(5)
    want[[0, 2, 3]] = e / e.sum()
    assert np.allclose(p, want, rtol=0, atol=1e-15) and not tie
    # top-p 0.5: the first token alone already reaches it
    p, _ = oracle.filtered_softmax(x, 1.0, top_k=3, top_p=0.5)
    assert p.tolist() == [1.0, 0.0, 0.0, 0.0, 0.0]
    # top-p 0.6: tokens 0 and 2 (the tie at logit 2 goes to the lower index)
    p, _ = oracle.filtered_softmax(x, 1.0, top_k=3, top_p=0.6)
    a = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(p, [a, 0.0, 1.0 - a, 0.0, 0.0], rtol=0, atol=1e-15)
    # a cut exactly at the threshold is flagged as a near tie
    p0 = 1.0 / (1.0 + 2.0 * math.exp(-1.0))
    _, tie = oracle.filtered_softmax(x, 1.0, top_k=3, top_p=p0)
    assert tie
    # temperature applies before the cut: T = 2 flattens the top-3
    p, _ = oracle.filtered_softmax(x, 2.0, top_k=3)
    e2 = np.exp(np.array([0.0, -0.5, -0.5]))
    assert np.allclose(p[[0, 2, 3]], e2 / e2.sum(), rtol=0, atol=1e-15)


def _chain(seed, B=12, k=4, V=40, T=0.8):
    rng = np.random.default_rng(seed)
    target = rng.normal(0, 2, size=(B, k + 1, V)).astype(np.float32)
    draft = (target[:, :k] + rng.normal(0, 0.8, size=(B, k, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    r = rng.random((B, k + 1), dtype=np.float32)
    return target, draft, x, r, T


def test_top_k_at_least_v_is_the_plain_verify():
    target, draft, x, r, T = _chain(1)
    a = oracle.verify_chain(target, draft, x, r, T)
    b = oracle.verify_chain_filtered(target, draft, x, r, T, top_k=64)
    for key in ("tokens", "num_accepted"):
        assert np.array_equal(a[key], b[key]), key
    assert np.allclose(a["probs"], b["probs"], rtol=1e-12, atol=0)


def test_top_1_is_greedy_verify():
    # top_k = 1 makes p and q one-hot at the argmaxes; with drafts at the
    # draft argmax, acceptance is argmax agreement and the correction/bonus
    # is the target argmax: greedy verify.
    target, draft, _, r, T = _chain(2)
    x = np.argmax(draft, axis=-1).astype(np.int32)
    x[::3, 0] = np.argmax(target[::3, 0], axis=-1)     # some first drafts agree
    draft[np.arange(0, 12, 3), 0, x[::3, 0]] += 100.0    # and are the draft argmax too
    g = oracle.verify_greedy(target, x)
    f = oracle.verify_chain_filtered(target, draft, x, r, T, top_k=1)
    assert np.array_equal(f["tokens"], g["tokens"]) and np.array_equal(f["num_accepted"], g["num_accepted"])
    assert (g["num_accepted"] > 0).any()


def test_filtered_probs_are_the_filtered_rows():
    target, draft, x, r, T = _chain(3, V=300)
    res = oracle.verify_chain_filtered(target, draft, x, r, T, top_k=20, top_p=0.9)
    for b in range(3):
        for i in range(4):
            p, _ = oracle.filtered_softmax(target[b, i], T, 20, 0.9)
            q, _ = oracle.filtered_softmax(draft[b, i], T, 20, 0.9)
            assert res["probs"][b, i, 0] == p[x[b, i]] and res["probs"][b, i, 1] == q[x[b, i]]
