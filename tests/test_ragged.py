"""Ragged per-request draft lengths and paged block accounting (TensorRT-LLM
walkthrough: pad_draft_tokens_for_cuda_graph keeps the real draft count in
py_draft_tokens_effective_len while the buffer is padded to the static
maximum; update_requests rewinds verified_len - accepted; rewind_cache
returns the whole surplus blocks).  Oracle pins on the CPU; the CUDA path
against the oracle on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _chain(seed=4, B=6, k=5, V=700, T=0.9):
    rng = np.random.default_rng(seed)
    target = rng.normal(0, 2, size=(B, k + 1, V)).astype(np.float32)
    draft = (target[:, :k] + rng.normal(0, 0.6, size=(B, k, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    r = rng.random((B, k + 1), dtype=np.float32)
    return target, draft, x, r, T


def test_full_lengths_equal_the_plain_call():
    target, draft, x, r, T = _chain()
    a = oracle.verify_chain(target, draft, x, r, T)
    b = oracle.verify_chain(target, draft, x, r, T, draft_lens=np.full(6, 5, np.int32))
    for key in ("tokens", "num_accepted", "probs", "flags"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_each_request_is_the_truncated_chain():
    target, draft, x, r, T = _chain()
    B, k = x.shape
    lens = np.array([1, 2, 3, 4, 5, 3], np.int32)
    x = x.copy()
    x[0, 1:] = -7          # padding: never read or checked
    got = oracle.verify_chain(target, draft, x, r, T, draft_lens=lens)
    for b in range(B):
        kb = int(lens[b])
        rr = np.concatenate([r[b, :kb], r[b, kb:kb + 1]])[None]
        want = oracle.verify_chain(target[b:b + 1, :kb + 1], draft[b:b + 1, :kb], x[b:b + 1, :kb], rr, T)
        assert got["num_accepted"][b] == want["num_accepted"][0]
        assert np.array_equal(got["tokens"][b, :kb + 1], want["tokens"][0])
        assert np.all(got["tokens"][b, kb + 1:] == -1)
        assert np.array_equal(got["probs"][b, :kb], want["probs"][0])
        assert np.all(np.isnan(got["probs"][b, kb:]))


def test_zero_drafts_is_one_draw_from_the_first_target_row():
    target, draft, x, r, T = _chain()
    lens = np.zeros(6, np.int32)
    got = oracle.verify_chain(target, draft, x, r, T, draft_lens=lens)
    for b in range(6):
        p = oracle.softmax(target[b, 0], T)
        tok, _ = oracle.inverse_cdf(p, float(r[b, 0]))
        assert got["num_accepted"][b] == 0
        assert got["tokens"][b, 0] == tok and np.all(got["tokens"][b, 1:] == -1)


@pytest.mark.parametrize("bad", [-1, 6])
def test_length_out_of_range_fails_closed(bad):
    target, draft, x, r, T = _chain()
    lens = np.full(6, 3, np.int32)
    lens[2] = bad
    got = oracle.verify_chain(target, draft, x, r, T, draft_lens=lens)
    assert got["num_accepted"][2] == -1 and np.all(got["tokens"][2] == -1)
    assert got["rc"] == oracle.EBADINDEX
    assert np.all(got["num_accepted"][[0, 1, 3, 4, 5]] >= 0)


def test_greedy_ragged_is_the_truncated_greedy():
    target, _, x, _, _ = _chain(seed=9)
    lens = np.array([0, 1, 2, 5, 4, 3], np.int32)
    x = x.copy()
    for b in range(6):  # make some prefixes match the argmax so acceptance is not trivially 0
        for i in range(lens[b]):
            if (b + i) % 2 == 0:
                x[b, i] = int(np.argmax(target[b, i]))
    got = oracle.verify_greedy(target, x, draft_lens=lens)
    for b in range(6):
        kb = int(lens[b])
        if kb == 0:
            assert got["num_accepted"][b] == 0 and got["tokens"][b, 0] == int(np.argmax(target[b, 0]))
            continue
        want = oracle.verify_greedy(target[b:b + 1, :kb + 1], x[b:b + 1, :kb])
        assert got["num_accepted"][b] == want["num_accepted"][0]
        assert np.array_equal(got["tokens"][b, :kb + 1], want["tokens"][0])
        assert np.all(got["tokens"][b, kb + 1:] == -1)


def test_paged_rollback_closed_forms():
    # old 10, 2 of 3 drafts accepted: 13 tokens, rewind 1; 4 per block -> 4 blocks needed
    res = oracle.rollback_paged([10, 10, 7, 0], [2, 0, 3, 0], k=4, tokens_per_block=4,
                                draft_lens=[3, 0, 3, 2], blocks_held=[5, 3, 2, 1])
    assert res["new_lens"].tolist() == [13, 11, 11, 1]
    assert res["rewind_lens"].tolist() == [1, 0, 0, 2]
    assert res["free_blocks"].tolist() == [1, 0, 0, 0]   # ceil(13/4)=4, ceil(11/4)=3, 3>2 keeps 0, 1-1=0
    # n > k_b and k_b > k are refused entry by entry
    bad = oracle.rollback_paged([5, 5], [3, 1], k=4, tokens_per_block=4, draft_lens=[2, 9], blocks_held=[9, 9])
    assert bad["rc"] == oracle.EBADINDEX
    assert bad["new_lens"].tolist() == [5, 5] and bad["free_blocks"].tolist() == [0, 0]
    # without lengths it is the plain rollback
    rng = np.random.default_rng(2)
    old = rng.integers(0, 1000, 50).astype(np.int32)
    n = rng.integers(0, 8, 50).astype(np.int32)
    a = oracle.rollback(old, n, 7)
    b = oracle.rollback_paged(old, n, 7, tokens_per_block=16)
    assert np.array_equal(a["new_lens"], b["new_lens"]) and np.array_equal(a["rewind_lens"], b["rewind_lens"])
