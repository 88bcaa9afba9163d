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


# ------------------------------------------------------------------ GPU parity
def _ragged_workload(name, seed, **over):
    w = workloads.make(name, seed=seed, **over)
    rng = np.random.default_rng(seed)
    k = w["k"]
    lens = rng.integers(0, k + 1, size=w["B"]).astype(np.int32)
    lens[0], lens[-1] = 0, k
    x = w["draft_tokens"].copy()
    for b in range(w["B"]):
        x[b, lens[b]:] = -3 if b % 2 else w["V"] + 11   # padding outside [0, V): never checked
    w["draft_tokens"] = x
    w["draft_lens"] = lens
    return w


@pytest.mark.gpu
@pytest.mark.parametrize("philox", [False, True])
@pytest.mark.parametrize("name,over", [("chain_b64_k7_v128256_bf16", dict(B=24, V=30000)),
                                       ("chain_b8_k4_v32000_f32", dict(V=9000)),
                                       ("chain_b256_k3_v129280_bf16", dict(B=40, V=20000))])
def test_chain_ragged_matches_oracle(name, over, philox):
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import check_chain, to_dev, i32
    w = _ragged_workload(name, 31, **over)
    B, k = w["B"], w["k"]
    kw = {}
    if philox:
        seeds = np.full(B, 77, dtype=np.int64)
        offsets = np.arange(B, dtype=np.int64) * 1000 + 5
        w["uniforms"] = oracle.philox_uniforms(seeds.view(np.uint64), offsets.view(np.uint64), k + 1)
        kw = dict(seeds=torch.from_numpy(seeds).cuda(), offsets=torch.from_numpy(offsets).cuda())
        u = None
    else:
        u = torch.from_numpy(w["uniforms"]).cuda()
    seq = i32(w["seq_lens"])
    tok, n, probs = sv.verify_chain(to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"]),
                                    i32(w["draft_tokens"]), u, w["temperature"], want_probs=True,
                                    seq_lens=seq, draft_lens=i32(w["draft_lens"]), **kw)
    torch.cuda.synchronize()
    o = oracle.verify(w)
    assert o["rc"] == oracle.OK                      # padding tokens are never checked
    g = dict(tokens=tok.cpu().numpy(), num_accepted=n.cpu().numpy(), probs=probs.cpu().numpy(),
             seq_lens=seq.cpu().numpy())
    pad = np.isnan(o["probs"])
    assert np.array_equal(np.isnan(g["probs"]), pad)  # padded positions are NaN on both sides
    g["probs"][pad] = 0.0
    o = dict(o, probs=np.where(pad, 0.0, o["probs"]))
    check_chain(w, g, o, f"ragged {name}{' philox' if philox else ''}")


@pytest.mark.gpu
def test_chain_ragged_bad_length_fails_closed():
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import to_dev, i32
    w = _ragged_workload("chain_b64_k7_v128256_bf16", 5, B=6, V=5000)
    w["draft_lens"][2] = 9                            # > k
    w["draft_lens"][4] = -1
    ws = sv.Workspace()
    tok, n, _ = sv.verify_chain(to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"]),
                                i32(w["draft_tokens"]), torch.from_numpy(w["uniforms"]).cuda(),
                                w["temperature"], draft_lens=i32(w["draft_lens"]), workspace=ws)
    torch.cuda.synchronize()
    o = oracle.verify(w)
    assert np.array_equal(n.cpu().numpy(), o["num_accepted"])
    assert np.array_equal(tok.cpu().numpy()[[2, 4]], o["tokens"][[2, 4]])
    assert n.cpu().numpy()[2] == -1 and n.cpu().numpy()[4] == -1
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX


@pytest.mark.gpu
@pytest.mark.parametrize("name,over", [("chain_b8_k4_v32000_f32", {}),
                                       ("chain_b64_k7_v128256_bf16", dict(B=16, V=40000))])
def test_greedy_ragged_matches_oracle(name, over):
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import to_dev, i32
    w = _ragged_workload(name, 8, **over)
    # let some requests accept: copy the target argmax into the draft
    for b in range(w["B"]):
        for i in range(w["draft_lens"][b]):
            if (b + i) % 3:
                w["draft_tokens"][b, i] = oracle.argmax(w["target"][b, i], w["dtype"])
    seq = i32(w["seq_lens"])
    tok, n = sv.verify_greedy(to_dev(w["target"], w["dtype"]), i32(w["draft_tokens"]), seq_lens=seq,
                              draft_lens=i32(w["draft_lens"]))
    torch.cuda.synchronize()
    o = oracle.verify(w, greedy=True)
    assert np.array_equal(n.cpu().numpy(), o["num_accepted"])
    assert np.array_equal(tok.cpu().numpy(), o["tokens"])
    assert (o["num_accepted"] > 0).sum() >= 3
    want_seq = oracle.rollback(w["seq_lens"], o["num_accepted"], w["k"])["new_lens"]
    assert np.array_equal(seq.cpu().numpy(), want_seq)


@pytest.mark.gpu
def test_rollback_paged_matches_oracle():
    import speculative_decoding_verification_row_gb300 as sv
    rng = np.random.default_rng(12)
    B, k, tpb = 3000, 7, 16
    lens = rng.integers(-1, k + 2, size=B).astype(np.int32)
    n = np.array([rng.integers(-1, max(int(l), 0) + 2) for l in lens], dtype=np.int32)
    old = rng.integers(0, 5000, size=B).astype(np.int32)
    held = ((old + k + 1 + tpb - 1) // tpb + rng.integers(0, 3, size=B)).astype(np.int32)
    want = oracle.rollback_paged(old, n, k, tpb, draft_lens=lens, blocks_held=held)
    d = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    new, rew, fre = sv.rollback_paged(d(old), d(n), k, tpb, draft_lens=d(lens), blocks_held=d(held))
    torch.cuda.synchronize()
    assert np.array_equal(new.cpu().numpy(), want["new_lens"])
    assert np.array_equal(rew.cpu().numpy(), want["rewind_lens"])
    assert np.array_equal(fre.cpu().numpy(), want["free_blocks"])
    assert (want["free_blocks"] > 0).any() and (want["rc"] == oracle.EBADINDEX)
