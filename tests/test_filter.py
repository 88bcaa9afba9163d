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


# ---------------------------------------------------------------- CUDA path
def _filtered_tokens(w, top_k, top_p, seed, min_p=0.0):
    """Draft tokens sampled from the filtered draft rows (as a drafter that
    filters its own sampling would produce them)."""
    rng = np.random.default_rng(seed)
    B, k = w["B"], w["k"]
    x = np.empty((B, k), np.int32)
    for b in range(B):
        for i in range(k):
            q, _ = oracle.filtered_softmax(w["draft"][b, i], w["temperature"], top_k, top_p,
                                           w["dtype"], min_p=float(np.float32(min_p)))
            x[b, i] = rng.choice(q.size, p=q / q.sum())
    return x


def _run_filtered(w, top_k, top_p, *, misalign=False, workspace=None, philox=None,
                  draft_lens=None, min_p=0.0):
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import _offset_copy, i32, to_dev
    t, d = to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"])
    if misalign:
        t, d = _offset_copy(t), _offset_copy(d)
    seq = i32(w["seq_lens"])
    kw = {}
    if philox is not None:
        kw = dict(seeds=torch.from_numpy(philox[0]).cuda(), offsets=torch.from_numpy(philox[1]).cuda())
        u = None
    else:
        u = torch.from_numpy(w["uniforms"]).cuda()
    if draft_lens is not None:
        kw["draft_lens"] = i32(draft_lens)
    tok, n, probs = sv.verify_chain(t, d, i32(w["draft_tokens"]), u, w["temperature"],
                                    want_probs=True, seq_lens=seq, workspace=workspace,
                                    top_k=top_k, top_p=top_p, min_p=min_p, **kw)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), num_accepted=n.cpu().numpy(), probs=probs.cpu().numpy(),
                seq_lens=seq.cpu().numpy())


def _oracle_filtered(w, top_k, top_p, min_p=0.0):
    mp = float(np.float32(min_p))
    o = oracle.verify_chain_filtered(w["target"], w["draft"], w["draft_tokens"], w["uniforms"],
                                     w["temperature"], top_k, float(np.float32(top_p)), w["dtype"],
                                     min_p=mp)
    o["filter"] = (top_k, float(np.float32(top_p)), mp)
    return o


FILTER_CASES = [
    # (workload, overrides, top_k, top_p)
    ("chain_b1_k4_v1024_f32", dict(B=16), 1, 1.0),
    ("chain_b1_k4_v1024_f32", dict(B=16), 8, 0.9),
    ("chain_b1_k4_v1024_f32", dict(B=16), 50, 0.5),
    ("chain_b1_k4_v1024_f32", dict(B=16, V=200), 256, 1.0),       # top_k >= V: plain verify
    ("chain_b8_k4_v32000_f32", dict(B=8), 40, 0.95),                # peaked rows, 8 slices
    ("chain_b64_k7_v128256_bf16", dict(B=6, V=70000), 64, 0.9),     # bf16, 5 slices, ragged tail
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 256, 0.8),    # the largest top_k
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 150, 0.95),   # 129..256 keys held
    ("chain_b64_k7_v128256_bf16", dict(B=2, k=3, V=300000), 40, 0.9),  # 19 slices: 3 selection segments, 3-level draw
    ("chain_b8_k4_v32000_f32", dict(B=2, V=300000), 30, 0.95),      # f32, 37 slices: 5 segments
    ("chain_b8_k4_v32000_f32", dict(B=1, k=2, V=458752), 16, 0.9),  # 56 slices: the most codes a pick CTA holds
    ("chain_b8_k4_v32000_f32", dict(B=1, k=2, V=480000), 16, 0.9),  # 59 slices: the per-row kernel
    ("chain_b256_k3_v129280_bf16", dict(B=16, V=20000), 20, 1.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,over,top_k,top_p", FILTER_CASES)
def test_cuda_filtered_matches_oracle(name, over, top_k, top_p):
    from test_gpu_parity import check_chain
    w = workloads.make(name, seed=31, **over)
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 31)
    g = _run_filtered(w, top_k, top_p)
    check_chain(w, g, _oracle_filtered(w, top_k, top_p), f"filtered {name} k={top_k} p={top_p}")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [workloads.F32, workloads.BF16])
def test_cuda_filtered_misaligned_and_arbitrary_tokens(dtype):
    # Unaligned rows take the one-element-per-vector path (3 slices of
    # V = 5003); draft tokens drawn from the unfiltered draft are often outside the draft's
    # kept set (q = 0: accepted by the rule) or the target's (p = 0).
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b1_k4_v1024_f32", seed=32, B=12, V=5003, dtype=dtype)
    g = _run_filtered(w, 30, 0.8, misalign=True)
    check_chain(w, g, _oracle_filtered(w, 30, 0.8), f"filtered misaligned {dtype}")


@pytest.mark.gpu
def test_cuda_filtered_wide_unaligned_rows():
    # V = 140001 fp32 with unaligned rows: 69 slices of 2048 logits, more
    # group codes than one CTA holds, so each row streams through one CTA
    # with a running candidate threshold (and the heavy-tie case with it).
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b1_k4_v1024_f32", seed=39, B=3, k=2, V=140001)
    w["draft_tokens"] = _filtered_tokens(w, 40, 0.9, 39)
    g = _run_filtered(w, 40, 0.9, misalign=True)
    check_chain(w, g, _oracle_filtered(w, 40, 0.9), "filtered wide unaligned rows")
    rng = np.random.default_rng(39)
    w["target"] = rng.integers(0, 2, size=w["target"].shape).astype(np.float32)
    w["draft"] = (w["target"][:, :2] + rng.integers(0, 2, size=w["draft"].shape)).astype(np.float32)
    w["draft_tokens"] = _filtered_tokens(w, 40, 0.935, 39)
    g = _run_filtered(w, 40, 0.935, misalign=True)
    check_chain(w, g, _oracle_filtered(w, 40, 0.935), "filtered wide unaligned rows, ties")


@pytest.mark.gpu
@pytest.mark.parametrize("levels", [3, 1])
def test_cuda_filtered_ties(levels):
    # Logits on a few levels: thousands of equal values per slice force the
    # exact selection (ties broken by token index); one level = constant rows.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=33, B=4, k=3, V=40000)
    rng = np.random.default_rng(33)
    tgt = rng.integers(0, levels, size=(4, 4, 40000)).astype(np.float32)
    drf = tgt[:, :3] + rng.integers(0, 2, size=(4, 3, 40000)).astype(np.float32)
    w["target"] = workloads._store(tgt, w["dtype"])
    w["draft"] = workloads._store(drf, w["dtype"])
    # 100 equal kept logits: top_p = 0.935 cuts after 94 of them, clear of
    # the exact multiples of 1/100 where the cut itself would be a near tie.
    w["draft_tokens"] = _filtered_tokens(w, 100, 0.935, 33)
    g = _run_filtered(w, 100, 0.935)
    check_chain(w, g, _oracle_filtered(w, 100, 0.935), f"filtered ties levels={levels}")


@pytest.mark.gpu
def test_cuda_filtered_masked_vocab():
    # Most of each row is -inf (a constrained vocabulary): fewer finite logits
    # than top_k in some rows; -inf tokens carry no mass and are never drawn.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b1_k4_v1024_f32", seed=34, B=8, V=30000)
    rng = np.random.default_rng(34)
    for arr in (w["target"], w["draft"]):
        keep = rng.random(arr.shape) < 0.001
        keep[..., 7] = True
        arr[~keep] = -np.inf
    w["draft_tokens"] = _filtered_tokens(w, 64, 0.95, 34)
    g = _run_filtered(w, 64, 0.95)
    check_chain(w, g, _oracle_filtered(w, 64, 0.95), "filtered masked vocab")


@pytest.mark.gpu
def test_cuda_filtered_philox_and_ragged():
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=35, B=8, V=30000)
    B, k = w["B"], w["k"]
    rng = np.random.default_rng(35)
    seeds = rng.integers(0, 2**62, size=B, dtype=np.int64)
    offsets = rng.integers(0, 2**40, size=B, dtype=np.int64)
    w["uniforms"] = oracle.philox_uniforms(seeds.view(np.uint64), offsets.view(np.uint64), k + 1)
    w["draft_tokens"] = _filtered_tokens(w, 32, 0.9, 35)
    g = _run_filtered(w, 32, 0.9, philox=(seeds, offsets))
    check_chain(w, g, _oracle_filtered(w, 32, 0.9), "filtered philox")
    # Ragged: request b verified as the chain of its first k_b drafts, with
    # uniform column k_b for the final draw.
    lens = np.array([0, 1, 2, 3, 7, 5, 6, 4], np.int32)
    g = _run_filtered(w, 32, 0.9, philox=(seeds, offsets), draft_lens=lens)
    for b in range(B):
        kb = int(lens[b])
        sub = dict(w, B=1, k=kb, target=w["target"][b:b + 1, :kb + 1],
                   draft=w["draft"][b:b + 1, :kb] if kb else w["draft"][b:b + 1, :1],
                   draft_tokens=w["draft_tokens"][b:b + 1, :kb] if kb else w["draft_tokens"][b:b + 1, :1],
                   uniforms=np.concatenate([w["uniforms"][b, :kb], w["uniforms"][b, kb:kb + 1]])[None])
        if kb == 0:  # one draw from filtered target row 0 with uniform column 0
            p, tie = oracle.filtered_softmax(w["target"][b, 0], w["temperature"], 32,
                                             float(np.float32(0.9)), w["dtype"])
            tok, tie2 = oracle.inverse_cdf(p, float(w["uniforms"][b, 0]))
            assert g["num_accepted"][b] == 0
            if not (tie or tie2):
                assert g["tokens"][b, 0] == tok
            continue
        o = _oracle_filtered(sub, 32, 0.9)
        flagged = o["flags"][0].any()
        if not flagged:
            assert g["num_accepted"][b] == o["num_accepted"][0]
            assert np.array_equal(g["tokens"][b, :kb + 1], o["tokens"][0])
            assert (g["tokens"][b, kb + 1:] == -1).all()
        assert np.allclose(g["probs"][b, :kb], o["probs"][0], rtol=1e-5, atol=1e-30)
        assert np.isnan(g["probs"][b, kb:]).all()


@pytest.mark.gpu
def test_cuda_filtered_bad_token_fails_closed_and_workspace_stays_clean():
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import check_chain, run_chain
    ws = sv.Workspace()
    w = workloads.make("chain_b8_k4_v32000_f32", seed=36, B=6)
    w["draft_tokens"] = _filtered_tokens(w, 16, 0.9, 36)
    bad = dict(w, draft_tokens=w["draft_tokens"].copy())
    bad["draft_tokens"][2, 1] = w["V"] + 5
    g = _run_filtered(bad, 16, 0.9, workspace=ws)
    assert g["num_accepted"][2] == -1 and (g["tokens"][2] == -1).all()
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX
    assert sv.last_error(ws) == sv.SPEC_OK
    # The same workspace then serves a filtered call of other sizes, the
    # plain chain and the first call again, with unchanged results.
    w2 = workloads.make("chain_b64_k7_v128256_bf16", seed=37, B=3, V=50000)
    w2["draft_tokens"] = _filtered_tokens(w2, 64, 0.7, 37)
    g2 = _run_filtered(w2, 64, 0.7, workspace=ws)
    check_chain(w2, g2, _oracle_filtered(w2, 64, 0.7), "filtered after a failed call")
    run_chain(w, workspace=ws)
    again = _run_filtered(bad, 16, 0.9, workspace=ws)
    for key in ("tokens", "num_accepted"):
        assert np.array_equal(g[key], again[key]), key
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX


@pytest.mark.gpu
def test_cuda_filtered_full_size_sampled():
    # The 64-request, k = 7, V = 128256 bf16 workload with top_k = 50,
    # top_p = 0.9, in the launch configuration the benchmark times; the
    # oracle checks every fourth request.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=38)
    w["draft_tokens"] = _filtered_tokens(w, 50, 0.9, 38)
    g = _run_filtered(w, 50, 0.9)
    sel = np.arange(0, w["B"], 4)
    sub = dict(w, B=sel.size, target=w["target"][sel], draft=w["draft"][sel],
               draft_tokens=w["draft_tokens"][sel], uniforms=w["uniforms"][sel],
               seq_lens=w["seq_lens"][sel])
    gs = {key: g[key][sel] for key in g}
    check_chain(sub, gs, _oracle_filtered(sub, 50, 0.9), "filtered full size (sampled)",
                full_size="filtered")


def test_filtered_softmax_properties():
    # Against numpy's own ordering and exponential on random rows (with
    # repeated values): the kept set is the top_k by (logit desc, index asc)
    # cut to the shortest prefix reaching top_p; the kept sets nest as top_p
    # grows; p is the softmax of x / T restricted to the kept set.
    rng = np.random.default_rng(7)
    for trial in range(200):
        V = int(rng.integers(2, 60))
        x = rng.integers(-4, 5, size=V).astype(np.float32) * 0.5
        T = float(rng.choice([0.5, 1.0, 1.7]))
        K = int(rng.integers(1, V + 3))
        order = np.lexsort((np.arange(V), -x.astype(np.float64)))[: min(K, V)]
        prev = None
        for top_p in (0.3, 0.6, 0.9, 1.0):
            p, tie = oracle.filtered_softmax(x, T, K, float(np.float32(top_p)))
            kept = np.flatnonzero(p > 0)
            m = kept.size
            assert set(kept) == set(order[:m])          # a prefix of the order
            w = np.exp(x[order].astype(np.float64) / np.float64(np.float32(T)) -
                       x[order[0]] / np.float64(np.float32(T)))
            cum = np.cumsum(w / w.sum())
            if top_p < 1.0 and not tie:
                assert cum[m - 1] >= np.float32(top_p) - 1e-12
                assert m == 1 or cum[m - 2] < np.float32(top_p) + 1e-12
            else:
                assert top_p < 1.0 or m == min(K, V)
            ref = np.zeros(V)
            ref[order[:m]] = w[:m] / w[:m].sum()
            assert np.allclose(p, ref, rtol=1e-12, atol=1e-15)
            if prev is not None:
                assert set(prev) <= set(kept)
            prev = kept


@pytest.mark.gpu
def test_cuda_filtered_b256_full_size_sampled():
    # The 256-request, k = 3, V = 129280 bf16 workload with top_k = 20,
    # top_p = 0.95; the oracle checks every sixteenth request.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b256_k3_v129280_bf16", seed=40)
    sel = np.arange(0, w["B"], 16)
    x = w["draft_tokens"].copy()
    for b in sel:  # drafts from the filtered draft rows where the oracle checks
        sub = dict(w, B=1, draft=w["draft"][b:b + 1])
        x[b] = _filtered_tokens(sub, 20, 0.95, 40 + int(b))[0]
    w["draft_tokens"] = x
    g = _run_filtered(w, 20, 0.95)
    sub = dict(w, B=sel.size, target=w["target"][sel], draft=w["draft"][sel],
               draft_tokens=w["draft_tokens"][sel], uniforms=w["uniforms"][sel],
               seq_lens=w["seq_lens"][sel])
    gs = {key: g[key][sel] for key in g}
    check_chain(sub, gs, _oracle_filtered(sub, 20, 0.95), "filtered b256 full size (sampled)",
                full_size="filtered b256")


# ------------------------------------------------------------------ min_p, top-p without top-k
@pytest.mark.gpu
@pytest.mark.parametrize("top_k,top_p,min_p", [(50, 0.9, 0.05), (0, 1.0, 0.05), (0, 1.0, 0.03),
                                               (0, 0.9, 0.04), (8, 1.0, 0.3)])
def test_cuda_filtered_min_p(top_k, top_p, min_p):
    # min_p after top-k and top-p (kept lists), and min_p / top-p with no
    # top-k (per-row cuts)
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=41, B=6, V=60000)
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 41, min_p)
    g = _run_filtered(w, top_k, top_p, min_p=min_p)
    check_chain(w, g, _oracle_filtered(w, top_k, top_p, min_p), f"filtered top_k={top_k} top_p={top_p} min_p={min_p}")
