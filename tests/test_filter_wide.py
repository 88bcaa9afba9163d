"""Filtered chain verify with kept sets of any size (TensorRT-LLM walkthrough,
rejection-sampling section: target and draft filtered alike by temperature,
top-k, top-p and min_p): top-p or min_p without top-k and top-k above the
kept-list size take per-row cuts (mass histogram, candidate list, radix
selection).  The CUDA path against the oracle, exact outside its flagged
near-ties."""
import numpy as np
import pytest

import oracle
import workloads
from test_filter import _filtered_tokens, _oracle_filtered, _run_filtered

pytestmark = pytest.mark.gpu


def _kept_sizes(w, top_k, top_p, min_p=0.0):
    return [int((oracle.filtered_softmax(w["target"][b, i], w["temperature"], top_k,
                                         float(np.float32(top_p)), w["dtype"],
                                         min_p=float(np.float32(min_p)))[0] > 0).sum())
            for b in range(w["B"]) for i in range(w["k"] + 1)]


WIDE_CASES = [
    # (workload, overrides, top_k, top_p, min_p)
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 0, 0.9, 0.0),      # ~1000 kept per row
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 0, 0.99, 0.0),     # ~10^4 kept
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 1000, 1.0, 0.0),   # top-k above the lists
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 300, 0.95, 0.0),   # top-k, then top-p in it
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 5000, 0.9, 1e-3),  # all three filters
    ("chain_b64_k7_v128256_bf16", dict(B=4, V=70000), 0, 0.9, 0.01),     # min_p cuts inside top-p
    ("chain_b8_k4_v32000_f32", dict(B=6), 0, 0.5, 0.0),                  # fp32, 16-byte vectors
    ("chain_b8_k4_v32000_f32", dict(B=4, V=30011), 0, 0.8, 0.0),         # fp32, one element per vector
    ("chain_b1_k4_v1024_f32", dict(B=16), 0, 0.9, 0.0),                  # one slice per row
    ("chain_b1_k4_v1024_f32", dict(B=16), 2000, 0.7, 0.0),               # top_k >= V: top-p alone
    ("chain_b256_k3_v129280_bf16", dict(B=8, V=40000), 0, 0.8, 0.0),
    ("chain_b64_k7_v128256_bf16", dict(B=1, k=2, V=1000003), 0, 0.9, 0.0),  # 1M unaligned logits
]


@pytest.mark.parametrize("name,over,top_k,top_p,min_p", WIDE_CASES)
def test_cuda_wide_filter_matches_oracle(name, over, top_k, top_p, min_p):
    from test_gpu_parity import check_chain
    w = workloads.make(name, seed=51, **over)
    sizes = _kept_sizes(w, top_k, top_p, min_p)
    if top_k == 0 and min_p == 0.0 and top_p >= 0.9 and w["V"] >= 30000:
        assert max(sizes) > 256, sizes  # beyond any explicit kept list
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 51, min_p)
    g = _run_filtered(w, top_k, top_p, min_p=min_p)
    check_chain(w, g, _oracle_filtered(w, top_k, top_p, min_p),
                f"wide {name} top_k={top_k} top_p={top_p} min_p={min_p}")


@pytest.mark.parametrize("V,levels,top_k,top_p", [(40000, 1, 0, 0.93513), (40000, 3, 0, 0.93513),
                                                  (3000, 1, 0, 0.71113), (40000, 1, 1500, 1.0),
                                                  (40000, 2, 20000, 0.61117)])
def test_cuda_wide_filter_ties(V, levels, top_k, top_p):
    # Logits on a few levels (one level: constant rows): the cut falls inside
    # a run of thousands of equal logits and is decided by token index.  The
    # crossing bin then holds more tokens than the candidate list (V = 40000:
    # each row rescans itself) or than the staging buffer (V = 3000).
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=52, B=3, k=3, V=V)
    rng = np.random.default_rng(52)
    tgt = rng.integers(0, levels, size=(3, 4, V)).astype(np.float32)
    drf = tgt[:, :3] + rng.integers(0, 2, size=(3, 3, V)).astype(np.float32)
    w["target"] = workloads._store(tgt, w["dtype"])
    w["draft"] = workloads._store(drf, w["dtype"])
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 52)
    o = _oracle_filtered(w, top_k, top_p)
    g = _run_filtered(w, top_k, top_p)
    check_chain(w, g, o, f"wide ties V={V} levels={levels} top_k={top_k} top_p={top_p}")
    assert not o["flags"].all(), "every decision flagged: the case checks nothing"


@pytest.mark.parametrize("V,top_k,top_p", [(40000, 0, 0.93513), (3000, 0, 0.71113), (30000, 700, 0.9)])
def test_cuda_wide_filter_leaves_the_workspace_zero(V, top_k, top_p):
    # Every call returns its histograms, candidate lists, row records and
    # statistics words to zero (another call's layout may place its own
    # statistics there): constant rows (the crossing bin holds every token:
    # the row rescans itself, or its list is not staged) and ordinary rows.
    import torch
    import speculative_decoding_verification_row_gb300 as sv
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=59, B=2, k=2, V=V)
    if top_k == 0:
        w["target"][:] = w["target"][..., :1]
        w["draft"][:] = w["draft"][..., :1]
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 59)
    ws = sv.Workspace()
    _run_filtered(w, top_k, top_p, workspace=ws)
    buf = ws.buf.cpu().numpy()
    nz = np.flatnonzero(buf[256:])
    assert nz.size == 0, f"{nz.size} nonzero workspace bytes after the call, first at {256 + nz[0]}"
    torch.cuda.synchronize()


@pytest.mark.parametrize("T,top_k,top_p,min_p", [(0.7, 0, 1.0, 0.999), (1.5, 0, 0.95, 0.0), (0.05, 0, 0.9, 0.0),
                                                  (5.0, 0, 0.9, 0.0), (5.0, 3000, 0.95, 0.01),
                                                  (1.0, 0, float(np.nextafter(np.float32(1), np.float32(0))), 0.0)])
def test_cuda_wide_filter_edge_parameters(T, top_k, top_p, min_p):
    # min_p near 1 keeps the maxima only; a very low temperature (a few
    # tokens hold the mass) and high ones (flat rows: tens of thousands of
    # tokens kept, the tail bound deep in the row); top_p one float below 1
    # (the a-priori tail bound, (1 - top_p) Z / 2, is then within the
    # rounding of the row's total; a row whose cut the bound does not place
    # is binned token by token).
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=60, B=4, V=50000)
    w["temperature"] = T
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 60, min_p)
    g = _run_filtered(w, top_k, top_p, min_p=min_p)
    check_chain(w, g, _oracle_filtered(w, top_k, top_p, min_p), f"wide edge T={T} {top_k} {top_p} {min_p}")


def test_cuda_wide_filter_masked_vocab():
    # Most of each row is -inf: top_k above the finite count, and top-p over
    # the finite tokens; -inf tokens carry no mass and are never drawn.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b1_k4_v1024_f32", seed=53, B=8, V=30000)
    rng = np.random.default_rng(53)
    for arr in (w["target"], w["draft"]):
        keep = rng.random(arr.shape) < 0.01
        keep[..., 7] = True
        arr[~keep] = -np.inf
    for top_k, top_p in ((5000, 0.95), (0, 0.9), (400, 1.0)):
        w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 53)
        g = _run_filtered(w, top_k, top_p)
        check_chain(w, g, _oracle_filtered(w, top_k, top_p), f"wide masked vocab {top_k} {top_p}")


def test_cuda_wide_filter_philox_and_ragged():
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=54, B=8, V=30000)
    B, k = w["B"], w["k"]
    rng = np.random.default_rng(54)
    seeds = rng.integers(0, 2**62, size=B, dtype=np.int64)
    offsets = rng.integers(0, 2**40, size=B, dtype=np.int64)
    w["uniforms"] = oracle.philox_uniforms(seeds.view(np.uint64), offsets.view(np.uint64), k + 1)
    w["draft_tokens"] = _filtered_tokens(w, 0, 0.9, 54)
    g = _run_filtered(w, 0, 0.9, philox=(seeds, offsets))
    check_chain(w, g, _oracle_filtered(w, 0, 0.9), "wide philox")
    lens = np.array([0, 1, 2, 3, 7, 5, 6, 4], np.int32)
    g = _run_filtered(w, 0, 0.9, philox=(seeds, offsets), draft_lens=lens)
    for b in range(B):
        kb = int(lens[b])
        if kb == 0:  # one draw from filtered target row 0 with uniform column 0
            p, tie = oracle.filtered_softmax(w["target"][b, 0], w["temperature"], 0,
                                             float(np.float32(0.9)), w["dtype"])
            tok, tie2 = oracle.inverse_cdf(p, float(w["uniforms"][b, 0]))
            assert g["num_accepted"][b] == 0
            if not (tie or tie2):
                assert g["tokens"][b, 0] == tok
            continue
        sub = dict(w, B=1, k=kb, target=w["target"][b:b + 1, :kb + 1], draft=w["draft"][b:b + 1, :kb],
                   draft_tokens=w["draft_tokens"][b:b + 1, :kb],
                   uniforms=np.concatenate([w["uniforms"][b, :kb], w["uniforms"][b, kb:kb + 1]])[None])
        o = _oracle_filtered(sub, 0, 0.9)
        if not o["flags"][0].any():
            assert g["num_accepted"][b] == o["num_accepted"][0]
            assert np.array_equal(g["tokens"][b, :kb + 1], o["tokens"][0])
            assert (g["tokens"][b, kb + 1:] == -1).all()
        assert np.allclose(g["probs"][b, :kb], o["probs"][0], rtol=1e-5, atol=1e-30)
        assert np.isnan(g["probs"][b, kb:]).all()


def test_cuda_wide_filter_bad_token_and_workspace_reuse():
    # A bad draft token fails its request closed; the same workspace then
    # serves kept-list, per-cut and unfiltered calls of other sizes, and the
    # first call again, with unchanged results (every call leaves the
    # histograms, counters and statistics words zero).
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import check_chain, run_chain
    ws = sv.Workspace()
    w = workloads.make("chain_b8_k4_v32000_f32", seed=55, B=6)
    w["draft_tokens"] = _filtered_tokens(w, 0, 0.8, 55)
    bad = dict(w, draft_tokens=w["draft_tokens"].copy())
    bad["draft_tokens"][2, 1] = -3
    g = _run_filtered(bad, 0, 0.8, workspace=ws)
    assert g["num_accepted"][2] == -1 and (g["tokens"][2] == -1).all()
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX
    assert sv.last_error(ws) == sv.SPEC_OK
    keep = [b for b in range(6) if b != 2]
    o = _oracle_filtered(w, 0, 0.8)
    sub = {key: (v[keep] if isinstance(v, np.ndarray) and v.shape[:1] == (6,) else v) for key, v in w.items()}
    sub["B"] = len(keep)
    check_chain(sub, {key: v[keep] for key, v in g.items()},
                {key: (v[keep] if isinstance(v, np.ndarray) else v) for key, v in o.items()},
                "wide filter: the other requests")
    w2 = workloads.make("chain_b64_k7_v128256_bf16", seed=56, B=3, V=50000)
    for top_k, top_p in ((64, 0.7), (700, 0.9), (0, 0.95)):
        w2["draft_tokens"] = _filtered_tokens(w2, top_k, top_p, 56)
        g2 = _run_filtered(w2, top_k, top_p, workspace=ws)
        check_chain(w2, g2, _oracle_filtered(w2, top_k, top_p), f"after a failed call {top_k} {top_p}")
    run_chain(w, workspace=ws)
    again = _run_filtered(bad, 0, 0.8, workspace=ws)
    for key in ("tokens", "num_accepted"):
        assert np.array_equal(g[key], again[key]), key
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX


def test_cuda_wide_filter_full_size_sampled():
    # The 64-request, k = 7, V = 128256 bf16 workload with top-p 0.9 and no
    # top-k (kept sets of ~600 to ~2300 tokens), in the launch configuration
    # the benchmark times; the oracle checks every fourth request.
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=57)
    sel = np.arange(0, w["B"], 4)
    x = w["draft_tokens"].copy()
    for b in sel:
        sub = dict(w, B=1, draft=w["draft"][b:b + 1])
        x[b] = _filtered_tokens(sub, 0, 0.9, 57 + int(b))[0]
    w["draft_tokens"] = x
    g = _run_filtered(w, 0, 0.9)
    sub = dict(w, B=sel.size, target=w["target"][sel], draft=w["draft"][sel],
               draft_tokens=w["draft_tokens"][sel], uniforms=w["uniforms"][sel],
               seq_lens=w["seq_lens"][sel])
    check_chain(sub, {key: g[key][sel] for key in g}, _oracle_filtered(sub, 0, 0.9),
                "wide filter full size (sampled)", full_size="wide top-p")


def test_cuda_wide_filter_b256_full_size_sampled():
    # The 256-request, k = 3, V = 129280 bf16 workload with top-p 0.7 and no
    # top-k (kept sets of ~9000 tokens); every sixteenth request checked.
    # (At top-p 0.95 the cut falls among tokens of probability ~2e-6, so the
    # oracle flags ~90 % of these rows as near ties and the case checks
    # little.)
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b256_k3_v129280_bf16", seed=58)
    sel = np.arange(0, w["B"], 16)
    x = w["draft_tokens"].copy()
    for b in sel:
        sub = dict(w, B=1, draft=w["draft"][b:b + 1])
        x[b] = _filtered_tokens(sub, 0, 0.7, 58 + int(b))[0]
    w["draft_tokens"] = x
    g = _run_filtered(w, 0, 0.7)
    sub = dict(w, B=sel.size, target=w["target"][sel], draft=w["draft"][sel],
               draft_tokens=w["draft_tokens"][sel], uniforms=w["uniforms"][sel],
               seq_lens=w["seq_lens"][sel])
    check_chain(sub, {key: g[key][sel] for key in g}, _oracle_filtered(sub, 0, 0.7),
                "wide filter b256 full size (sampled)", full_size="wide top-p b256")


def _misleading_rows(w, ntop, seed):
    """Rows whose first 2048 logits of every 16384 (each slice's sample, for
    bf16 rows of a multiple of 16384) hold `ntop` tokens at the top and
    nothing else of weight, while the rest of the row carries most of the
    mass a little lower: a depth estimated from those 2048 falls far above
    the cut, so the exact check must send the row to the rebuild."""
    rng = np.random.default_rng(seed)
    B, k, V = w["B"], w["k"], w["V"]
    tgt = (-3.0 + 0.5 * rng.standard_normal((B, k + 1, V))).astype(np.float32)
    for s in range(0, V, 16384):
        hi = min(V, s + 2048)
        tgt[..., s:hi] = -60.0
        for b in range(B):
            for r in range(k + 1):
                pos = s + rng.choice(hi - s, size=min(ntop, hi - s), replace=False)
                tgt[b, r, pos] = (0.1 * rng.standard_normal(pos.size)).astype(np.float32)
    drf = tgt[:, :k] + (0.3 * rng.standard_normal((B, k, V))).astype(np.float32)
    w["target"] = workloads.f32_to_bf16_bits(tgt)
    w["draft"] = workloads.f32_to_bf16_bits(drf)
    w["temperature"] = 1.0


@pytest.mark.parametrize("V,ntop,top_k,top_p", [(49152, 40, 0, 0.9), (49152, 250, 1000, 0.95),
                                                (16384, 40, 0, 0.9), (16384, 450, 1000, 0.95)])
def test_cuda_wide_filter_misleading_sample(V, ntop, top_k, top_p):
    # The histogram grid bins only the tokens above a light depth each CTA
    # estimates from a sample of its first slice; the bins step checks
    # exactly that the cut lies above the row's shallowest such depth and
    # otherwise rebuilds the row's histogram with the a-priori depth (or
    # every token counted, for top-k).  These rows take that path: in the
    # bins grid (three slices, several histogram CTAs per row) and in the
    # histogram CTA itself (one slice: the CTA holds the whole row).
    from test_gpu_parity import check_chain
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=63, B=3, V=V)
    _misleading_rows(w, ntop, 63)
    w["draft_tokens"] = _filtered_tokens(w, top_k, top_p, 63)
    g = _run_filtered(w, top_k, top_p)
    check_chain(w, g, _oracle_filtered(w, top_k, top_p), f"wide misleading sample V={V} {ntop} {top_k} {top_p}")
