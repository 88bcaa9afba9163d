"""Seeded synthetic inputs for the speculative-decoding verification row.

This module is the only code shared by the CPU oracle tests and the CUDA path.
It holds none of the verification arithmetic: it makes random draws, rounds
stored logits from fp32 to bf16 (round-to-nearest-even), and picks the draft
tokens with the Gumbel-max trick, which is the drafter's job and sits outside
the verify step.

Workload recipes follow the shapes and value distributions of the pages'
workloads (the vLLM anatomy page, "Speculative Decoding"; the vLLM learning
book, section 2; the TensorRT-LLM walkthrough, rejection-sampling section and
EAGLE tree section of the TensorRT-LLM deployment page).  Real model logits are
not available, so Gaussian logits with peaked or Zipf-ranked biases stand in.

All draws use ``numpy.random.default_rng(seed)`` (PCG64) in a fixed order:
target -> bias/peaks -> draft noise -> draft-token Gumbel noise ->
accept/sample uniforms -> seq_lens.  Tree workloads draw
target -> tree shape -> child-token noise -> seq_lens.
"""
from __future__ import annotations

import numpy as np

F32 = "f32"
BF16 = "bf16"

# dtype codes of the C ABI (SPEC_F32 / SPEC_BF16)
DTYPE_CODE = {F32: 0, BF16: 1}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to fp32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def stored_as_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """The stored logits as fp32 values (exact for both storage types)."""
    return bf16_bits_to_f32(arr) if dtype == BF16 else np.asarray(arr, dtype=np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x) if dtype == BF16 else np.ascontiguousarray(x, dtype=np.float32)


def _gumbel_max_tokens(rng, logits_f32: np.ndarray, temperature: float) -> np.ndarray:
    """Draw one token per row of ``logits_f32 / temperature`` by the Gumbel-max trick.

    argmax(z + G) with G = -log(-log U) is an exact sample of softmax(z); it is
    the drafter's sampler and shares nothing with the verifier's inverse-CDF step.
    """
    rows, V = logits_f32.shape
    out = np.empty(rows, dtype=np.int32)
    for r in range(rows):
        u = rng.random(V, dtype=np.float64)
        u = np.maximum(u, np.finfo(np.float64).tiny)
        g = -np.log(-np.log(u))
        out[r] = int(np.argmax(logits_f32[r].astype(np.float64) / temperature + g))
    return out


def make_chain(*, B: int, k: int, V: int, dtype: str, temperature: float, seed: int,
               target_std: float, draft_noise_std: float, peaks: int = 0,
               peak_boost: float = 0.0, zipf_max: float = 0.0, zipf_s: float = 1.1,
               seq_len_range=(128, 2048), name: str = "chain") -> dict:
    """Chain workload: target logits [B,k+1,V], draft logits [B,k,V] and the rest.

    target ~ N(0, target_std^2) (+ ``peaks`` distinct ids per row raised by
    ``peak_boost``) (+ a Zipf-ranked bias ``zipf_max * r^-zipf_s`` over a random
    permutation of the vocabulary per row); draft = target[:, :k] + N(0,
    draft_noise_std^2), both rounded to the storage dtype after the additions;
    draft tokens are samples of softmax(stored draft / temperature); uniforms
    are U[0,1) of shape [B,k+1]; seq_lens uniform integers in ``seq_len_range``.
    """
    rng = np.random.default_rng(seed)
    tgt = rng.standard_normal((B, k + 1, V), dtype=np.float32)
    tgt *= np.float32(target_std)
    rows = tgt.reshape(B * (k + 1), V)
    if peaks > 0:
        for r in range(rows.shape[0]):
            ids = rng.choice(V, size=peaks, replace=False)
            rows[r, ids] += np.float32(peak_boost)
    if zipf_max > 0.0:
        ranks = np.arange(1, V + 1, dtype=np.float64)
        bias = (zipf_max * ranks ** (-zipf_s)).astype(np.float32)
        for r in range(rows.shape[0]):
            perm = rng.permutation(V)
            rows[r, perm] += bias
    noise = rng.standard_normal((B, k, V), dtype=np.float32)
    noise *= np.float32(draft_noise_std)
    drf = tgt[:, :k, :] + noise
    del noise
    target = _store(tgt, dtype)
    draft = _store(drf, dtype)
    del tgt, drf
    draft_f32 = stored_as_f32(draft, dtype).reshape(B * k, V)
    draft_tokens = _gumbel_max_tokens(rng, draft_f32, temperature).reshape(B, k)
    del draft_f32
    uniforms = rng.random((B, k + 1), dtype=np.float32)
    lo, hi = seq_len_range
    seq_lens = rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    return dict(kind="chain", name=name, dtype=dtype, B=B, k=k, V=V,
                temperature=float(temperature), target=target, draft=draft,
                draft_tokens=draft_tokens, uniforms=uniforms, seq_lens=seq_lens)


def _tree_shape(rng, N: int, depth: int, top_k: int, level_sizes):
    """Parent index per node for an EAGLE-style tree: node 0 is the root.

    Level 1 holds ``level_sizes[0]`` children of the root; every later level
    draws each node's parent uniformly from the previous level among parents
    that still have fewer than ``top_k`` children.  Nodes are numbered level by
    level, and within a level in order of their parent.
    """
    assert sum(level_sizes) + 1 == N and len(level_sizes) == depth
    parent = [-1]
    prev = [0]
    nxt_id = 1
    for lvl, size in enumerate(level_sizes):
        counts = {p: 0 for p in prev}
        chosen = []
        for _ in range(size):
            open_ = [p for p in prev if counts[p] < top_k]
            p = open_[int(rng.integers(0, len(open_)))]
            counts[p] += 1
            chosen.append(p)
        chosen.sort()
        cur = []
        for p in chosen:
            parent.append(p)
            cur.append(nxt_id)
            nxt_id += 1
        prev = cur
    return np.asarray(parent, dtype=np.int64)


def make_tree(*, B: int, N: int, L: int, V: int, dtype: str, seed: int, target_std: float,
              top_k: int = 8, level_sizes=None, child_noise_std: float = 1.0,
              seq_len_range=(256, 4096), temperature: float = 0.5, name: str = "tree") -> dict:
    """EAGLE-style tree workload: target [B,N,V], tree_tokens [B,N], paths [B,N,L].

    Node 0 is the root (the last committed token); target row n is the
    distribution after node n.  The tokens of node n's c children are the top-c
    ids of target[b,n] + N(0, child_noise_std^2), so siblings are distinct.
    ``paths`` has one root-to-leaf row per leaf, -1 padded, then all-(-1) rows.
    For the stochastic tree verify, uniforms [B,N] U[0,1) (column n >= 1:
    node n's accept test, column 0: the final draw) are drawn last, and
    ``temperature`` is the softmax temperature of the target rows.
    """
    depth = L - 1
    if level_sizes is None:
        first = min(top_k, N - 1)
        rest = N - 1 - first
        level_sizes = [first] + [rest // (depth - 1) + (1 if i < rest % (depth - 1) else 0)
                                 for i in range(depth - 1)] if depth > 1 else [first]
    rng = np.random.default_rng(seed)
    tgt = rng.standard_normal((B, N, V), dtype=np.float32)
    tgt *= np.float32(target_std)
    target = _store(tgt, dtype)
    tgt_stored = stored_as_f32(target, dtype)
    del tgt
    tree_tokens = np.zeros((B, N), dtype=np.int32)
    paths = np.full((B, N, L), -1, dtype=np.int32)
    parents = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        parent = _tree_shape(rng, N, depth, top_k, level_sizes)
        parents[b] = parent
        children = {n: [] for n in range(N)}
        for n in range(1, N):
            children[int(parent[n])].append(n)
        tree_tokens[b, 0] = int(rng.integers(0, V))
        for n in range(N):
            ch = children[n]
            if not ch:
                continue
            noisy = tgt_stored[b, n].astype(np.float64) + child_noise_std * rng.standard_normal(V)
            top = np.argpartition(-noisy, len(ch) - 1)[: len(ch)]
            top = top[np.argsort(-noisy[top], kind="stable")]
            for c, tok in zip(ch, top):
                tree_tokens[b, c] = int(tok)
        leaves = [n for n in range(N) if not children[n]]
        for pi, leaf in enumerate(leaves):
            chain = [leaf]
            while chain[-1] != 0:
                chain.append(int(parent[chain[-1]]))
            chain.reverse()
            paths[b, pi, : len(chain)] = chain
    lo, hi = seq_len_range
    seq_lens = rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)
    uniforms = rng.random((B, N), dtype=np.float32)
    return dict(kind="tree", name=name, dtype=dtype, B=B, N=N, P=N, L=L, V=V,
                target=target, tree_tokens=tree_tokens, paths=paths, parents=parents,
                seq_lens=seq_lens, uniforms=uniforms, temperature=float(temperature))


# Named workloads (shapes and distributions of the pages' configurations).
CONFIGS = {
    # chain stochastic, B=1 k=4 V=1024 fp32, T=1.0
    "chain_b1_k4_v1024_f32": dict(
        kind="chain", B=1, k=4, V=1024, dtype=F32, temperature=1.0,
        target_std=2.0, draft_noise_std=0.5),
    # chain greedy + stochastic at T=0.8, B=8 k=4 V=32000 fp32, 5 peaks +8.0
    "chain_b8_k4_v32000_f32": dict(
        kind="chain", B=8, k=4, V=32000, dtype=F32, temperature=0.8,
        target_std=3.0, draft_noise_std=1.0, peaks=5, peak_boost=8.0,
        seq_len_range=(128, 2048)),
    # chain stochastic, B=64 k=7 V=128256 bf16, Zipf(1.1) bias up to +6, T=0.7
    "chain_b64_k7_v128256_bf16": dict(
        kind="chain", B=64, k=7, V=128256, dtype=BF16, temperature=0.7,
        target_std=2.5, draft_noise_std=0.7, zipf_max=6.0, zipf_s=1.1),
    # tree greedy (and stochastic at T=0.25), B=16 N=60 L=4 V=151936 bf16, topK=8, depth 3
    "tree_b16_n60_l4_v151936_bf16": dict(
        kind="tree", B=16, N=60, L=4, V=151936, dtype=BF16, target_std=2.0,
        top_k=8, level_sizes=[8, 25, 26], temperature=0.25),
    # MTP-style chain stochastic, B=256 k=3 V=129280 bf16, 3 peaks +7.0, T=1.0
    "chain_b256_k3_v129280_bf16": dict(
        kind="chain", B=256, k=3, V=129280, dtype=BF16, temperature=1.0,
        target_std=2.0, draft_noise_std=1.2, peaks=3, peak_boost=7.0,
        seq_len_range=(512, 8192)),
}

# The headline workload of the benchmark.
HEADLINE = "chain_b64_k7_v128256_bf16"


def make(name: str, seed: int = 0, **overrides) -> dict:
    """Build a named workload (``CONFIGS``) with optional size overrides."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    kind = cfg.pop("kind")
    if kind == "chain":
        return make_chain(seed=seed, name=name, **cfg)
    return make_tree(seed=seed, name=name, **cfg)


def algorithmic_bytes(w: dict, greedy: bool = False) -> int:
    """Logit bytes one verify call must read once (the roofline numerator)."""
    es = 2 if w["dtype"] == BF16 else 4
    if w["kind"] == "tree":
        return w["B"] * w["N"] * w["V"] * es
    rows = w["B"] * (w["k"] + 1) if greedy else w["B"] * (2 * w["k"] + 1)
    return rows * w["V"] * es
