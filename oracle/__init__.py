"""CPU oracle for the speculative-decoding verification row (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never does.  The arithmetic lives in ``spec_oracle.c`` (plain C,
double precision, single-threaded); this module compiles it with gcc on first
use and exposes numpy-friendly wrappers through ctypes.

Each wrapper names the passage it follows in the C source header.  Pins that
tie the oracle to the pages and to mathematics (closed forms, exact enumerated
distributions, a chi-square test, library special cases, brute force) are in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spec_oracle.c")
LIB = os.path.join(HERE, "libspec_oracle.so")

OK, EINVAL, EBADINDEX = 0, -1, -2
ACCEPT_TIE = 1e-5   # |r - p/q| window of a flagged accept test
SAMPLE_TIE = 1e-6   # window (in units of Z) of a flagged final sample
DTYPE_CODE = {"f32": 0, "bf16": 1}

_lock = threading.Lock()
_lib = None


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compile the oracle C source into a shared library (gcc, -O2, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_softmax.argtypes = [P, I, ctypes.c_double, I, P]
    lib.oracle_inverse_cdf.argtypes = [P, I, ctypes.c_double, ctypes.c_double, P]
    lib.oracle_argmax.argtypes = [P, I, I]
    lib.oracle_verify_chain.argtypes = [P, P, I, P, P, P, ctypes.c_float, I, I, I, P, P, P, P]
    lib.oracle_verify_greedy.argtypes = [P, I, P, P, I, I, I, P, P]
    lib.oracle_rollback_paged.argtypes = [P, P, P, I, P, I, I, P, P, P]
    lib.oracle_filtered_softmax.argtypes = [P, I, ctypes.c_double, I, I, ctypes.c_double, P, P]
    lib.oracle_filter_row.argtypes = [P, I, ctypes.c_double, I, I, ctypes.c_double, ctypes.c_double,
                                      P, P]
    lib.oracle_verify_chain_filtered.argtypes = [P, P, I, P, P, ctypes.c_float, I, ctypes.c_double,
                                                 ctypes.c_double, I, I, I, P, P, P, P]
    lib.oracle_verify_tree.argtypes = [P, I, P, P, I, I, I, I, I, P, P, P, P]
    lib.oracle_rollback.argtypes = [P, P, I, I, P, P]
    lib.oracle_verify_tree_sampled.argtypes = [P, I, P, P, P, ctypes.c_float, I, I, I, I, I,
                                               P, P, P, P, P]
    lib.oracle_philox4x32_10.argtypes = [P, P, P]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_philox_uniforms.argtypes = [P, P, I, I, P]
    for f in ("oracle_softmax", "oracle_inverse_cdf", "oracle_argmax", "oracle_verify_chain",
              "oracle_verify_greedy", "oracle_verify_tree", "oracle_rollback",
              "oracle_philox_uniforms", "oracle_rollback_paged", "oracle_filtered_softmax",
              "oracle_verify_chain_filtered", "oracle_verify_tree_sampled", "oracle_filter_row"):
        getattr(lib, f).restype = I
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _logits(a, dtype: str):
    return _c(a, np.uint16 if dtype == "bf16" else np.float32)


def softmax(x, temperature: float, dtype: str = "f32", lib=None) -> np.ndarray:
    """softmax(x / T) in double (vLLM learning book, section 2).

    T is rounded to float32 first, as the verify calls take it."""
    lib = lib or load()
    x = _logits(x, dtype)
    p = np.empty(x.shape[-1], dtype=np.float64)
    rc = lib.oracle_softmax(_ptr(x), DTYPE_CODE[dtype], float(np.float32(temperature)),
                            x.shape[-1], _ptr(p))
    if rc != OK:
        raise ValueError(f"oracle_softmax rc={rc}")
    return p


def inverse_cdf(w, u: float, tol: float = SAMPLE_TIE, lib=None):
    """(token, near_tie) of the inverse-CDF draw from weights ``w`` at uniform ``u``."""
    lib = lib or load()
    w = _c(w, np.float64)
    tie = np.zeros(1, dtype=np.int32)
    t = lib.oracle_inverse_cdf(_ptr(w), w.shape[0], float(u), float(tol), _ptr(tie))
    return int(t), bool(tie[0])


def argmax(x, dtype: str = "f32", lib=None) -> int:
    lib = lib or load()
    x = _logits(x, dtype)
    return int(lib.oracle_argmax(_ptr(x), DTYPE_CODE[dtype], x.shape[-1]))


def verify_chain(target, draft, draft_tokens, uniforms, temperature: float, dtype: str = "f32",
                 lib=None, draft_lens=None) -> dict:
    """Chain rejection-sampling verify (vLLM anatomy page, "Speculative Decoding").

    target [B,k+1,V], draft [B,k,V] (fp32 values or raw bf16 bits),
    draft_tokens int [B,k], uniforms float32 [B,k+1].  Returns a dict with
    tokens [B,k+1], num_accepted [B], probs [B,k,2] (p_i(x_i), q_i(x_i)),
    flags [B,k+1] and the return code.  draft_lens (int [B], optional): each
    request's real draft length k_b <= k (ragged verify).
    """
    lib = lib or load()
    target = _logits(target, dtype)
    draft = _logits(draft, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    assert draft.shape == (B, k, V)
    x = _c(draft_tokens, np.int32)
    r = _c(uniforms, np.float32)
    assert x.shape == (B, k) and r.shape == (B, k + 1)
    tokens = np.empty((B, k + 1), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    probs = np.empty((B, k, 2), dtype=np.float64)
    flags = np.empty((B, k + 1), dtype=np.int32)
    lens = None if draft_lens is None else _c(draft_lens, np.int32)
    rc = lib.oracle_verify_chain(_ptr(target), _ptr(draft), DTYPE_CODE[dtype], _ptr(x), _ptr(r),
                                 None if lens is None else _ptr(lens), float(temperature), B, k, V,
                                 _ptr(tokens), _ptr(n_acc), _ptr(probs), _ptr(flags))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_verify_chain rc={rc}")
    return dict(tokens=tokens, num_accepted=n_acc, probs=probs, flags=flags, rc=rc)


def filtered_softmax(x, temperature: float, top_k: int, top_p: float = 1.0, dtype: str = "f32",
                     lib=None, min_p: float = 0.0):
    """(p, near_tie): softmax(x / T) restricted to the top_k tokens by (logit
    descending, index ascending; top_k = 0: all), then to the shortest prefix
    reaching top_p, then to the tokens whose probability is at least min_p
    times the largest (TensorRT-LLM walkthrough, rejection-sampling section)."""
    lib = lib or load()
    x = _logits(x, dtype)
    p = np.empty(x.shape[-1], dtype=np.float64)
    tie = np.zeros(1, dtype=np.int32)
    rc = lib.oracle_filter_row(_ptr(x), DTYPE_CODE[dtype], float(np.float32(temperature)),
                               x.shape[-1], int(top_k), float(top_p), float(min_p), _ptr(p), _ptr(tie))
    if rc != OK:
        raise ValueError(f"oracle_filtered_softmax rc={rc}")
    return p, bool(tie[0])


def verify_chain_filtered(target, draft, draft_tokens, uniforms, temperature: float, top_k: int,
                          top_p: float = 1.0, dtype: str = "f32", lib=None, min_p: float = 0.0) -> dict:
    """verify_chain on top-k / top-p / min_p filtered target and draft rows."""
    lib = lib or load()
    target = _logits(target, dtype)
    draft = _logits(draft, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    x = _c(draft_tokens, np.int32)
    r = _c(uniforms, np.float32)
    tokens = np.empty((B, k + 1), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    probs = np.empty((B, k, 2), dtype=np.float64)
    flags = np.empty((B, k + 1), dtype=np.int32)
    rc = lib.oracle_verify_chain_filtered(_ptr(target), _ptr(draft), DTYPE_CODE[dtype], _ptr(x), _ptr(r),
                                          float(temperature), int(top_k), float(top_p), float(min_p), B, k, V,
                                          _ptr(tokens), _ptr(n_acc), _ptr(probs), _ptr(flags))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_verify_chain_filtered rc={rc}")
    return dict(tokens=tokens, num_accepted=n_acc, probs=probs, flags=flags, rc=rc)


def verify_greedy(target, draft_tokens, dtype: str = "f32", lib=None, draft_lens=None) -> dict:
    """Greedy chain verify (Kestrel article, section 3.3); draft_lens as for verify_chain."""
    lib = lib or load()
    target = _logits(target, dtype)
    B, k1, V = target.shape
    k = k1 - 1
    d = _c(draft_tokens, np.int32)
    assert d.shape == (B, k)
    tokens = np.empty((B, k + 1), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    lens = None if draft_lens is None else _c(draft_lens, np.int32)
    rc = lib.oracle_verify_greedy(_ptr(target), DTYPE_CODE[dtype], _ptr(d),
                                  None if lens is None else _ptr(lens), B, k, V,
                                  _ptr(tokens), _ptr(n_acc))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_verify_greedy rc={rc}")
    return dict(tokens=tokens, num_accepted=n_acc, rc=rc)


def verify_tree(target, tree_tokens, paths, dtype: str = "f32", lib=None) -> dict:
    """Greedy tree verify (TensorRT-LLM deployment page, "Eagle-2" section)."""
    lib = lib or load()
    target = _logits(target, dtype)
    B, N, V = target.shape
    tok = _c(tree_tokens, np.int32)
    pth = _c(paths, np.int32)
    _, P, L = pth.shape
    assert tok.shape == (B, N) and pth.shape[0] == B
    tokens = np.empty((B, L), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    best = np.empty(B, dtype=np.int32)
    nodes = np.empty((B, L), dtype=np.int32)
    rc = lib.oracle_verify_tree(_ptr(target), DTYPE_CODE[dtype], _ptr(tok), _ptr(pth), B, N, P, L,
                                V, _ptr(tokens), _ptr(n_acc), _ptr(best), _ptr(nodes))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_verify_tree rc={rc}")
    return dict(tokens=tokens, num_accepted=n_acc, best_path=best, accepted_nodes=nodes, rc=rc)


def verify_tree_sampled(target, tree_tokens, paths, uniforms, temperature: float,
                        dtype: str = "f32", lib=None) -> dict:
    """Stochastic tree verify (TensorRT-LLM deployment page, tree verification
    by rejection sampling; children are point-mass proposals): target [B,N,V],
    tree_tokens [B,N], paths [B,P,L], uniforms float32 [B,N] (column n >= 1 is
    node n's accept test, column 0 the final draw).  Returns tokens [B,L],
    num_accepted [B], best_path [B], accepted_nodes [B,L], flags [B,N], rc."""
    lib = lib or load()
    target = _logits(target, dtype)
    B, N, V = target.shape
    tok = _c(tree_tokens, np.int32)
    pth = _c(paths, np.int32)
    _, P, L = pth.shape
    u = _c(uniforms, np.float32)
    assert tok.shape == (B, N) and u.shape == (B, N) and pth.shape[0] == B
    tokens = np.empty((B, L), dtype=np.int32)
    n_acc = np.empty(B, dtype=np.int32)
    best = np.empty(B, dtype=np.int32)
    nodes = np.empty((B, L), dtype=np.int32)
    flags = np.empty((B, N), dtype=np.int32)
    rc = lib.oracle_verify_tree_sampled(_ptr(target), DTYPE_CODE[dtype], _ptr(tok), _ptr(pth), _ptr(u),
                                        float(temperature), B, N, P, L, V, _ptr(tokens), _ptr(n_acc),
                                        _ptr(best), _ptr(nodes), _ptr(flags))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_verify_tree_sampled rc={rc}")
    return dict(tokens=tokens, num_accepted=n_acc, best_path=best, accepted_nodes=nodes, flags=flags,
                rc=rc)


def rollback(old_lens, num_accepted, k: int, lib=None) -> dict:
    """KV cursor rollback (TensorRT-LLM walkthrough, update_requests / rewind_cache)."""
    lib = lib or load()
    old = _c(old_lens, np.int32)
    n = _c(num_accepted, np.int32)
    B = old.shape[0]
    new = np.empty(B, dtype=np.int32)
    rew = np.empty(B, dtype=np.int32)
    rc = lib.oracle_rollback(_ptr(old), _ptr(n), int(k), B, _ptr(new), _ptr(rew))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_rollback rc={rc}")
    return dict(new_lens=new, rewind_lens=rew, rc=rc)


def relocate_kv(pool, block_tables, base_lens, accepted_nodes, num_accepted,
                tokens_per_block: int):
    """Accepted-KV relocation (TensorRT-LLM walkthrough, the "moving to the
    right place" step, _update_kv_cache_draft_token_location): returns a copy
    of ``pool`` [rows, ...] in which, for every request b with 0 < n < L whose
    path starts at node 0 with strictly increasing nodes, all rows mapped, the
    row at logical position base + j becomes the ORIGINAL row at base +
    accepted_nodes[b, j] for j = 1..n.  Logical position t of request b is pool
    row block_tables[b, t // tpb] * tpb + t % tpb."""
    pool = np.asarray(pool)
    bt = np.asarray(block_tables)
    base = np.asarray(base_lens)
    nodes = np.asarray(accepted_nodes)
    nacc = np.asarray(num_accepted)
    tpb = int(tokens_per_block)
    nblocks = pool.shape[0] // tpb
    out = pool.copy()

    def row(b, t):
        if t < 0 or t >= bt.shape[1] * tpb:
            return None
        blk = int(bt[b, t // tpb])
        if blk < 0 or blk >= nblocks:
            return None
        return blk * tpb + t % tpb

    L = nodes.shape[1]
    for b in range(bt.shape[0]):
        n = int(nacc[b])
        if n <= 0 or n >= L or nodes[b, 0] != 0:
            continue
        path = [int(x) for x in nodes[b, :n + 1]]
        if any(path[j] <= path[j - 1] for j in range(1, n + 1)):
            continue
        src = [row(b, int(base[b]) + path[j]) for j in range(n + 1)]
        dst = [row(b, int(base[b]) + j) for j in range(n + 1)]
        if any(r is None for r in src + dst):
            continue
        for j in range(1, n + 1):
            out[dst[j]] = pool[src[j]]
    return out


def rollback_paged(old_lens, num_accepted, k: int, tokens_per_block: int, draft_lens=None,
                   blocks_held=None, lib=None) -> dict:
    """Rollback with ragged draft lengths and paged block accounting
    (TensorRT-LLM walkthrough, update_requests and rewind_cache)."""
    lib = lib or load()
    old = _c(old_lens, np.int32)
    n = _c(num_accepted, np.int32)
    B = old.shape[0]
    lens = None if draft_lens is None else _c(draft_lens, np.int32)
    held = None if blocks_held is None else _c(blocks_held, np.int32)
    new = np.empty(B, dtype=np.int32)
    rew = np.empty(B, dtype=np.int32)
    free = np.empty(B, dtype=np.int32)
    rc = lib.oracle_rollback_paged(_ptr(old), _ptr(n), None if lens is None else _ptr(lens), int(k),
                                   None if held is None else _ptr(held), int(tokens_per_block), B,
                                   _ptr(new), _ptr(rew), _ptr(free))
    if rc not in (OK, EBADINDEX):
        raise ValueError(f"oracle_rollback_paged rc={rc}")
    return dict(new_lens=new, rewind_lens=rew, free_blocks=free, rc=rc)


def philox4x32_10(ctr, key, lib=None) -> np.ndarray:
    """One Philox4x32-10 block (Salmon et al., SC'11): 4 counter words, 2 key words -> 4 words."""
    lib = lib or load()
    c = _c(np.asarray(ctr, dtype=np.uint32), np.uint32)
    k = _c(np.asarray(key, dtype=np.uint32), np.uint32)
    out = np.empty(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def philox_uniforms(seeds, offsets, n: int, lib=None) -> np.ndarray:
    """[B, n] float32 uniforms of each request's (seed, offset) Philox stream
    (TensorRT-LLM walkthrough, rejection-sampling section: one Philox state
    per request)."""
    lib = lib or load()
    s = _c(np.asarray(seeds, dtype=np.uint64), np.uint64)
    o = _c(np.asarray(offsets, dtype=np.uint64), np.uint64)
    B = s.shape[0]
    out = np.empty((B, n), dtype=np.float32)
    rc = lib.oracle_philox_uniforms(_ptr(s), _ptr(o), B, int(n), _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_philox_uniforms rc={rc}")
    return out


def verify(w: dict, greedy: bool = False, lib=None) -> dict:
    """Run the oracle on a workload dict from ``workloads.make``."""
    if w["kind"] == "tree":
        return verify_tree(w["target"], w["tree_tokens"], w["paths"], w["dtype"], lib=lib)
    if greedy:
        return verify_greedy(w["target"], w["draft_tokens"], w["dtype"], lib=lib,
                             draft_lens=w.get("draft_lens"))
    return verify_chain(w["target"], w["draft"], w["draft_tokens"], w["uniforms"],
                        w["temperature"], w["dtype"], lib=lib, draft_lens=w.get("draft_lens"))
