"""GB300-native speculative-decoding verification row.

A thin ctypes binding over ``libspecverify.so`` (C ABI in
``include/spec_verify.h``).  The functions here only check and marshal
arguments: every step of verification runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  If the library has
not been built the first call raises; there is no CPU fallback.

Calls (same names as the C ABI):
  verify_chain     chain rejection-sampling verify (vLLM anatomy page,
                   "Speculative Decoding")
  verify_greedy    greedy chain verify (Kestrel article 32, section 3.3)
  verify_tree      greedy EAGLE tree verify (TensorRT-LLM deployment page,
                   "Eagle-2" section)
  rollback_lengths KV cursor rollback (TensorRT-LLM walkthrough,
                   update_requests / rewind_cache)
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .stats import acceptance_stats, anchored_emitted  # noqa: F401  (host bookkeeping)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspecverify.so")

SPEC_OK, SPEC_EINVAL, SPEC_EBADINDEX, SPEC_ECUDA, SPEC_EWORKSPACE, SPEC_ETIMEOUT = 0, -1, -2, -3, -4, -5
SPEC_ELIMIT = -6
SPEC_F32, SPEC_BF16 = 0, 1
SPEC_MAX_DRAFT = 64
SPEC_MAX_BATCH = 8192
SPEC_MAX_TREE_NODES = 1024
SPEC_MAX_PATH_LEN = 64
SPEC_MAX_TOPK = 256

# Every entry point the header declares.
SYMBOLS = ("spec_workspace_size", "spec_workspace_init", "spec_verify_chain",
           "spec_verify_greedy", "spec_verify_tree", "spec_rollback_lengths",
           "spec_last_error", "spec_status_string", "spec_verify_chain_noalloc",
           "spec_relocate_accepted_kv", "spec_verify_chain_philox", "spec_philox_uniforms",
           "spec_verify_chain_ex", "spec_verify_greedy_ex", "spec_rollback_paged",
           "spec_workspace_size_filtered", "spec_test_timeout_chain", "spec_test_timeout_greedy",
           "spec_verify_tree_sampled")
SPEC_NOALLOC_SCRATCH_BYTES = 4 << 20

class ChainParams(ctypes.Structure):
    """spec_chain_params (include/spec_verify.h), field for field."""
    _fields_ = [("size", ctypes.c_size_t), ("target_logits", ctypes.c_void_p),
                ("draft_logits", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("draft_tokens", ctypes.c_void_p), ("draft_lens", ctypes.c_void_p),
                ("uniforms", ctypes.c_void_p), ("seeds", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("temperature", ctypes.c_float),
                ("B", ctypes.c_int), ("k", ctypes.c_int), ("V", ctypes.c_int),
                ("out_tokens", ctypes.c_void_p), ("out_num_accepted", ctypes.c_void_p),
                ("out_probs", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("top_k", ctypes.c_int), ("top_p", ctypes.c_float), ("min_p", ctypes.c_float)]


class GreedyParams(ctypes.Structure):
    """spec_greedy_params (include/spec_verify.h), field for field."""
    _fields_ = [("size", ctypes.c_size_t), ("target_logits", ctypes.c_void_p),
                ("dtype", ctypes.c_int), ("draft_tokens", ctypes.c_void_p),
                ("draft_lens", ctypes.c_void_p), ("B", ctypes.c_int), ("k", ctypes.c_int),
                ("V", ctypes.c_int), ("out_tokens", ctypes.c_void_p),
                ("out_num_accepted", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def _bind(lib):
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.spec_workspace_size.argtypes = [I, I, I]
    lib.spec_workspace_size.restype = S
    lib.spec_workspace_init.argtypes = [P, S, P]
    lib.spec_workspace_size_filtered.argtypes = [I, I, I, I]
    lib.spec_workspace_size_filtered.restype = S
    lib.spec_verify_chain.argtypes = [P, P, I, P, P, ctypes.c_float, I, I, I, P, P, P, P, P, S, P]
    lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, P, S, P]
    lib.spec_verify_tree.argtypes = [P, I, P, P, I, I, I, I, I, P, P, P, P, P, P, S, P]
    lib.spec_verify_tree_sampled.argtypes = [P, I, P, P, P, ctypes.c_float, I, I, I, I, I, P, P, P, P, P,
                                             P, S, P]
    lib.spec_rollback_lengths.argtypes = [P, P, I, I, P, P, P]
    lib.spec_verify_chain_noalloc.argtypes = [P, P, I, P, P, ctypes.c_float, I, I, I, P, P, P, P, P]
    lib.spec_last_error.argtypes = [P, S, P, ctypes.POINTER(ctypes.c_int)]
    lib.spec_relocate_accepted_kv.argtypes = [P, S, I, I, P, I, P, P, P, I, I, P]
    lib.spec_verify_chain_philox.argtypes = [P, P, I, P, P, P, ctypes.c_float, I, I, I, P, P, P, P, P, S, P]
    lib.spec_philox_uniforms.argtypes = [P, P, I, I, P, P]
    lib.spec_verify_chain_ex.argtypes = [ctypes.POINTER(ChainParams), P, S, P]
    lib.spec_verify_greedy_ex.argtypes = [ctypes.POINTER(GreedyParams), P, S, P]
    lib.spec_rollback_paged.argtypes = [P, P, P, I, P, I, I, P, P, P, P]
    lib.spec_test_timeout_chain.argtypes = [ctypes.POINTER(ChainParams), ctypes.c_longlong, P, S, P]
    lib.spec_test_timeout_greedy.argtypes = [ctypes.POINTER(GreedyParams), ctypes.c_longlong, P, S, P]
    lib.spec_status_string.argtypes = [I]
    lib.spec_status_string.restype = ctypes.c_char_p
    for f in ("spec_workspace_init", "spec_verify_chain", "spec_verify_greedy", "spec_verify_tree",
              "spec_rollback_lengths", "spec_last_error", "spec_verify_chain_noalloc",
              "spec_relocate_accepted_kv", "spec_verify_chain_philox", "spec_philox_uniforms",
              "spec_verify_chain_ex", "spec_verify_greedy_ex", "spec_rollback_paged",
              "spec_test_timeout_chain", "spec_test_timeout_greedy", "spec_verify_tree_sampled"):
        getattr(lib, f).restype = I
    return lib


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
                _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(code: int) -> str:
    return lib().spec_status_string(int(code)).decode()


# ---------------------------------------------------------------- marshalling helpers
def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on(device):
    """The C calls run on the current device: make the arrays' device current
    for the duration of a call."""
    return torch.cuda.device(device)


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream), stream
    return ctypes.c_void_p(int(stream)), None


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _logit_code(t: torch.Tensor, name: str) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise ValueError(f"{name} must be bfloat16 or float32, got {t.dtype}")


def _out(t, name, shape, dtype, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _dev(t, name, dtype, shape)


class Workspace:
    """Device scratch for verify calls on one stream (grown on demand).

    A workspace must not be shared by calls that may overlap on the GPU."""

    def __init__(self, device=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.buf = None

    def ensure(self, B: int, rows: int, V: int, stream_handle, need: int | None = None) -> torch.Tensor:
        """Grow to spec_workspace_size(B, rows, V) bytes, or to `need` bytes."""
        if need is None:
            need = lib().spec_workspace_size(B, rows, V)
        if need == 0:
            raise SpecError("spec_workspace_size", SPEC_EINVAL)
        if self.buf is None or self.buf.numel() < need:
            self.buf = torch.empty(need, dtype=torch.uint8, device=self.device)
            with _on(self.buf.device):
                rc = lib().spec_workspace_init(_ptr(self.buf), self.buf.numel(), stream_handle)
            if rc != SPEC_OK:
                raise SpecError("spec_workspace_init", rc)
        return self.buf

    @property
    def nbytes(self) -> int:
        return 0 if self.buf is None else self.buf.numel()


_default_ws: dict = {}


def default_workspace(device, stream_handle) -> Workspace:
    key = (torch.device(device).index, int(stream_handle.value or 0))
    ws = _default_ws.get(key)
    if ws is None:
        ws = _default_ws[key] = Workspace(device)
    return ws


# ---------------------------------------------------------------- calls
def verify_chain(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
                 out_tokens=None, out_num_accepted=None, out_probs=None, want_probs=False,
                 seq_lens=None, workspace: Workspace | None = None, stream=None,
                 seeds=None, offsets=None, draft_lens=None, top_k: int = 0, top_p: float = 1.0,
                 min_p: float = 0.0):
    """Chain rejection-sampling verify; returns (tokens [B,k+1], num_accepted [B], probs [B,k,2] or None).

    seq_lens (int32 [B], optional) is advanced in place by n_acc + 1.  With
    uniforms=None, seeds and offsets (int64 [B]) select each request's Philox
    stream and the uniforms are drawn inside the kernel.  draft_lens (int32
    [B], optional): each request's real draft length (ragged verify).
    top_k > 0, top_p < 1 or min_p > 0: verify on the top-k / top-p / min_p
    filtered target and draft distributions (spec_chain_params.top_k /
    top_p / min_p; top_k = 0 ranks no top-k set)."""
    t = _dev(target_logits, "target_logits")
    if t.dim() != 3:
        raise ValueError("target_logits must be [B, k+1, V]")
    B, k1, V = t.shape
    k = k1 - 1
    code = _logit_code(t, "target_logits")
    d = _dev(draft_logits, "draft_logits", t.dtype, (B, k, V))
    x = _dev(draft_tokens, "draft_tokens", torch.int32, (B, k))
    if uniforms is not None:
        u = _dev(uniforms, "uniforms", torch.float32, (B, k + 1))
    else:
        sd = _dev(seeds, "seeds", torch.int64, (B,))
        of = _dev(offsets, "offsets", torch.int64, (B,))
    dev = t.device
    tok = _out(out_tokens, "out_tokens", (B, k + 1), torch.int32, dev)
    n = _out(out_num_accepted, "out_num_accepted", (B,), torch.int32, dev)
    probs = None
    if out_probs is not None or want_probs:
        probs = _out(out_probs, "out_probs", (B, k, 2), torch.float32, dev)
    if seq_lens is not None:
        _dev(seq_lens, "seq_lens", torch.int32, (B,))
    sh, _ = _stream_handle(stream, dev)
    ws = workspace or default_workspace(dev, sh)
    filtered = top_k != 0 or top_p != 1.0 or min_p != 0.0
    need = lib().spec_workspace_size_filtered(B, k, V, int(top_k)) if filtered else None
    buf = ws.ensure(B, 2 * k + 1, V, sh, need)
    if draft_lens is not None or filtered:
        lens = None if draft_lens is None else _dev(draft_lens, "draft_lens", torch.int32, (B,))
        prm = ChainParams(ctypes.sizeof(ChainParams), _ptr(t), _ptr(d), code, _ptr(x), _ptr(lens),
                          _ptr(u) if uniforms is not None else None,
                          None if uniforms is not None else _ptr(sd),
                          None if uniforms is not None else _ptr(of), float(temperature), B, k, V,
                          _ptr(tok), _ptr(n), _ptr(probs), _ptr(seq_lens), int(top_k),
                          float(top_p), float(min_p))
        with _on(dev):
            rc = lib().spec_verify_chain_ex(ctypes.byref(prm), _ptr(buf), buf.numel(), sh)
        name = "spec_verify_chain_ex"
    elif uniforms is not None:
        with _on(dev):
            rc = lib().spec_verify_chain(_ptr(t), _ptr(d), code, _ptr(x), _ptr(u), float(temperature),
                                         B, k, V, _ptr(tok), _ptr(n), _ptr(probs), _ptr(seq_lens),
                                         _ptr(buf), buf.numel(), sh)
        name = "spec_verify_chain"
    else:
        with _on(dev):
            rc = lib().spec_verify_chain_philox(_ptr(t), _ptr(d), code, _ptr(x), _ptr(sd), _ptr(of),
                                                float(temperature), B, k, V, _ptr(tok), _ptr(n),
                                                _ptr(probs), _ptr(seq_lens), _ptr(buf), buf.numel(), sh)
        name = "spec_verify_chain_philox"
    if rc != SPEC_OK:
        raise SpecError(name, rc)
    return tok, n, probs


def verify_chain_noalloc(target_logits, draft_logits, draft_tokens, uniforms, temperature: float, *,
                         out_tokens=None, out_num_accepted=None, out_probs=None, want_probs=False,
                         seq_lens=None, stream=None):
    """verify_chain without a workspace: for callers that cannot allocate device
    scratch.  The library's fixed device array serves as scratch (problems up to
    SPEC_NOALLOC_SCRATCH_BYTES of scratch); calls that overlap on the GPU race.
    Output tensors are allocated here unless passed in."""
    t = _dev(target_logits, "target_logits")
    if t.dim() != 3:
        raise ValueError("target_logits must be [B, k+1, V]")
    B, k1, V = t.shape
    k = k1 - 1
    code = _logit_code(t, "target_logits")
    d = _dev(draft_logits, "draft_logits", t.dtype, (B, k, V))
    x = _dev(draft_tokens, "draft_tokens", torch.int32, (B, k))
    u = _dev(uniforms, "uniforms", torch.float32, (B, k + 1))
    dev = t.device
    tok = _out(out_tokens, "out_tokens", (B, k + 1), torch.int32, dev)
    n = _out(out_num_accepted, "out_num_accepted", (B,), torch.int32, dev)
    probs = None
    if out_probs is not None or want_probs:
        probs = _out(out_probs, "out_probs", (B, k, 2), torch.float32, dev)
    if seq_lens is not None:
        _dev(seq_lens, "seq_lens", torch.int32, (B,))
    sh, _ = _stream_handle(stream, dev)
    with _on(dev):
        rc = lib().spec_verify_chain_noalloc(_ptr(t), _ptr(d), code, _ptr(x), _ptr(u), float(temperature),
                                             B, k, V, _ptr(tok), _ptr(n), _ptr(probs), _ptr(seq_lens), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_verify_chain_noalloc", rc)
    return tok, n, probs


def verify_greedy(target_logits, draft_tokens, *, out_tokens=None, out_num_accepted=None,
                  seq_lens=None, workspace: Workspace | None = None, stream=None,
                  draft_lens=None):
    """Greedy chain verify; returns (tokens [B,k+1], num_accepted [B]).
    draft_lens (int32 [B], optional): each request's real draft length."""
    t = _dev(target_logits, "target_logits")
    if t.dim() != 3:
        raise ValueError("target_logits must be [B, k+1, V]")
    B, k1, V = t.shape
    k = k1 - 1
    code = _logit_code(t, "target_logits")
    x = _dev(draft_tokens, "draft_tokens", torch.int32, (B, k))
    dev = t.device
    tok = _out(out_tokens, "out_tokens", (B, k + 1), torch.int32, dev)
    n = _out(out_num_accepted, "out_num_accepted", (B,), torch.int32, dev)
    if seq_lens is not None:
        _dev(seq_lens, "seq_lens", torch.int32, (B,))
    sh, _ = _stream_handle(stream, dev)
    ws = workspace or default_workspace(dev, sh)
    buf = ws.ensure(B, k + 1, V, sh)
    if draft_lens is not None:
        lens = _dev(draft_lens, "draft_lens", torch.int32, (B,))
        prm = GreedyParams(ctypes.sizeof(GreedyParams), _ptr(t), code, _ptr(x), _ptr(lens), B, k, V,
                           _ptr(tok), _ptr(n), _ptr(seq_lens))
        with _on(dev):
            rc = lib().spec_verify_greedy_ex(ctypes.byref(prm), _ptr(buf), buf.numel(), sh)
    else:
        with _on(dev):
            rc = lib().spec_verify_greedy(_ptr(t), code, _ptr(x), B, k, V, _ptr(tok), _ptr(n),
                                          _ptr(seq_lens), _ptr(buf), buf.numel(), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_verify_greedy", rc)
    return tok, n


def verify_tree(target_logits, tree_tokens, paths, *, out_tokens=None, out_num_accepted=None,
                out_best_path=None, out_accepted_nodes=None, seq_lens=None,
                workspace: Workspace | None = None, stream=None):
    """Greedy tree verify; returns (tokens [B,L], num_accepted [B], best_path [B], accepted_nodes [B,L])."""
    t = _dev(target_logits, "target_logits")
    if t.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = t.shape
    code = _logit_code(t, "target_logits")
    tt = _dev(tree_tokens, "tree_tokens", torch.int32, (B, N))
    p = _dev(paths, "paths", torch.int32)
    if p.dim() != 3 or p.shape[0] != B:
        raise ValueError("paths must be [B, P, L]")
    P, L = p.shape[1], p.shape[2]
    dev = t.device
    tok = _out(out_tokens, "out_tokens", (B, L), torch.int32, dev)
    n = _out(out_num_accepted, "out_num_accepted", (B,), torch.int32, dev)
    best = _out(out_best_path, "out_best_path", (B,), torch.int32, dev)
    nodes = _out(out_accepted_nodes, "out_accepted_nodes", (B, L), torch.int32, dev)
    if seq_lens is not None:
        _dev(seq_lens, "seq_lens", torch.int32, (B,))
    sh, _ = _stream_handle(stream, dev)
    ws = workspace or default_workspace(dev, sh)
    buf = ws.ensure(B, N, V, sh)
    with _on(dev):
        rc = lib().spec_verify_tree(_ptr(t), code, _ptr(tt), _ptr(p), B, N, P, L, V, _ptr(tok),
                                    _ptr(n), _ptr(best), _ptr(nodes), _ptr(seq_lens), _ptr(buf),
                                    buf.numel(), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_verify_tree", rc)
    return tok, n, best, nodes


def verify_tree_sampled(target_logits, tree_tokens, paths, uniforms, temperature: float, *,
                        out_tokens=None, out_num_accepted=None, out_best_path=None,
                        out_accepted_nodes=None, seq_lens=None, workspace: Workspace | None = None,
                        stream=None):
    """Stochastic tree verify (chosen children as point-mass proposals);
    uniforms float32 [B, N] (column n >= 1: node n's accept test, column 0:
    the final draw).  Returns (tokens [B,L], num_accepted [B], best_path [B],
    accepted_nodes [B,L])."""
    t = _dev(target_logits, "target_logits")
    if t.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = t.shape
    code = _logit_code(t, "target_logits")
    tt = _dev(tree_tokens, "tree_tokens", torch.int32, (B, N))
    p = _dev(paths, "paths", torch.int32)
    if p.dim() != 3 or p.shape[0] != B:
        raise ValueError("paths must be [B, P, L]")
    P, L = p.shape[1], p.shape[2]
    u = _dev(uniforms, "uniforms", torch.float32, (B, N))
    dev = t.device
    tok = _out(out_tokens, "out_tokens", (B, L), torch.int32, dev)
    n = _out(out_num_accepted, "out_num_accepted", (B,), torch.int32, dev)
    best = _out(out_best_path, "out_best_path", (B,), torch.int32, dev)
    nodes = _out(out_accepted_nodes, "out_accepted_nodes", (B, L), torch.int32, dev)
    if seq_lens is not None:
        _dev(seq_lens, "seq_lens", torch.int32, (B,))
    sh, _ = _stream_handle(stream, dev)
    ws = workspace or default_workspace(dev, sh)
    buf = ws.ensure(B, N, V, sh)
    with _on(dev):
        rc = lib().spec_verify_tree_sampled(_ptr(t), code, _ptr(tt), _ptr(p), _ptr(u), float(temperature),
                                            B, N, P, L, V, _ptr(tok), _ptr(n), _ptr(best), _ptr(nodes),
                                            _ptr(seq_lens), _ptr(buf), buf.numel(), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_verify_tree_sampled", rc)
    return tok, n, best, nodes


def rollback_lengths(old_lens, num_accepted, k: int, *, new_lens=None, rewind_lens=None,
                     stream=None):
    """KV cursor rollback lengths; returns (new_lens [B], rewind_lens [B])."""
    o = _dev(old_lens, "old_lens", torch.int32)
    B = o.shape[0]
    n = _dev(num_accepted, "num_accepted", torch.int32, (B,))
    new = _out(new_lens, "new_lens", (B,), torch.int32, o.device)
    rew = _out(rewind_lens, "rewind_lens", (B,), torch.int32, o.device)
    sh, _ = _stream_handle(stream, o.device)
    with _on(o.device):
        rc = lib().spec_rollback_lengths(_ptr(o), _ptr(n), int(k), B, _ptr(new), _ptr(rew), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_rollback_lengths", rc)
    return new, rew


def relocate_accepted_kv(kv_pool, block_tables, base_lens, accepted_nodes, num_accepted,
                         tokens_per_block: int, *, stream=None):
    """Gather the accepted tree nodes' KV rows to consecutive positions after
    each request's prefix, in place.  kv_pool: [num_blocks * tokens_per_block,
    ...] (any dtype; a token's row is its trailing dims), block_tables
    [B, max_blocks] int32, base_lens [B], accepted_nodes [B, L], num_accepted [B]."""
    if not isinstance(kv_pool, torch.Tensor) or not kv_pool.is_cuda or not kv_pool.is_contiguous():
        raise ValueError("kv_pool must be a contiguous CUDA tensor")
    rows = kv_pool.shape[0]
    if rows % tokens_per_block:
        raise ValueError("kv_pool rows must be num_blocks * tokens_per_block")
    row_bytes = kv_pool.numel() * kv_pool.element_size() // max(rows, 1)
    bt = _dev(block_tables, "block_tables", torch.int32)
    B = bt.shape[0]
    base = _dev(base_lens, "base_lens", torch.int32, (B,))
    nodes = _dev(accepted_nodes, "accepted_nodes", torch.int32)
    n = _dev(num_accepted, "num_accepted", torch.int32, (B,))
    sh, _ = _stream_handle(stream, kv_pool.device)
    with _on(kv_pool.device):
        rc = lib().spec_relocate_accepted_kv(_ptr(kv_pool), ctypes.c_size_t(row_bytes),
                                             int(tokens_per_block), rows // tokens_per_block, _ptr(bt),
                                             bt.shape[1], _ptr(base), _ptr(nodes), _ptr(n), B,
                                             nodes.shape[1], sh)
    if rc != SPEC_OK:
        raise SpecError("spec_relocate_accepted_kv", rc)
    return kv_pool


def rollback_paged(old_lens, num_accepted, k: int, tokens_per_block: int, *, draft_lens=None,
                   blocks_held=None, new_lens=None, rewind_lens=None, free_blocks=None,
                   stream=None):
    """Rollback with ragged draft lengths and paged block accounting; returns
    (new_lens [B], rewind_lens [B], free_blocks [B])."""
    o = _dev(old_lens, "old_lens", torch.int32)
    B = o.shape[0]
    n = _dev(num_accepted, "num_accepted", torch.int32, (B,))
    lens = None if draft_lens is None else _dev(draft_lens, "draft_lens", torch.int32, (B,))
    held = None if blocks_held is None else _dev(blocks_held, "blocks_held", torch.int32, (B,))
    new = _out(new_lens, "new_lens", (B,), torch.int32, o.device)
    rew = _out(rewind_lens, "rewind_lens", (B,), torch.int32, o.device)
    fre = _out(free_blocks, "free_blocks", (B,), torch.int32, o.device)
    sh, _ = _stream_handle(stream, o.device)
    with _on(o.device):
        rc = lib().spec_rollback_paged(_ptr(o), _ptr(n), _ptr(lens), int(k), _ptr(held),
                                       int(tokens_per_block), B, _ptr(new), _ptr(rew), _ptr(fre), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_rollback_paged", rc)
    return new, rew, fre


def philox_uniforms(seeds, offsets, n: int, *, stream=None):
    """[B, n] float32: the uniforms verify_chain draws for each request's
    (seed, offset) Philox stream when called without uniforms."""
    sd = _dev(seeds, "seeds", torch.int64)
    B = sd.shape[0]
    of = _dev(offsets, "offsets", torch.int64, (B,))
    out = torch.empty((B, n), dtype=torch.float32, device=sd.device)
    sh, _ = _stream_handle(stream, sd.device)
    with _on(sd.device):
        rc = lib().spec_philox_uniforms(_ptr(sd), _ptr(of), B, int(n), _ptr(out), sh)
    if rc != SPEC_OK:
        raise SpecError("spec_philox_uniforms", rc)
    return out


def last_error(workspace: Workspace, stream=None) -> int:
    """Synchronise, read and clear the workspace's data-dependent status."""
    if workspace.buf is None:
        return SPEC_OK
    sh, _ = _stream_handle(stream, workspace.buf.device)
    out = ctypes.c_int(0)
    with _on(workspace.buf.device):
        rc = lib().spec_last_error(_ptr(workspace.buf), workspace.buf.numel(), sh, ctypes.byref(out))
    if rc != SPEC_OK:
        raise SpecError("spec_last_error", rc)
    return out.value
