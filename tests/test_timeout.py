"""Bounded device waits (the fail-closed guard of the TensorRT-LLM
walkthrough's rejection-sampling section, _rejection_buffers_valid: a verify
whose inputs are not ready must not emit tokens).  The test hooks run a
verify with its first phase left out, so the words its second phase waits
for are never written, and with a wait bound of 10^5 SM cycles: every wait
runs out and returns on its own (no fault, no hang).  The status word must
read SPEC_ETIMEOUT, every request must fail closed, and the workspace must
serve an ordinary call again after spec_workspace_init."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_row_gb300 as sv
from test_gpu_parity import check_chain, check_greedy, i32, run_chain, run_greedy, to_dev

pytestmark = pytest.mark.gpu

WAIT_CYCLES = 100_000  # about 50 us at 2 GHz


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _sh():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _chain_timeout(w, ws, top_k=0, top_p=1.0):
    B, k, V = w["B"], w["k"], w["V"]
    t, d = to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"])
    x, u = i32(w["draft_tokens"]), torch.from_numpy(w["uniforms"]).cuda()
    tok = torch.full((B, k + 1), 7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    probs = torch.zeros((B, k, 2), dtype=torch.float32, device="cuda")
    seq = i32(w["seq_lens"])
    need = (sv.lib().spec_workspace_size_filtered(B, k, V, top_k) if top_k
            else sv.lib().spec_workspace_size(B, 2 * k + 1, V))
    buf = ws.ensure(B, 2 * k + 1, V, _sh(), need)
    prm = sv.ChainParams(ctypes.sizeof(sv.ChainParams), _ptr(t), _ptr(d), workloads.DTYPE_CODE[w["dtype"]],
                         _ptr(x), None, _ptr(u), None, None, w["temperature"], B, k, V, _ptr(tok), _ptr(n),
                         _ptr(probs), _ptr(seq), top_k, top_p)
    rc = sv.lib().spec_test_timeout_chain(ctypes.byref(prm), WAIT_CYCLES, _ptr(buf), buf.numel(), _sh())
    assert rc == sv.SPEC_OK, sv.status_string(rc)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), n.cpu().numpy(), probs.cpu().numpy(), seq.cpu().numpy()


def _assert_failed_closed(w, tok, n, seq, probs=None):
    assert np.all(n == -1), n
    assert np.all(tok == -1), tok
    assert np.array_equal(seq, w["seq_lens"])
    if probs is not None:
        assert np.all(np.isnan(probs))


@pytest.mark.parametrize("name,over", [("chain_b64_k7_v128256_bf16", dict(B=3, V=20000)),
                                       ("chain_b8_k4_v32000_f32", dict(B=4, V=4097))])
def test_chain_wait_runs_out_and_fails_closed(name, over):
    w = workloads.make(name, seed=21, **over)
    ws = sv.Workspace()
    tok, n, probs, seq = _chain_timeout(w, ws)
    _assert_failed_closed(w, tok, n, seq, probs)
    assert sv.last_error(ws) == sv.SPEC_ETIMEOUT
    assert sv.last_error(ws) == sv.SPEC_OK
    sv.lib().spec_workspace_init(_ptr(ws.buf), ws.buf.numel(), _sh())
    check_chain(w, run_chain(w, workspace=ws), oracle.verify(w), f"{name} after a timeout")


def test_filtered_wait_runs_out_and_fails_closed():
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=22, B=3, V=20000)
    x = np.argmax(workloads.bf16_bits_to_f32(w["draft"]), axis=-1).astype(np.int32)
    w["draft_tokens"] = x
    ws = sv.Workspace()
    tok, n, probs, seq = _chain_timeout(w, ws, top_k=20, top_p=0.9)
    _assert_failed_closed(w, tok, n, seq, probs)
    assert sv.last_error(ws) == sv.SPEC_ETIMEOUT
    sv.lib().spec_workspace_init(_ptr(ws.buf), ws.buf.numel(), _sh())
    g = sv.verify_chain(to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"]), i32(x),
                        torch.from_numpy(w["uniforms"]).cuda(), w["temperature"], want_probs=True,
                        seq_lens=i32(w["seq_lens"]), workspace=ws, top_k=20, top_p=0.9)
    o = oracle.verify_chain_filtered(w["target"], w["draft"], x, w["uniforms"], w["temperature"], 20,
                                     float(np.float32(0.9)), w["dtype"])
    o["filter"] = (20, float(np.float32(0.9)))
    torch.cuda.synchronize()
    res = dict(tokens=g[0].cpu().numpy(), num_accepted=g[1].cpu().numpy(), probs=g[2].cpu().numpy(),
               seq_lens=oracle.rollback(w["seq_lens"], g[1].cpu().numpy(), w["k"])["new_lens"])
    check_chain(w, res, o, "filtered after a timeout")


def test_greedy_wait_runs_out_and_fails_closed():
    w = workloads.make("chain_b8_k4_v32000_f32", seed=23, B=5, V=9000)
    B, k, V = w["B"], w["k"], w["V"]
    ws = sv.Workspace()
    t, x = to_dev(w["target"], w["dtype"]), i32(w["draft_tokens"])
    tok = torch.full((B, k + 1), 7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    seq = i32(w["seq_lens"])
    buf = ws.ensure(B, k + 1, V, _sh())
    prm = sv.GreedyParams(ctypes.sizeof(sv.GreedyParams), _ptr(t), workloads.DTYPE_CODE[w["dtype"]], _ptr(x),
                          None, B, k, V, _ptr(tok), _ptr(n), _ptr(seq))
    rc = sv.lib().spec_test_timeout_greedy(ctypes.byref(prm), WAIT_CYCLES, _ptr(buf), buf.numel(), _sh())
    assert rc == sv.SPEC_OK
    torch.cuda.synchronize()
    _assert_failed_closed(w, tok.cpu().numpy(), n.cpu().numpy(), seq.cpu().numpy())
    assert sv.last_error(ws) == sv.SPEC_ETIMEOUT
    sv.lib().spec_workspace_init(_ptr(ws.buf), ws.buf.numel(), _sh())
    check_greedy(w, run_greedy(w, workspace=ws), oracle.verify(w, greedy=True), "greedy after a timeout")


def test_hooks_refuse_bad_arguments():
    w = workloads.make("chain_b1_k4_v1024_f32", seed=24, B=2, V=300)
    prm = sv.ChainParams(ctypes.sizeof(sv.ChainParams))
    assert sv.lib().spec_test_timeout_chain(ctypes.byref(prm), WAIT_CYCLES, None, 0, None) == sv.SPEC_EINVAL
    assert sv.lib().spec_test_timeout_chain(None, WAIT_CYCLES, None, 0, None) == sv.SPEC_EINVAL
    assert sv.lib().spec_test_timeout_greedy(None, 0, None, 0, None) == sv.SPEC_EINVAL
