"""The allocation-free chain entry point, for callers that cannot allocate
device memory (an allocator that forbids allocations during a step, or host
code without a CUDA allocator).  It must give the same results as the
workspace entry point and agree with the CPU oracle, call after call,
although every call reuses the same fixed device scratch array.  Collected
last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import speculative_decoding_verification_row_gb300 as sv
from test_gpu_parity import check_chain

pytestmark = pytest.mark.gpu


def _dev(arr, dtype):
    if dtype == workloads.BF16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("name,over", [("chain_b64_k7_v128256_bf16", dict(B=8, V=40000)),
                                       ("chain_b8_k4_v32000_f32", dict(B=4, V=4097))])
def test_noalloc_matches_workspace_entry_point(name, over):
    w = workloads.make(name, seed=21, **over)
    t, d = _dev(w["target"], w["dtype"]), _dev(w["draft"], w["dtype"])
    x, u = _i32(w["draft_tokens"]), torch.from_numpy(w["uniforms"]).cuda()
    seq = _i32(w["seq_lens"])
    ref_tok, ref_n, ref_p = sv.verify_chain(t, d, x, u, w["temperature"], want_probs=True, seq_lens=seq)
    ref_seq = seq.cpu().numpy()
    lib = sv.lib()
    code = workloads.DTYPE_CODE[w["dtype"]]
    B, k, V = w["B"], w["k"], w["V"]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):  # two calls in a row share the same scratch array
        tok = torch.full((B, k + 1), 7, dtype=torch.int32, device="cuda")
        n = torch.full((B,), 7, dtype=torch.int32, device="cuda")
        probs = torch.zeros((B, k, 2), dtype=torch.float32, device="cuda")
        s = _i32(w["seq_lens"])
        P = lambda z: ctypes.c_void_p(z.data_ptr())  # noqa: E731
        rc = lib.spec_verify_chain_noalloc(P(t), P(d), code, P(x), P(u), ctypes.c_float(w["temperature"]),
                                           B, k, V, P(tok), P(n), P(probs), P(s), stream)
        assert rc == sv.SPEC_OK, sv.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok), f"call {call}: tokens"
        assert torch.equal(n, ref_n), f"call {call}: accepted counts"
        assert np.array_equal(s.cpu().numpy(), ref_seq), f"call {call}: seq_lens"
        rel = ((probs - ref_p).abs() / ref_p.abs().clamp_min(1e-30)).max().item()
        assert rel <= 1e-5, f"call {call}: probabilities differ by {rel}"
        # and against the oracle itself (exact outside flagged near-ties)
        g = dict(tokens=tok.cpu().numpy(), num_accepted=n.cpu().numpy(), probs=probs.cpu().numpy(),
                 seq_lens=s.cpu().numpy())
        check_chain(w, g, oracle.verify(w), f"noalloc {name} call {call}")


def test_noalloc_refuses_host_arrays_and_leaves_its_scratch_usable():
    # Arrays outside the current device's memory are refused (SPEC_EINVAL)
    # before the shared scratch array is written; the next call is correct.
    w = workloads.make("chain_b8_k4_v32000_f32", seed=25, B=3, V=3000)
    host_tokens = np.ascontiguousarray(w["draft_tokens"], dtype=np.int32)
    t, d = _dev(w["target"], w["dtype"]), _dev(w["draft"], w["dtype"])
    u = torch.from_numpy(w["uniforms"]).cuda()
    B, k, V = w["B"], w["k"], w["V"]
    tok = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
    n = torch.empty((B,), dtype=torch.int32, device="cuda")
    P = lambda z: ctypes.c_void_p(z.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = sv.lib().spec_verify_chain_noalloc(P(t), P(d), 0, host_tokens.ctypes.data_as(ctypes.c_void_p), P(u),
                                            ctypes.c_float(w["temperature"]), B, k, V, P(tok), P(n),
                                            None, None, stream)
    assert rc == sv.SPEC_EINVAL
    tk, nn, pr = sv.verify_chain_noalloc(t, d, _i32(w["draft_tokens"]), u, w["temperature"], want_probs=True)
    torch.cuda.synchronize()
    g = dict(tokens=tk.cpu().numpy(), num_accepted=nn.cpu().numpy(), probs=pr.cpu().numpy(),
             seq_lens=oracle.rollback(w["seq_lens"], nn.cpu().numpy(), k)["new_lens"])
    check_chain(w, g, oracle.verify(w), "noalloc after a refused call")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = sv.lib()
    dummy = ctypes.c_void_p(256)
    # B=4096, k=16, V=262144 needs far more than the fixed scratch: refused before any launch
    rc = lib.spec_verify_chain_noalloc(dummy, dummy, 1, dummy, dummy, ctypes.c_float(1.0),
                                       4096, 16, 262144, dummy, dummy, None, None, None)
    assert rc == sv.SPEC_EWORKSPACE
    assert lib.spec_workspace_size(4096, 33, 262144) > sv.SPEC_NOALLOC_SCRATCH_BYTES
