"""Stream order around a verify call.  Each call's first grid is launched as
a programmatic dependent of the stream's previous kernel and begins by
waiting for it, so the call must still see every write queued before it: an
asynchronous host-to-device copy of its logits, or a kernel that produced
them.  Each case zeroes the inputs on the device first, queues the producer
and the verify back to back with no synchronisation between them, and must
give the results of a fully synchronised call."""
import numpy as np
import pytest
import torch

import workloads
import speculative_decoding_verification_row_gb300 as sv

pytestmark = pytest.mark.gpu


def _host(w, key):
    a = np.ascontiguousarray(w[key])
    if w["dtype"] == workloads.BF16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


def _as_logits(t, w):
    return t.view(torch.bfloat16) if w["dtype"] == workloads.BF16 else t


@pytest.mark.parametrize("top_k,top_p", [(0, 1.0), (50, 0.9), (0, 0.9)])
def test_verify_sees_async_copies_and_producer_kernels(top_k, top_p):
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=71, B=24)
    ht, hd = _host(w, "target"), _host(w, "draft")
    dt, dd = torch.empty_like(ht, device="cuda"), torch.empty_like(hd, device="cuda")
    x = torch.from_numpy(w["draft_tokens"]).cuda()
    u = torch.from_numpy(w["uniforms"]).cuda()
    ws = sv.Workspace()

    def verify():
        tok, n, _ = sv.verify_chain(_as_logits(dt, w), _as_logits(dd, w), x, u, w["temperature"],
                                    workspace=ws, top_k=top_k, top_p=top_p)
        return tok, n

    dt.copy_(ht)
    dd.copy_(hd)
    torch.cuda.synchronize()
    ref_tok, ref_n = verify()
    torch.cuda.synchronize()
    ref_tok, ref_n = ref_tok.clone(), ref_n.clone()

    # 1. an asynchronous pinned copy right before the call
    for _ in range(3):
        dt.zero_()
        dd.zero_()
        torch.cuda.synchronize()
        dt.copy_(ht, non_blocking=True)
        dd.copy_(hd, non_blocking=True)
        tok, n = verify()
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(n, ref_n)

    # 2. a device kernel that produces the logits right before the call
    st, sd = dt.clone(), dd.clone()
    for _ in range(3):
        dt.zero_()
        dd.zero_()
        torch.cuda.synchronize()
        dt.copy_(st)
        dd.copy_(sd)
        tok, n = verify()
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok) and torch.equal(n, ref_n)


def test_tree_and_greedy_see_producer_kernels():
    w = workloads.make("tree_b16_n60_l4_v151936_bf16", seed=72, B=8)
    ht = _host(w, "target")
    dt = torch.empty_like(ht, device="cuda")
    tt = torch.from_numpy(w["tree_tokens"].astype(np.int32)).cuda()
    pp = torch.from_numpy(w["paths"].astype(np.int32)).cuda()
    uu = torch.from_numpy(w["uniforms"]).cuda()
    dt.copy_(ht)
    torch.cuda.synchronize()
    ref = [t.clone() for t in sv.verify_tree(_as_logits(dt, w), tt, pp)]
    ref_s = [t.clone() for t in sv.verify_tree_sampled(_as_logits(dt, w), tt, pp, uu, w["temperature"])]
    torch.cuda.synchronize()
    src = dt.clone()
    for _ in range(3):
        dt.zero_()
        torch.cuda.synchronize()
        dt.copy_(src)
        got = sv.verify_tree(_as_logits(dt, w), tt, pp)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
        dt.zero_()
        torch.cuda.synchronize()
        dt.copy_(ht, non_blocking=True)
        got = sv.verify_tree_sampled(_as_logits(dt, w), tt, pp, uu, w["temperature"])
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(got, ref_s))
