"""Stochastic tree verify: the CUDA path (through the C ABI binding) against
the oracle's point-mass reading of the deployment page's tree verification by
rejection sampling.  Tokens, counts, best paths, accepted nodes and sequence
lengths must match exactly outside the near-ties the oracle flags (a child's
accept test within 1e-5 of its residual probability, scaled by the
residual's normaliser, or a final draw within 1e-6 * Z of a CDF boundary).
The CPU-only checks here cover the host side; the oracle's own pins are in
tests/_pins.py (pin_tree_sampled)."""
import numpy as np
import pytest
import torch

import _report
import oracle
import workloads
import speculative_decoding_verification_row_gb300 as sv
from test_gpu_parity import _offset_copy, i32, to_dev

pytestmark = pytest.mark.gpu


def run_tree_sampled(w, misalign=False, workspace=None):
    t = to_dev(w["target"], w["dtype"])
    if misalign:
        t = _offset_copy(t)
    seq = i32(w["seq_lens"])
    tok, n, best, nodes = sv.verify_tree_sampled(t, i32(w["tree_tokens"]), i32(w["paths"]),
                                                 torch.from_numpy(w["uniforms"]).cuda(), w["temperature"],
                                                 seq_lens=seq, workspace=workspace)
    torch.cuda.synchronize()
    return dict(tokens=tok.cpu().numpy(), num_accepted=n.cpu().numpy(), best_path=best.cpu().numpy(),
                accepted_nodes=nodes.cpu().numpy(), seq_lens=seq.cpu().numpy())


def oracle_tree_sampled(w):
    return oracle.verify_tree_sampled(w["target"], w["tree_tokens"], w["paths"], w["uniforms"],
                                      w["temperature"], w["dtype"])


def check_tree_sampled(w, g, o, label, full_size=False):
    flagged = mism = 0
    for b in range(w["B"]):
        f = bool(o["flags"][b].any())
        flagged += f
        same = all(np.array_equal(g[key][b], o[key][b])
                   for key in ("tokens", "num_accepted", "best_path", "accepted_nodes"))
        if not same:
            mism += 1
            assert f, (f"{label}: unflagged mismatch at request {b}: gpu {g['tokens'][b]} "
                       f"nodes {g['accepted_nodes'][b]}, oracle {o['tokens'][b]} nodes {o['accepted_nodes'][b]}")
            assert g["num_accepted"][b] >= 0
    want_seq = np.where(g["num_accepted"] >= 0, w["seq_lens"] + g["num_accepted"] + 1, w["seq_lens"])
    assert np.array_equal(g["seq_lens"], want_seq), label
    _report.record(case=label, kind="chain", requests=w["B"], flagged=flagged, mismatched=mism,
                   full_size=full_size, mean_accepted=float(np.mean(o["num_accepted"])))


def _peaked_tree(seed, B=6, N=20, L=4, V=3000, dtype=workloads.BF16, T=0.6, level_sizes=None):
    # children are the top tokens of their parent's row, and the rows are
    # peaked enough that walks go deep
    w = workloads.make("tree_b16_n60_l4_v151936_bf16", seed=seed, B=B, N=N, L=L, V=V, dtype=dtype,
                       temperature=T, target_std=3.0, child_noise_std=0.3,
                       level_sizes=level_sizes)
    return w


@pytest.mark.parametrize("dtype", [workloads.BF16, workloads.F32])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_sampled_small(dtype, seed):
    w = _peaked_tree(seed, dtype=dtype, level_sizes=[6, 7, 6])
    check_tree_sampled(w, run_tree_sampled(w), oracle_tree_sampled(w), f"tree sampled {dtype}/s{seed}")


@pytest.mark.parametrize("over", [dict(V=5001, N=12, L=5, level_sizes=[3, 3, 3, 2]),   # element path, ragged
                                  dict(V=300000, N=9, L=3, level_sizes=[4, 4]),        # beyond 2^18 tokens
                                  dict(V=64, N=2, L=2, level_sizes=[1]),               # smallest tree
                                  dict(V=4096, N=60, L=4, level_sizes=[8, 25, 26])])   # the workload's shape
def test_tree_sampled_shapes(over):
    w = _peaked_tree(7, **over)
    o = oracle_tree_sampled(w)
    check_tree_sampled(w, run_tree_sampled(w), o, f"tree sampled {over}")
    check_tree_sampled(w, run_tree_sampled(w, misalign=True), o, f"tree sampled {over} misaligned")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_sampled_full(seed):
    w = workloads.make("tree_b16_n60_l4_v151936_bf16", seed=seed)
    check_tree_sampled(w, run_tree_sampled(w), oracle_tree_sampled(w),
                       f"tree_b16_n60_l4_v151936_bf16 sampled/s{seed}", full_size=True)


def test_tree_sampled_one_hot_rows_equal_greedy_tree():
    # One-hot target rows: the walk accepts exactly the argmax children, as
    # the greedy tree verify does.
    w = _peaked_tree(11, B=8, N=30, L=4, V=2000, dtype=workloads.F32, level_sizes=[8, 12, 9])
    rng = np.random.default_rng(11)
    g = rng.integers(0, w["V"], (w["B"], w["N"]))
    for b in range(w["B"]):
        for n in range(1, w["N"]):
            if rng.random() < 0.5:
                g[b, w["parents"][b, n]] = w["tree_tokens"][b, n]
    tgt = np.full((w["B"], w["N"], w["V"]), -np.inf, np.float32)
    tgt[np.arange(w["B"])[:, None], np.arange(w["N"])[None, :], g] = 1.0
    w["target"] = tgt
    s = run_tree_sampled(w)
    t = to_dev(tgt, workloads.F32)
    tok, n, best, nodes = sv.verify_tree(t, i32(w["tree_tokens"]), i32(w["paths"]))
    assert np.array_equal(s["tokens"], tok.cpu().numpy())
    assert np.array_equal(s["accepted_nodes"], nodes.cpu().numpy())
    check_tree_sampled(w, s, oracle_tree_sampled(w), "tree sampled one-hot rows")


def test_tree_sampled_repeated_sibling_tokens_and_no_paths():
    w = _peaked_tree(12, B=4, N=10, L=3, V=500, level_sizes=[5, 4])
    w["tree_tokens"][1, 2] = w["tree_tokens"][1, 1]  # two children of the root share a token
    w["paths"][3] = -1                               # request 3 has no used path
    g = run_tree_sampled(w)
    o = oracle_tree_sampled(w)
    check_tree_sampled(w, g, o, "tree sampled repeated tokens / no paths")
    assert g["num_accepted"][3] == 0 and g["best_path"][3] == -1


def test_tree_sampled_bad_indices_fail_closed_and_workspace_is_reusable():
    ws = sv.Workspace()
    w = _peaked_tree(13, B=4, N=16, L=4, V=3000, level_sizes=[5, 6, 4])
    w["paths"][1, 0, 2] = 16         # node id out of range
    w["tree_tokens"][2, 5] = 3000    # token out of range
    g = run_tree_sampled(w, workspace=ws)
    assert sv.last_error(ws) == sv.SPEC_EBADINDEX
    o = oracle_tree_sampled(w)
    assert o["rc"] == oracle.EBADINDEX
    for b in (1, 2):
        assert g["num_accepted"][b] == -1 and np.all(g["tokens"][b] == -1) and g["best_path"][b] == -1
    keep = [0, 3]
    sub = {key: (v[keep] if isinstance(v, np.ndarray) and v.shape[:1] == (4,) else v) for key, v in w.items()}
    sub["B"] = 2
    check_tree_sampled(sub, {key: v[keep] for key, v in g.items()},
                       {key: (v[keep] if isinstance(v, np.ndarray) else v) for key, v in o.items()},
                       "tree sampled others of a failed batch")
    # the same workspace then serves other calls correctly
    w2 = _peaked_tree(14, B=3, N=20, L=4, V=6000, level_sizes=[6, 7, 6])
    check_tree_sampled(w2, run_tree_sampled(w2, workspace=ws), oracle_tree_sampled(w2), "tree sampled reuse")
    wc = workloads.make("chain_b64_k7_v128256_bf16", seed=15, B=3, V=9000)
    from test_gpu_parity import check_chain, run_chain
    check_chain(wc, run_chain(wc, workspace=ws), oracle.verify(wc), "chain after tree sampled")
    check_tree_sampled(w2, run_tree_sampled(w2, workspace=ws), oracle_tree_sampled(w2), "tree sampled again")
