"""Accepted-KV relocation (TensorRT-LLM walkthrough, the "moving to the right
place" step): oracle pins on the CPU, and the CUDA kernel against the oracle
on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _pool(rows, width, seed=0):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 2**16, size=(rows, width), dtype=np.int64).astype(np.uint16)


# ------------------------------------------------------------------ oracle pins (CPU)
def test_linear_path_moves_nothing():
    # The page: with a linear draft the accepted rows already sit in place.
    pool = _pool(32, 8)
    bt = np.arange(8, dtype=np.int32)[None, :]
    out = oracle.relocate_kv(pool, bt, [5], [[0, 1, 2, 3]], [3], 4)
    assert np.array_equal(out, pool)


def test_hand_example_contiguous():
    # base 2, accepted nodes 0, 3, 5: logical rows 3 <- 5 and 4 <- 7.
    pool = np.arange(16, dtype=np.int64)[:, None] * np.ones((1, 3), dtype=np.int64)
    bt = np.arange(4, dtype=np.int32)[None, :]
    out = oracle.relocate_kv(pool, bt, [2], [[0, 3, 5, -1]], [2], 4)
    want = pool.copy()
    want[3] = 5
    want[4] = 7
    assert np.array_equal(out, want)


def test_hand_example_paged():
    # Two tokens per block; the request's logical blocks 0,1,2,3 live in pool
    # blocks 3,0,2,1.  base 1, nodes 0, 2, 4: logical 2 <- 3 and 3 <- 5.
    pool = np.arange(8, dtype=np.int64)[:, None]
    bt = np.array([[3, 0, 2, 1]], dtype=np.int32)
    phys = lambda t: bt[0, t // 2] * 2 + t % 2  # noqa: E731
    out = oracle.relocate_kv(pool, bt, [1], [[0, 2, 4]], [2], 2)
    want = pool.copy()
    want[phys(2)] = pool[phys(3)]
    want[phys(3)] = pool[phys(5)]
    assert np.array_equal(out, want)
    assert phys(2) == 0 and phys(3) == 1 and phys(5) == 5  # the mapping is not the identity


@pytest.mark.parametrize("nodes,n", [([0, 2, 1, -1], 2),      # not increasing
                                     ([1, 2, 3, -1], 2),      # does not start at the root
                                     ([0, 2, 3, -1], -1),     # failed closed
                                     ([0, 2, 3, 5], 4),       # n >= L
                                     ([0, 2, 30, -1], 2)])    # reads past the mapped blocks
def test_untouched_requests(nodes, n):
    pool = _pool(16, 4)
    bt = np.arange(4, dtype=np.int32)[None, :]
    out = oracle.relocate_kv(pool, bt, [1], [nodes], [n], 4)
    assert np.array_equal(out, pool)


def test_in_place_increasing_order_equals_the_gather():
    # The kernel moves rows in place in increasing j; that equals the gather
    # from the original rows whenever the path starts at 0 and increases.
    rng = np.random.default_rng(7)
    for _ in range(200):
        L = int(rng.integers(2, 9))
        n = int(rng.integers(1, L))
        path = np.concatenate([[0], np.sort(rng.choice(np.arange(1, 40), size=n, replace=False))])
        pool = _pool(64, 2, seed=int(rng.integers(1 << 30)))
        base = int(rng.integers(0, 64 - 41))
        want = oracle.relocate_kv(pool, np.arange(16, dtype=np.int32)[None, :], [base],
                                  [np.concatenate([path, -np.ones(L - n - 1, dtype=np.int64)])], [n], 4)
        got = pool.copy()
        for j in range(1, n + 1):
            got[base + j] = got[base + path[j]]
        assert np.array_equal(got, want)


# ------------------------------------------------------------------ GPU parity
def _tree_case(B, row_bytes, tpb, seed):
    w = workloads.make("tree_b16_n60_l4_v151936_bf16", seed=seed, B=B, V=4096)
    o = oracle.verify(w)
    N, L = w["N"], w["L"]
    rng = np.random.default_rng(seed)
    base = rng.integers(0, 300, size=B).astype(np.int32)
    max_blocks = (300 + N + tpb - 1) // tpb + 1
    nblocks = B * max_blocks
    bt = rng.permutation(nblocks).astype(np.int32).reshape(B, max_blocks)
    width = row_bytes // 2
    pool = _pool(nblocks * tpb, width, seed=seed + 1)
    return pool, bt, base, o["accepted_nodes"].astype(np.int32), o["num_accepted"].astype(np.int32), L


@pytest.mark.gpu
@pytest.mark.parametrize("row_bytes,tpb", [(16, 1), (4096 + 48, 16), (16384, 8)])
def test_relocate_matches_oracle(row_bytes, tpb):
    import speculative_decoding_verification_row_gb300 as sv
    pool, bt, base, nodes, n, L = _tree_case(16, row_bytes, tpb, seed=row_bytes % 97)
    # edge cases on top of the tree's own results
    n[0] = 0                                   # nothing accepted
    n[1] = -1                                  # failed closed
    bt[2, (int(base[2]) + 1) // tpb] = -1      # an unmapped block in the window
    want = oracle.relocate_kv(pool, bt, base, nodes, n, tpb)
    d = torch.from_numpy(pool.view(np.int16)).cuda()
    sv.relocate_accepted_kv(d, torch.from_numpy(bt).cuda(), torch.from_numpy(base).cuda(),
                            torch.from_numpy(nodes).cuda(), torch.from_numpy(n).cuda(), tpb)
    torch.cuda.synchronize()
    got = d.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert (n > 0).sum() >= 8 and not np.array_equal(want, pool)  # rows really moved
