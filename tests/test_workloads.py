"""The seeded input generator: determinism, shapes, bf16 rounding, tree shape."""
import numpy as np
import torch

import workloads


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100_000) * 50).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.00390625, 1.01171875]  # exact ties to even
    ours = workloads.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(workloads.bf16_bits_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_chain_deterministic_and_shaped():
    a = workloads.make("chain_b8_k4_v32000_f32", seed=3, V=2000)
    b = workloads.make("chain_b8_k4_v32000_f32", seed=3, V=2000)
    for key in ("target", "draft", "draft_tokens", "uniforms", "seq_lens"):
        assert np.array_equal(a[key], b[key])
    assert a["target"].shape == (8, 5, 2000) and a["draft"].shape == (8, 4, 2000)
    assert a["draft_tokens"].dtype == np.int32 and a["draft_tokens"].max() < 2000
    assert np.all((a["uniforms"] >= 0) & (a["uniforms"] < 1))
    assert np.all((a["seq_lens"] >= 128) & (a["seq_lens"] <= 2048))
    c = workloads.make("chain_b8_k4_v32000_f32", seed=4, V=2000)
    assert not np.array_equal(a["target"], c["target"])


def test_bf16_chain_draft_is_noisy_target():
    w = workloads.make("chain_b64_k7_v128256_bf16", seed=0, B=2, V=4096)
    t = workloads.bf16_bits_to_f32(w["target"])
    d = workloads.bf16_bits_to_f32(w["draft"])
    diff = d - t[:, :7]
    assert 0.5 < diff.std() < 0.9  # N(0, 0.7^2) noise plus bf16 rounding
    assert w["target"].dtype == np.uint16


def test_tree_shape():
    w = workloads.make("tree_b16_n60_l4_v151936_bf16", seed=1, B=3, V=512)
    assert w["paths"].shape == (3, 60, 4) and w["tree_tokens"].shape == (3, 60)
    for b in range(3):
        parent = w["parents"][b]
        kids = np.bincount(parent[1:], minlength=60)
        assert kids.max() <= 8 and kids[0] == 8
        depth = np.zeros(60, int)
        for n in range(1, 60):
            depth[n] = depth[parent[n]] + 1
        assert list(np.bincount(depth)) == [1, 8, 25, 26]
        for n in range(60):  # sibling tokens are distinct
            sib = [w["tree_tokens"][b, m] for m in range(1, 60) if parent[m] == n]
            assert len(sib) == len(set(sib))
        used = w["paths"][b][w["paths"][b, :, 0] == 0]
        assert len(used) == int(np.sum(kids == 0))
        for row in used:
            nodes = [v for v in row if v >= 0]
            assert all(parent[nodes[i + 1]] == nodes[i] for i in range(len(nodes) - 1))
