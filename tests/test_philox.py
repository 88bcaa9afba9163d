"""Per-request Philox uniforms (TensorRT-LLM walkthrough, rejection-sampling
section: chain_speculative_sampling keeps a (seed, offset) Philox state per
request).  The oracle's Philox4x32-10 is pinned to the generator's published
known-answer vectors; the CUDA generator and the in-kernel draw are checked
against the oracle on the GPU."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def test_philox_known_answers():
    kat = json.load(open(os.path.join(HERE, "golden", "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        h = lambda xs: [int(x, 16) for x in xs]  # noqa: E731
        assert oracle.philox4x32_10(h(v["ctr"]), h(v["key"])).tolist() == h(v["out"])


def test_uniform_mapping_uses_the_stated_counter_and_word():
    seeds = np.array([0x0123456789ABCDEF, 7], dtype=np.uint64)
    offsets = np.array([0xFEDCBA9876543210, 0], dtype=np.uint64)
    u = oracle.philox_uniforms(seeds, offsets, 9)
    for b in range(2):
        key = [int(seeds[b]) & 0xFFFFFFFF, int(seeds[b]) >> 32]
        for i in range(9):
            ctr = [int(offsets[b]) & 0xFFFFFFFF, int(offsets[b]) >> 32, i // 4, 0]
            word = int(oracle.philox4x32_10(ctr, key)[i % 4])
            assert u[b, i] == np.float32((word >> 8) / 2.0**24)


def test_uniforms_are_uniform_and_streams_distinct():
    rng = np.random.default_rng(3)
    B, n = 4096, 16
    seeds = np.full(B, 1234, dtype=np.uint64)               # constant seed, as the page allows
    offsets = rng.integers(0, 2**62, size=B, dtype=np.uint64)
    u = oracle.philox_uniforms(seeds, offsets, n)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * 2**24 == np.floor(u * 2**24))         # multiples of 2^-24
    counts = np.histogram(u.ravel(), bins=64, range=(0, 1))[0]
    expect = u.size / 64
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 120.0                                      # 63 dof: p ~ 1e-5
    # distinct offsets give distinct streams; equal states give equal streams
    assert len({tuple(r) for r in u[:256].tolist()}) == 256
    again = oracle.philox_uniforms(seeds[:8], offsets[:8], n)
    assert np.array_equal(again, u[:8])
    other_seed = oracle.philox_uniforms(seeds[:8] + np.uint64(1), offsets[:8], n)
    assert not np.array_equal(other_seed, u[:8])


# ------------------------------------------------------------------ GPU
@pytest.mark.gpu
def test_cuda_philox_uniforms_bit_exact():
    import speculative_decoding_verification_row_gb300 as sv
    rng = np.random.default_rng(5)
    B, n = 1000, 65
    seeds = rng.integers(-2**63, 2**63 - 1, size=B, dtype=np.int64)
    offsets = rng.integers(-2**63, 2**63 - 1, size=B, dtype=np.int64)
    got = sv.philox_uniforms(torch.from_numpy(seeds).cuda(), torch.from_numpy(offsets).cuda(), n)
    want = oracle.philox_uniforms(seeds.view(np.uint64), offsets.view(np.uint64), n)
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.gpu
@pytest.mark.parametrize("name,over", [("chain_b1_k4_v1024_f32", {}),
                                       ("chain_b64_k7_v128256_bf16", dict(B=12, V=40000)),
                                       ("chain_b256_k3_v129280_bf16", dict(B=32, V=20000))])
def test_chain_philox_matches_oracle(name, over):
    import speculative_decoding_verification_row_gb300 as sv
    from test_gpu_parity import check_chain, to_dev, i32
    w = workloads.make(name, seed=21, **over)
    B, k = w["B"], w["k"]
    rng = np.random.default_rng(21)
    seeds = np.full(B, 0x5EED, dtype=np.int64)
    offsets = rng.integers(0, 2**40, size=B, dtype=np.int64)
    w["uniforms"] = oracle.philox_uniforms(seeds.view(np.uint64), offsets.view(np.uint64), k + 1)
    seq = i32(w["seq_lens"])
    tok, n, probs = sv.verify_chain(to_dev(w["target"], w["dtype"]), to_dev(w["draft"], w["dtype"]),
                                    i32(w["draft_tokens"]), None, w["temperature"], want_probs=True,
                                    seq_lens=seq, seeds=torch.from_numpy(seeds).cuda(),
                                    offsets=torch.from_numpy(offsets).cuda())
    torch.cuda.synchronize()
    g = dict(tokens=tok.cpu().numpy(), num_accepted=n.cpu().numpy(), probs=probs.cpu().numpy(),
             seq_lens=seq.cpu().numpy())
    check_chain(w, g, oracle.verify(w), f"philox {name}")
