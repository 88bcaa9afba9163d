"""Host-side logic that needs no GPU: the C ABI exports, acceptance
bookkeeping, and the binding's argument checks."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import speculative_decoding_verification_row_gb300 as sv
from speculative_decoding_verification_row_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def libso():
    _build.build()
    return ctypes.CDLL(_build.LIB)


def _declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(spec_[a-z_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(libso):
    declared = _declared_functions()
    assert set(declared) == set(sv.SYMBOLS), declared
    for name in declared:
        assert hasattr(libso, name), f"{name} not exported"


def test_workspace_size_and_status_strings(libso):
    libso.spec_workspace_size.restype = ctypes.c_size_t
    libso.spec_status_string.restype = ctypes.c_char_p
    assert libso.spec_workspace_size(0, 3, 100) == 0
    assert libso.spec_workspace_size(2, 3, 1) == 0
    a = libso.spec_workspace_size(64, 15, 128256)
    b = libso.spec_workspace_size(64, 15, 1000)
    assert a > b > 0 and a % 256 == 0
    assert libso.spec_status_string(-2) == b"token or node id out of range"
    assert libso.spec_status_string(0) == b"ok"
    # filtered: kept lists up to SPEC_MAX_TOPK, per-row cuts beyond (and
    # without top-k): the chain's layout plus 24 KB of histogram, a 64-byte
    # record and a 16 KB candidate list per row
    f = libso.spec_workspace_size_filtered
    f.restype = ctypes.c_size_t
    rows = 64 * 15
    assert f(64, 7, 128256, -1) == 0
    wide = f(64, 7, 128256, 0)
    assert wide == f(64, 7, 128256, 257) == f(64, 7, 128256, 100000)
    assert wide >= a + rows * (2048 * 12 + 64 + 4096 * 4)
    assert 0 < f(64, 7, 128256, 256) != wide


def test_invalid_arguments_rejected_before_launch(libso):
    """Host-detectable errors return before any CUDA call (no GPU here)."""
    f = libso.spec_verify_chain
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, I, P, P, ctypes.c_float, I, I, I, P, P, P, P, P, ctypes.c_size_t, P]
    dummy = ctypes.c_void_p(4096)
    ok = dict(t=dummy, d=dummy, dt=1, x=dummy, u=dummy, T=0.7, B=2, k=3, V=100)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["t"], a["d"], a["dt"], a["x"], a["u"], a["T"], a["B"], a["k"], a["V"],
                 dummy, dummy, None, None, dummy, 1 << 30, None)

    assert call(T=0.0) == sv.SPEC_EINVAL
    assert call(T=float("nan")) == sv.SPEC_EINVAL
    assert call(T=float("inf")) == sv.SPEC_EINVAL
    assert call(k=0) == sv.SPEC_EINVAL
    assert call(k=sv.SPEC_MAX_DRAFT + 1) == sv.SPEC_EINVAL
    assert call(V=1) == sv.SPEC_EINVAL
    assert call(B=0) == sv.SPEC_EINVAL
    assert call(dt=7) == sv.SPEC_EINVAL
    assert call(t=None) == sv.SPEC_EINVAL
    small = f(dummy, dummy, 1, dummy, dummy, 0.7, 2, 3, 100, dummy, dummy, None, None, dummy, 16, None)
    assert small == sv.SPEC_EWORKSPACE
    g = libso.spec_verify_tree
    g.argtypes = [P, I, P, P, I, I, I, I, I, P, P, P, P, P, P, ctypes.c_size_t, P]
    assert g(dummy, 1, dummy, dummy, 2, 5, 5, 1, 100, dummy, dummy, None, None, None, dummy,
             1 << 30, None) == sv.SPEC_EINVAL  # L < 2
    assert g(dummy, 1, dummy, dummy, 2, sv.SPEC_MAX_TREE_NODES + 1, 5, 4, 100, dummy, dummy, None,
             None, None, dummy, 1 << 30, None) == sv.SPEC_EINVAL
    r = libso.spec_rollback_lengths
    r.argtypes = [P, P, I, I, P, P, P]
    assert r(None, dummy, 3, 4, dummy, None, None) == sv.SPEC_EINVAL
    assert r(dummy, dummy, 3, 0, dummy, None, None) == sv.SPEC_EINVAL


def test_kestrel_histogram_bookkeeping():
    """The n_ok log of Kestrel article 32, section 3.4, re-derived by the
    benchmark's bookkeeping: 45 rounds, 40 accepted, 0.889 per round, and in
    the article's anchored scheme 64 tokens = 1.422 per round."""
    g = json.load(open(os.path.join(GOLDEN, "kestrel_histogram.json")))
    hist = {int(n): c for n, c in g["histogram"].items()}
    n_acc = np.concatenate([np.full(c, n) for n, c in hist.items()])
    s = sv.acceptance_stats(n_acc, g["k"])
    assert s["rounds"] == g["rounds"] and s["accepted"] == g["accepted"]
    assert round(s["mean_accepted"], 3) == g["mean_accepted"]
    assert s["histogram"] == [hist[n] for n in range(g["k"] + 1)]
    emitted = sv.anchored_emitted(s["histogram"])
    assert emitted == g["tokens_emitted_anchored"]
    assert round(emitted / s["rounds"], 3) == g["tokens_per_round_anchored"]
    # acceptance length two ways (TensorRT-LLM walkthrough, statistics part)
    assert s["acceptance_length"] == pytest.approx(np.mean(n_acc + 1))


def test_binding_rejects_cpu_tensors():
    import torch
    t = torch.zeros(2, 4, 16)
    with pytest.raises((ValueError, RuntimeError)):
        sv.verify_chain(t, t[:, :3], torch.zeros(2, 3, dtype=torch.int32),
                        torch.zeros(2, 4), 1.0)


def test_relocate_rejects_bad_arguments_before_launch():
    import ctypes
    lib = sv.lib()
    P = ctypes.c_void_p
    fake = P(16 * 1024)  # never dereferenced: every check below fails on the host
    z = P(16 * 2048)
    args = dict(pool=fake, row_bytes=64, tpb=16, nblocks=4, bt=z, max_blocks=2, base=z, nodes=z, n=z, B=2, L=4)

    def call(**over):
        a = dict(args, **over)
        return lib.spec_relocate_accepted_kv(a["pool"], ctypes.c_size_t(a["row_bytes"]), a["tpb"], a["nblocks"],
                                             a["bt"], a["max_blocks"], a["base"], a["nodes"], a["n"],
                                             a["B"], a["L"], None)
    assert call(row_bytes=24) == sv.SPEC_EINVAL          # not a multiple of 16
    assert call(row_bytes=0) == sv.SPEC_EINVAL
    assert call(pool=P(16 * 1024 + 8)) == sv.SPEC_EINVAL  # misaligned pool
    assert call(pool=None) == sv.SPEC_EINVAL
    assert call(B=0) == sv.SPEC_EINVAL
    assert call(L=65) == sv.SPEC_EINVAL
    assert call(tpb=0) == sv.SPEC_EINVAL


def test_param_structs_match_the_header(tmp_path):
    # The binding's ctypes mirrors of spec_chain_params / spec_greedy_params
    # must have the header's size and field offsets.
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    fields = {"spec_chain_params": sv.ChainParams, "spec_greedy_params": sv.GreedyParams}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "spec_verify.h"', "int main(void) {"]
    for cname, py in fields.items():
        lines.append(f'  printf("%zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("%zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    want = []
    for py in fields.values():
        want.append(ctypes.sizeof(py))
        want += [getattr(py, f).offset for f, _ in py._fields_]
    assert got == want


def test_bench_counts_the_wide_launches():
    # bench.py's gpu_launches claim for per-row cuts follows wide.cu's launch
    # rule: the bins grid only when a row's slices are split over several
    # histogram CTAs, no bins and no candidates for min_p alone.
    import types
    import bench
    import workloads
    w = dict(B=64, k=7, V=128256, dtype=workloads.BF16)
    args = types.SimpleNamespace(top_k=0, top_p=0.9, min_p=0.0)
    assert bench.wide_launches(w, args, 152) == 5        # 8 slices, one CTA per row
    assert bench.wide_launches(dict(w, B=2), args, 152) == 6  # small batch: rows split
    assert bench.wide_launches(w, types.SimpleNamespace(top_k=1000, top_p=1.0, min_p=0.0), 152) == 5
    assert bench.wide_launches(w, types.SimpleNamespace(top_k=0, top_p=1.0, min_p=0.05), 152) == 4
