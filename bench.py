#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verification row on GB300.

One step = one verify call over one batch (chain: both passes plus the fused
KV cursor update) on seeded synthetic logits already resident in HBM.  The
headline workload is chain stochastic verify with B=64 requests, k=7 drafts,
V=128256, bf16 logits, T=0.7.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm

Under torchrun each rank verifies its own batch on its own GPU (weak scaling,
no collective on the data path); the timed region is bracketed by barriers
and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verified positions/sec and achieved HBM GB/s (B=64,k=7,V=128256 bf16)"
PREQUEUE = 3  # untimed calls queued right before the timed region
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "speculative_decoding_verification_row_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=workloads.HEADLINE, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--greedy", action="store_true", help="greedy chain verify instead of stochastic")
    ap.add_argument("--sampled", action="store_true",
                    help="tree workloads: the stochastic tree verify instead of the greedy one")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--philox", action="store_true",
                    help="chain: draw each request's uniforms in the kernel from a (seed, offset) Philox state")
    ap.add_argument("--top-k", type=int, default=0,
                    help="stochastic chain on top-k / top-p / min_p filtered rows (0: no top-k)")
    ap.add_argument("--top-p", type=float, default=1.0)
    ap.add_argument("--min-p", type=float, default=0.0)
    ap.add_argument("--op", choices=["verify", "relocate"], default="verify",
                    help="relocate: time the accepted-KV relocation after a tree verify instead")
    ap.add_argument("--kv-row-bytes", type=int, default=131072,
                    help="relocate: bytes of one token's KV row (32 layers x K,V x 8 heads x 128 x bf16)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) stamped on arrival."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.samples = []
        self.proc = None
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return
        self.proc = subprocess.Popen(
            [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", str(index),
             "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi not found"}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = None
        if not inside:  # region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:3]
            inside = [s for _, s in near]
            note = "timed region shorter than the sampling period; nearest samples used"
        sm = [float(s[0]) for s in inside if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        out = {"sm_mhz": float(np.median(sm)) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# --------------------------------------------------------------------- helpers
def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def csrc_digest(files=None) -> str:
    """sha256 of the named csrc files (all of csrc/ when None)."""
    h = hashlib.sha256()
    for name in sorted(files) if files else sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()


def recorded_traffic(key: str):
    """DRAM bytes per call from the committed ncu summary, if taken on this source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("csrc_sha256") != csrc_digest(rec.get("files")):
        return None
    return rec.get("dram_bytes_per_call")


def reduce_max(x: float, dist, device) -> float:
    """The largest value of x over all ranks (x itself on one process)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, positions_per_rank: int, ms_step_max: float) -> float:
    """Whole-job verified positions per second: every rank verifies its own
    batch each step (weak scaling), and a step lasts as long as the slowest
    rank's."""
    return world * positions_per_rank / (ms_step_max * 1e-3)


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch."""
    return seed + 1000 * rank


def positions_per_call(w, greedy):
    return w["B"] * (w["L"] - 1) if w["kind"] == "tree" else w["B"] * w["k"]


def dev_logits(arr, dtype, device):
    import torch
    if dtype == workloads.BF16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


# --------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch
    import speculative_decoding_verification_row_gb300 as sv

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    w = workloads.make(args.config, seed=rank_seed(args.seed, rank))
    tree = w["kind"] == "tree"
    sampled = tree and args.sampled
    greedy = args.greedy and not tree
    filtered = is_filtered(args) and not (tree or greedy)
    wide = filtered and (args.top_k == 0 or args.top_k > sv.SPEC_MAX_TOPK)
    if filtered:
        # The draft argmax is in every kept set (top_k >= 1, top_p > 0).
        w["draft_tokens"] = filtered_draft_tokens(w)
    lib = sv.lib()
    stream = torch.cuda.current_stream(device)
    sh = ctypes.c_void_p(stream.cuda_stream)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)  # noqa: E731
    code = workloads.DTYPE_CODE[w["dtype"]]
    B, V = w["B"], w["V"]

    # Two resident copies of the inputs, used alternately: each step reads
    # logits the previous step did not touch (2x the input size > L2).
    copies = []
    for _ in range(2):
        c = {"target": dev_logits(w["target"], w["dtype"], device)}
        if tree:
            c["tree_tokens"], c["paths"] = i32(w["tree_tokens"]), i32(w["paths"])
            c["uniforms"] = torch.from_numpy(w["uniforms"]).to(device)
        else:
            c["tokens"] = i32(w["draft_tokens"])
            if not greedy:
                c["draft"] = dev_logits(w["draft"], w["dtype"], device)
                c["uniforms"] = torch.from_numpy(w["uniforms"]).to(device)
                c["seeds"] = torch.full((w["B"],), 1234, dtype=torch.int64, device=device)
                c["offsets"] = torch.arange(w["B"], dtype=torch.int64, device=device) * 4096
        copies.append(c)
    seq = i32(w["seq_lens"])
    k = w["L"] - 1 if tree else w["k"]
    rows = w["N"] if tree else (k + 1 if greedy else 2 * k + 1)
    ws = sv.Workspace(device)
    buf = ws.ensure(B, rows, V, sh,
                    lib.spec_workspace_size_filtered(B, k, V, args.top_k) if filtered else None)
    out_tok = torch.empty((B, w["L"] if tree else k + 1), dtype=torch.int32, device=device)
    out_n = torch.empty(B, dtype=torch.int32, device=device)
    P = ctypes.c_void_p
    ptr = lambda t: P(t.data_ptr())  # noqa: E731
    call_args = []
    for c in copies:
        if sampled:
            best = torch.empty(B, dtype=torch.int32, device=device)
            nodes = torch.empty((B, w["L"]), dtype=torch.int32, device=device)
            fn = lib.spec_verify_tree_sampled
            call_args.append((ptr(c["target"]), code, ptr(c["tree_tokens"]), ptr(c["paths"]),
                              ptr(c["uniforms"]), ctypes.c_float(w["temperature"]), B, w["N"], w["P"],
                              w["L"], V, ptr(out_tok), ptr(out_n), ptr(best), ptr(nodes), ptr(seq),
                              ptr(buf), buf.numel(), sh))
        elif tree:
            best = torch.empty(B, dtype=torch.int32, device=device)
            nodes = torch.empty((B, w["L"]), dtype=torch.int32, device=device)
            fn = lib.spec_verify_tree
            call_args.append((ptr(c["target"]), code, ptr(c["tree_tokens"]), ptr(c["paths"]), B, w["N"],
                              w["P"], w["L"], V, ptr(out_tok), ptr(out_n), ptr(best), ptr(nodes),
                              ptr(seq), ptr(buf), buf.numel(), sh))
        elif greedy:
            fn = lib.spec_verify_greedy
            call_args.append((ptr(c["target"]), code, ptr(c["tokens"]), B, k, V, ptr(out_tok),
                              ptr(out_n), ptr(seq), ptr(buf), buf.numel(), sh))
        elif filtered:
            fn = lib.spec_verify_chain_ex
            prm = sv.ChainParams(ctypes.sizeof(sv.ChainParams), ptr(c["target"]), ptr(c["draft"]), code,
                                 ptr(c["tokens"]), None, None if args.philox else ptr(c["uniforms"]),
                                 ptr(c["seeds"]) if args.philox else None,
                                 ptr(c["offsets"]) if args.philox else None, w["temperature"], B, k, V,
                                 ptr(out_tok), ptr(out_n), None, ptr(seq), args.top_k, args.top_p,
                                 args.min_p)
            c["params"] = prm
            call_args.append((ctypes.byref(prm), ptr(buf), buf.numel(), sh))
        elif args.philox:
            fn = lib.spec_verify_chain_philox
            call_args.append((ptr(c["target"]), ptr(c["draft"]), code, ptr(c["tokens"]),
                              ptr(c["seeds"]), ptr(c["offsets"]), ctypes.c_float(w["temperature"]),
                              B, k, V, ptr(out_tok), ptr(out_n), None, ptr(seq), ptr(buf),
                              buf.numel(), sh))
        else:
            fn = lib.spec_verify_chain
            call_args.append((ptr(c["target"]), ptr(c["draft"]), code, ptr(c["tokens"]),
                              ptr(c["uniforms"]), ctypes.c_float(w["temperature"]), B, k, V,
                              ptr(out_tok), ptr(out_n), None, ptr(seq), ptr(buf), buf.numel(), sh))
    # pass 1 and its programmatic-dependent finish/draw grid; the wide filter
    # as wide_launches counts it
    launches_per_step = wide_launches(w, args, torch.cuda.get_device_properties(device).multi_processor_count) \
        if wide else 2

    for i in range(args.warmup):
        rc = fn(*call_args[i & 1])
        assert rc == 0, sv.status_string(rc)
    torch.cuda.synchronize()
    n_first = out_n.cpu().numpy()
    assert sv.last_error(ws) == sv.SPEC_OK

    clocks = ClockSampler(local)
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    # A few untimed calls queued right before the start event: the GPU is
    # busy (clocks up, the host ahead of it) when the timed region starts, so
    # it holds K calls back to back, as in a serving loop.
    bad = 0
    for i in range(PREQUEUE):
        bad |= fn(*call_args[i & 1])
    start.record(stream)
    for i in range(args.steps):
        bad |= fn(*call_args[(PREQUEUE + i) & 1])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    if dist:
        dist.barrier()
    clocks.stop()
    assert bad == 0
    ms_step = reduce_max(start.elapsed_time(end), dist, device) / args.steps
    # Per-step distribution, measured apart: an event after every step (each
    # event adds its own cost to the step it closes, so these read high).
    events = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    for i in range(PREQUEUE):
        fn(*call_args[i & 1])
    events[0].record(stream)
    for i in range(args.steps):
        fn(*call_args[(PREQUEUE + i) & 1])
        events[i + 1].record(stream)
    torch.cuda.synchronize()
    step_ms = [events[i].elapsed_time(events[i + 1]) for i in range(args.steps)]
    ms_median = reduce_max(float(np.median(step_ms)), dist, device)

    # End to end through the public binding: pinned host inputs copied in and
    # results read back inside every step.
    host = {key: torch.from_numpy(np.ascontiguousarray(
        w[key].view(np.int16) if (w["dtype"] == workloads.BF16 and key in ("target", "draft")) else w[key])).pin_memory()
        for key in ((["target", "tree_tokens", "paths"] + (["uniforms"] if sampled else [])) if tree else
                    ["target", "draft_tokens"] + ([] if greedy else ["draft", "uniforms"]))}
    host["seq_lens"] = torch.from_numpy(w["seq_lens"].copy()).pin_memory()
    dev_in = {key: torch.empty(t.shape, dtype=t.dtype, device=device) for key, t in host.items()}
    res_tok = torch.empty(tuple(out_tok.shape), dtype=torch.int32).pin_memory()
    res_n = torch.empty(B, dtype=torch.int32).pin_memory()
    res_seq = torch.empty(B, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (res_tok, res_n, res_seq))

    def e2e_step():
        for key, t in host.items():
            dev_in[key].copy_(t, non_blocking=True)
        lg = (lambda t: t.view(torch.bfloat16)) if w["dtype"] == workloads.BF16 else (lambda t: t)
        if sampled:
            tk, nn, _, _ = sv.verify_tree_sampled(lg(dev_in["target"]), dev_in["tree_tokens"], dev_in["paths"],
                                                  dev_in["uniforms"], w["temperature"],
                                                  seq_lens=dev_in["seq_lens"], workspace=ws)
        elif tree:
            tk, nn, _, _ = sv.verify_tree(lg(dev_in["target"]), dev_in["tree_tokens"], dev_in["paths"],
                                          seq_lens=dev_in["seq_lens"], workspace=ws)
        elif greedy:
            tk, nn = sv.verify_greedy(lg(dev_in["target"]), dev_in["draft_tokens"],
                                      seq_lens=dev_in["seq_lens"], workspace=ws)
        else:
            tk, nn, _ = sv.verify_chain(lg(dev_in["target"]), lg(dev_in["draft"]), dev_in["draft_tokens"],
                                        dev_in["uniforms"], w["temperature"], seq_lens=dev_in["seq_lens"],
                                        workspace=ws, top_k=args.top_k if filtered else 0,
                                        top_p=args.top_p if filtered else 1.0,
                                        min_p=args.min_p if filtered else 0.0)
        res_tok.copy_(tk, non_blocking=True)
        res_n.copy_(nn, non_blocking=True)
        res_seq.copy_(dev_in["seq_lens"], non_blocking=True)
        stream.synchronize()

    te = 0.0
    if args.e2e_steps > 0:
        for _ in range(3):
            e2e_step()
        if dist:
            dist.barrier()
        te0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        te = time.perf_counter() - te0
    if args.e2e_steps > 0:
        te = reduce_max(te, dist, device)

    pos = positions_per_call(w, greedy)
    value = job_throughput(world, pos, ms_step)
    algo_bytes = workloads.algorithmic_bytes(w, greedy=greedy or tree)
    achieved = algo_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_src = peak_hbm()
    kernel_key = ("tree_sampled" if sampled else "tree") if tree else \
        ("greedy" if greedy else (("wide" if wide else "filtered") if filtered else "chain"))
    traffic = recorded_traffic(f"{args.config}/{kernel_key}" + (filter_tag(args) if filtered else ""))
    stats = sv.acceptance_stats(n_first, k)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, greedy, args.cpu_seconds,
                           (args.top_k, args.top_p, args.min_p) if filtered else None, sampled=sampled)

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "ms_per_step_median_evented": ms_median,
        "requests_per_s": world * B / (ms_step * 1e-3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": args.config + ("/greedy" if greedy else "") + ("/sampled" if sampled else "")
                        + ("/philox" if args.philox and not (tree or greedy) else "")
                        + (filter_tag(args) if filtered else ""),
            "B": B, "k": k, "V": V, "logits": w["dtype"],
            "temperature": None if ((tree and not sampled) or greedy) else w["temperature"],
            "requests_per_step": B * world,
            "l2": "inputs larger than L2: two resident copies of the logits used alternately",
            "timing": f"one CUDA event pair around the K steps on the launching stream, {PREQUEUE} untimed "
                      "calls queued before the start event; ms_per_step_median_evented comes from a "
                      "separate pass with an event after every step",
        },
        "achieved_hbm_gbs": achieved,
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
            "kernel": {"chain": "spec_verify_chain call (chain_rowstats_kernel + chain_draw_kernel)",
                       "filtered": "spec_verify_chain_ex call (filter_max_kernel + filter_pick_kernel)",
                       "wide": "spec_verify_chain_ex call (chain_rowstats_kernel + wide_hist_kernel + "
                               "[wide_bins_kernel] + wide_cand_kernel + wide_cut_kernel + wide_draw_kernel; "
                               "min_p alone: no bins, no candidates)",
                       "greedy": "spec_verify_greedy call (argmax_kernel + argmax_finish_kernel)",
                       "tree": "spec_verify_tree call (argmax_kernel + argmax_finish_kernel)",
                       "tree_sampled": "spec_verify_tree_sampled call (chain_rowstats_kernel + tree_draw_kernel)"}[kernel_key],
            "algorithmic_bytes_per_call": algo_bytes,
        },
        "e2e": {"value": job_throughput(world, pos, 1e3 * te / args.e2e_steps), "unit": "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps} if args.e2e_steps > 0 else None,
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_untimed_prequeued": launches_per_step * PREQUEUE,
        "clocks": clocks.summary(t0, t1),
        "acceptance": stats,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def wide_launches(w, args, sms: int) -> int:
    """Grids one per-row-cut verify launches (the rule of wide.cu's launch):
    pass 1, the histogram, the bins grid when a row's slices are split over
    several histogram CTAs (up to 8 slices of 2048 16-byte vectors per CTA,
    as many as keep the grid at 4 CTAs per SM), the candidates, the cut and
    the draw; min_p alone has no bins and no candidates."""
    if args.top_k == 0 and args.top_p >= 1.0 and args.min_p > 0.0:
        return 4
    es = 2 if w["dtype"] == workloads.BF16 else 4
    nvec = w["V"] * es // 16 if (w["V"] * es) % 16 == 0 else w["V"]  # (the bench's rows are aligned)
    nsplit = -(-nvec // 2048)
    rows = w["B"] * (2 * w["k"] + 1)
    spc = max(1, min(8, rows * nsplit // (4 * sms)))
    return 6 if -(-nsplit // spc) > 1 else 5


def is_filtered(args):
    return args.top_k > 0 or args.top_p < 1.0 or args.min_p > 0.0


def filter_tag(args):
    return f"/top_k={args.top_k},top_p={args.top_p:g}" + (f",min_p={args.min_p:g}" if args.min_p > 0 else "")


def filtered_draft_tokens(w):
    """Draft tokens of a filtered run: each draft row's argmax (lowest index
    on ties), which every top-k / top-p kept set contains."""
    d = w["draft"]
    x = workloads.bf16_bits_to_f32(d) if w["dtype"] == workloads.BF16 else d
    return np.argmax(x, axis=-1).astype(np.int32)


def cpu_baseline(w, greedy, seconds, filt=None, sampled=False):
    import oracle
    reps, t0 = 0, time.perf_counter()
    while True:
        if sampled:
            oracle.verify_tree_sampled(w["target"], w["tree_tokens"], w["paths"], w["uniforms"],
                                       w["temperature"], w["dtype"])
        elif filt:
            oracle.verify_chain_filtered(w["target"], w["draft"], w["draft_tokens"], w["uniforms"],
                                         w["temperature"], filt[0], float(np.float32(filt[1])), w["dtype"],
                                         min_p=float(np.float32(filt[2])))
        else:
            oracle.verify(w, greedy=greedy)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    pos = positions_per_call(w, greedy) * reps
    return {"value": pos / el, "unit": "positions/s", "cores": 1, "kind": "oracle",
            "requests_per_s": w["B"] * reps / el, **host_cpu(),
            "sample": f"the full batch ({w['B']} requests) verified {reps} times by the single-threaded "
                      f"fp64 oracle ({el:.1f} s)"}


def host_cpu():
    """The host's logical CPU count and model name (the oracle uses one thread)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model"):
                    model = line.split(":", 1)[1].strip()
                    break
        if model is None:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"host_nproc": os.cpu_count(), "host_cpu_model": model}


# --------------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """The CPU oracle timed as the reference arm: each step verifies one
    request of the workload (cycling through the batch)."""
    if rank != 0:
        return
    import oracle
    w = workloads.make(args.config, seed=args.seed)
    tree = w["kind"] == "tree"
    sampled = tree and args.sampled
    greedy = args.greedy and not tree
    filtered = is_filtered(args) and not (tree or greedy)
    if filtered:
        w["draft_tokens"] = filtered_draft_tokens(w)

    def one(b):
        sub = {key: (v[b:b + 1] if isinstance(v, np.ndarray) and v.shape[:1] == (w["B"],) else v)
               for key, v in w.items()}
        sub["B"] = 1
        if sampled:
            return oracle.verify_tree_sampled(sub["target"], sub["tree_tokens"], sub["paths"],
                                              sub["uniforms"], sub["temperature"], sub["dtype"])
        if filtered:
            return oracle.verify_chain_filtered(sub["target"], sub["draft"], sub["draft_tokens"],
                                                sub["uniforms"], sub["temperature"], args.top_k,
                                                float(np.float32(args.top_p)), sub["dtype"],
                                                min_p=float(np.float32(args.min_p)))
        return oracle.verify(sub, greedy=greedy)

    for i in range(args.warmup):
        one(i % w["B"])
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i % w["B"])
    el = time.perf_counter() - t0
    per = (w["L"] - 1) if tree else w["k"]
    value = per * args.steps / el
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.config + ("/greedy" if greedy else "") + ("/sampled" if sampled else "")
                               + (filter_tag(args) if filtered else ""),
                   "B": w["B"],
                   "k": per, "V": w["V"], "logits": w["dtype"]},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": 1, "kind": "oracle",
                         "requests_per_s": args.steps / el, **host_cpu(),
                         "sample": "one request per step, cycling through the batch"},
        "requests_per_s": args.steps / el,
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_relocate(args, rank, world, local):
    """Accepted-KV relocation after the tree verify of a tree workload: a paged
    pool of --kv-row-bytes rows, 32 tokens per block, block tables shuffled."""
    import torch
    import speculative_decoding_verification_row_gb300 as sv

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    name = args.config if workloads.CONFIGS[args.config]["kind"] == "tree" else "tree_b16_n60_l4_v151936_bf16"
    w = workloads.make(name, seed=rank_seed(args.seed, rank))
    # The accepted nodes come from this batch's tree verify on the GPU (once,
    # before the timed region).
    i32d = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)  # noqa: E731
    _, n_dev, _, nodes_dev = sv.verify_tree(dev_logits(w["target"], w["dtype"], device),
                                            i32d(w["tree_tokens"]), i32d(w["paths"]))
    o = {"accepted_nodes": nodes_dev.cpu().numpy(), "num_accepted": n_dev.cpu().numpy()}
    B, N, L, tpb = w["B"], w["N"], w["L"], 32
    rng = np.random.default_rng(args.seed)
    base = rng.integers(512, 4096, size=B).astype(np.int32)
    max_blocks = (4096 + N + tpb - 1) // tpb + 1
    bt = rng.permutation(B * max_blocks).astype(np.int32).reshape(B, max_blocks)
    rows = B * max_blocks * tpb
    pool = torch.empty((rows, args.kv_row_bytes // 2), dtype=torch.bfloat16, device=device)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)  # noqa: E731
    bt_d, base_d, nodes_d, n_d = d(bt), d(base), nodes_dev, n_dev
    moved = sum(int(np.sum(o["accepted_nodes"][b, 1:o["num_accepted"][b] + 1] != np.arange(1, o["num_accepted"][b] + 1)))
                for b in range(B) if o["num_accepted"][b] > 0)
    algo = 2 * moved * args.kv_row_bytes      # read + write of every moved row
    sv.relocate_accepted_kv(pool, bt_d, base_d, nodes_d, n_d, tpb)  # argument checks once
    lib = sv.lib()
    P = ctypes.c_void_p
    stream = torch.cuda.current_stream(device)
    call = (P(pool.data_ptr()), ctypes.c_size_t(args.kv_row_bytes), tpb, B * max_blocks, P(bt_d.data_ptr()),
            max_blocks, P(base_d.data_ptr()), P(nodes_d.data_ptr()), P(n_d.data_ptr()), B, L,
            P(stream.cuda_stream))
    for _ in range(args.warmup):
        assert lib.spec_relocate_accepted_kv(*call) == 0
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        lib.spec_relocate_accepted_kv(*call)
    end.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * start.elapsed_time(end) / args.steps
    peak, src = peak_hbm()
    if rank == 0:
        print(json.dumps({
            "op": "relocate_accepted_kv", "workload": name, "B": B, "L": L, "tokens_per_block": tpb,
            "kv_row_bytes": args.kv_row_bytes, "rows_moved": moved, "us_per_call": us,
            "algorithmic_bytes_per_call": algo, "achieved_gbs": algo / (us * 1e-6) / 1e9,
            "frac_of_peak": algo / (us * 1e-6) / 1e9 / peak, "peak_gbs": peak, "peak_source": src,
            "steps": args.steps, "warmup": args.warmup,
        }), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.op == "relocate":
        run_relocate(args, rank, world, local)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
