import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.join(ROOT, "tests")):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C ABI)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near-tie bookkeeping of the stochastic parity cases: every case's
    flagged and mismatched counts (a mismatch is allowed only at a flagged
    near-tie, and is then checked to be a valid outcome of the other side of
    the tie), one line per full-size workload and a total."""
    import _report
    recs = [r for r in _report.RECORDS if r.get("kind") in ("chain", "filtered")]
    if not recs:
        return
    tr = terminalreporter
    tr.section("near-tie parity report")
    tot = {key: sum(r[key] for r in recs) for key in ("requests", "flagged", "mismatched")}
    tr.write_line(f"{len(recs)} stochastic cases, {tot['requests']} requests: "
                  f"{tot['flagged']} flagged, {tot['mismatched']} mismatched (each one flagged and valid)")
    tied = sum(r.get("tied_pq", 0) for r in recs)
    if tied:
        tr.write_line(f"  {tied} p/q entries beyond 1e-5 on rows whose filter cut the oracle flags "
                      f"(either kept set valid)")
    for r in recs:
        if r.get("full_size"):
            tr.write_line(f"  {r['case']}: {r['requests']} requests, {r['flagged']} flagged "
                          f"({r['flagged'] / r['requests']:.1%}), {r['mismatched']} mismatched, "
                          f"max p/q rel err {r.get('max_prob_rel_err', 0.0):.2e}")
    path = os.environ.get("SPEC_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump(_report.RECORDS, f, indent=1)
