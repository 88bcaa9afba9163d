"""The GPU parity checker on planted results (CPU only): the oracle's own
outputs pass; a flagged final draw resolved to the neighbouring token passes;
an unflagged change, a flagged draw moved outside its window, and a flagged
accept test resolved the other way with a wrong final token all fail."""
import numpy as np
import pytest

import _report
import oracle
from test_gpu_parity import check_chain, draw_allowed


@pytest.fixture(autouse=True)
def _planted_cases_are_not_reported():
    n = len(_report.RECORDS)
    yield
    del _report.RECORDS[n:]


def _case():
    # Bonus draws (identical rows accept every draft) with u placed next to
    # CDF boundaries of p_k, and a request whose first accept test sits
    # 3e-6 below p/q.
    rng = np.random.default_rng(5)
    B, k, V, T = 6, 2, 9, 1.0
    target = (rng.standard_normal((B, k + 1, V)) * 1.2).astype(np.float32)
    draft = target[:, :k].copy()
    draft[5] += (rng.standard_normal((k, V)) * 0.5).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    for b in range(5):
        p = oracle.softmax(target[b, k], T)
        c = np.cumsum(p)
        u[b, k] = np.float32(c[3] + (4e-7 if b % 2 else -4e-7))   # flagged draws
    p = oracle.softmax(target[5, 0], T)
    q = oracle.softmax(draft[5, 0], T)
    u[5, 0] = np.float32(p[x[5, 0]] / q[x[5, 0]] - 3e-6)        # flagged accept test
    w = dict(kind="chain", dtype="f32", B=B, k=k, V=V, target=target, draft=draft,
             draft_tokens=x, uniforms=u, temperature=T, seq_lens=np.arange(B, dtype=np.int32))
    o = oracle.verify(w)
    g = dict(tokens=o["tokens"].copy(), num_accepted=o["num_accepted"].copy(),
             probs=o["probs"].astype(np.float32),
             seq_lens=oracle.rollback(w["seq_lens"], o["num_accepted"], k)["new_lens"])
    return w, o, g


def test_checker_accepts_the_oracle_and_the_other_side_of_a_tie():
    w, o, g = _case()
    assert o["flags"][:5, w["k"]].all() and o["flags"][5, 0]
    check_chain(w, g, o, "exact")
    for b in range(5):  # each flagged draw resolved to the token across the boundary
        t = int(g["tokens"][b, w["k"]])
        other = sorted(draw_allowed(w, b, w["k"]) - {t})
        assert other, "a flagged draw has two tokens in its window"
        g2 = {key: v.copy() for key, v in g.items()}
        g2["tokens"][b, w["k"]] = other[0]
        check_chain(w, g2, o, f"tie {b}")


def test_checker_rejects_planted_mistakes():
    w, o, g = _case()
    k = w["k"]
    bad = {key: v.copy() for key, v in g.items()}
    bad["tokens"][3, k] = (int(bad["tokens"][3, k]) + 4) % w["V"]    # flagged, outside the window
    with pytest.raises(AssertionError):
        check_chain(w, bad, o, "far token")
    o2 = {key: (v.copy() if isinstance(v, np.ndarray) else v) for key, v in o.items()}
    o2["flags"][2, k] = 0                                             # the same change, unflagged
    bad = {key: v.copy() for key, v in g.items()}
    allowed = draw_allowed(w, 2, k) - {int(g["tokens"][2, k])}
    bad["tokens"][2, k] = min(allowed)
    with pytest.raises(AssertionError):
        check_chain(w, bad, o2, "unflagged")
    # the flagged accept test of request 5 resolved as a rejection: the count
    # drops to 0 and the token must be the residual draw of position 0
    n5 = int(o["num_accepted"][5])
    assert n5 >= 1
    alt = draw_allowed(w, 5, 0)
    good = {key: v.copy() for key, v in g.items()}
    good["num_accepted"][5] = 0
    good["tokens"][5] = [min(alt)] + [-1] * k
    good["seq_lens"] = oracle.rollback(w["seq_lens"], good["num_accepted"], k)["new_lens"]
    check_chain(w, good, o, "accept tie, valid")
    wrong = {key: v.copy() for key, v in good.items()}
    wrong["tokens"][5, 0] = next(t for t in range(w["V"]) if t not in alt)
    with pytest.raises(AssertionError):
        check_chain(w, wrong, o, "accept tie, wrong token")
