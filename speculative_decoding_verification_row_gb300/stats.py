"""Acceptance bookkeeping on the host (no GPU needed).

Acceptance length follows the TensorRT-LLM walkthrough ("statistics" part of
the SpecSampler section): AL = (accepted drafts + requests) / requests, since
every request emits at least one target token.  The acceptance rate is
accepted / proposed (vLLM learning book, section 3).  The histogram of
accepted counts is kept as well, because a mean alone hides the shape (Kestrel
article 32, section 4.3).
"""
from __future__ import annotations

import numpy as np


def acceptance_stats(num_accepted, k: int) -> dict:
    """Summary of per-request accepted counts (failed requests, n < 0, are skipped)."""
    n = np.asarray(num_accepted, dtype=np.int64).ravel()
    n = n[n >= 0]
    rounds = int(n.size)
    accepted = int(n.sum())
    hist = np.bincount(n, minlength=k + 1)[: k + 1] if rounds else np.zeros(k + 1, np.int64)
    return {
        "rounds": rounds,
        "accepted": accepted,
        "mean_accepted": accepted / rounds if rounds else 0.0,
        "acceptance_length": (accepted + rounds) / rounds if rounds else 0.0,
        "acceptance_rate": accepted / (rounds * k) if rounds and k else 0.0,
        "emitted": accepted + rounds,
        "histogram": [int(c) for c in hist],
    }


def anchored_emitted(histogram) -> int:
    """Tokens emitted under the anchored scheme of Kestrel article 32 (section
    2: a round with n >= 1 accepted emits those n drafts only, a round with
    n = 0 emits the target's own token)."""
    return int(sum(max(n, 1) * int(c) for n, c in enumerate(histogram)))
