"""Acceptance statistics over verification rounds (host-side bookkeeping).

Definitions follow the pages' counters:
  mean_accepted     accepted drafts per round, the "per-round acceptance
                    (out of K)" of mini-sglang PR #134, Accuracy Tests;
  tokens_per_pass   tokens emitted per target verify pass (accepted + 1), the
                    "tokens / target pass" of the spec-decode README;
  acceptance_rate   mean_accepted / K, the spec-decode README's "acceptance
                    rate" (its CLI example: (3.840 - 1) / 4 = 0.710);
  speedup           tokens_per_pass / (1 + K * c) with c the draft/target cost
                    ratio, the spec-decode README's cost model (3.840 / 1.4 =
                    2.74x at c = 0.1, k = 4).
"""

from __future__ import annotations

import numpy as np


def acceptance_stats(num_accepted, K):
    n = np.asarray(num_accepted, dtype=np.float64).ravel()
    rounds = int(n.size)
    tokens = float(np.sum(n + 1.0))
    mean_acc = float(n.mean()) if rounds else 0.0
    return {
        "rounds": rounds,
        "tokens": tokens,
        "mean_accepted": mean_acc,
        "tokens_per_pass": tokens / rounds if rounds else 0.0,
        "acceptance_rate": (mean_acc / K) if (rounds and K > 0) else 0.0,
    }


def tokens_per_pass(tokens, target_passes):
    return float(tokens) / float(target_passes)


def acceptance_rate_from_tokens_per_pass(tpp, K):
    return (float(tpp) - 1.0) / float(K)


def speedup(tpp, K, draft_cost):
    return float(tpp) / (1.0 + float(K) * float(draft_cost))
