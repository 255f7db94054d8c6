"""Float64/integer CPU oracle for the step after a verify call: stop-set and
max-new-tokens truncation, and per-request acceptance counters.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / --impl reference legs use this module. It shares no code with
the CUDA library.

Sources (page title and section):
[MS] mini-sglang PR #134 "[Feature] Vanilla speculative decoding", Known
     limitations: stopping on a single EOS id differs from generation with a
     multi-token stop set (e.g. Llama-3's end-of-turn and end-of-text ids);
     Modifications (engine.py): cumulative accept_length (tau) and
     accept_rate (alpha) counters.
[SD] spec-decode README, CLI output: tokens per target pass and acceptance
     rate over a run (5000 tokens in 1302 passes: 3.840 tokens/pass, and
     (3.840 - 1) / 4 = 0.710 with k = 4).

Readings taken (the pages give the quantities, not the bookkeeping):
  * a verify call emits tokens[0..n] (n = num_accepted); the request stops at
    the first emitted token that is in the stop set, which is itself kept;
  * max_new[b] (if given) caps the tokens the call may keep, clamped at 0;
  * kept = min(n + 1, first stop index + 1, cap); positions kept..n are
    cleared (token -1, log-prob 0, mu 0; tree node -1);
  * status bit STOPPED (64) when a stop token is among the kept tokens,
    CAPPED (128) when the cap removed at least one emitted token;
  * counters[b] accumulate (rounds, drafts offered, drafts accepted, tokens
    kept): one round per call, K drafts offered by a chain (max_depth by a
    tree), n accepted as decided by the rule (before truncation), kept tokens.
    tau = kept / rounds (tokens per target pass) and alpha = accepted /
    offered ((tau - 1) / k when nothing is truncated, as in [SD]).

Parity status: pinned by tests/test_oracle_finish.py (hand-derived cases,
and the [SD] numbers through the counters).
"""

from __future__ import annotations

import numpy as np

STATUS_STOPPED = 64
STATUS_CAPPED = 128


def finish(out, stop_ids=(), max_new=None, counters=None, offered=0):
    """Apply stop-set / cap truncation to one verify call's outputs.

    out: dict with tokens [B, W], num_accepted [B], logprob [B, W], mu [B, W],
    status [B] and optionally nodes [B, W] (copied, not modified).
    counters: int64 [B, 4] running totals or None (taken as zeros).
    Returns (new_out, out_len [B], new_counters [B, 4]).
    """
    res = {k: np.array(v, copy=True) for k, v in out.items()}
    tok = res["tokens"]
    B = tok.shape[0]
    stop = set(int(s) for s in stop_ids)
    out_len = np.zeros(B, dtype=np.int64)
    cnt = np.zeros((B, 4), dtype=np.int64) if counters is None else np.array(counters, dtype=np.int64, copy=True)
    for b in range(B):
        n = int(res["num_accepted"][b])
        kept = n + 1
        stopped = False
        for j in range(n + 1):
            if int(tok[b, j]) in stop:
                kept = j + 1
                stopped = True
                break
        capped = False
        if max_new is not None:
            cap = max(0, int(max_new[b]))
            if cap < kept:
                kept = cap
                capped = True
                stopped = False    # a stop token at index >= cap was cut off
        for j in range(kept, n + 1):
            tok[b, j] = -1
            res["logprob"][b, j] = 0.0
            res["mu"][b, j] = 0.0
            if "nodes" in res:
                res["nodes"][b, j] = -1
        res["status"][b] = int(res["status"][b]) | (STATUS_STOPPED if stopped else 0) | \
            (STATUS_CAPPED if capped else 0)
        out_len[b] = kept
        cnt[b] += (1, offered, n, kept)
    return res, out_len, cnt


def tau_alpha(counters):
    """Tokens per pass and acceptance rate from summed counters [.., 4]."""
    c = np.asarray(counters, dtype=np.int64).reshape(-1, 4).sum(axis=0)
    tau = c[3] / c[0] if c[0] else 0.0
    alpha = c[2] / c[1] if c[1] else 0.0
    return float(tau), float(alpha)
