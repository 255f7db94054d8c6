"""CPU oracle for early-exit greedy verification: what a verify call that
stops reading a request's rows after its first mismatch must still read.

TEST INFRASTRUCTURE: only tests/ and bench.py's oracle legs use this module;
it shares no code with the CUDA library.

Source: mini-sglang PR #134 "[Feature] Vanilla speculative decoding",
Modifications (verify.py): the accepted prefix ends at the first draft that
differs from its row's argmax, and the bonus token is that row's argmax, so
rows after the first mismatch never influence the outputs. Early exit must
therefore return exactly verify_greedy's outputs (spec_oracle) while reading,
per request, at least rows 0..n (n = num_accepted) and at most all K+1.

Parity status: pinned by tests/test_oracle_early_exit.py (hand counts and the
dependence of verify_greedy on rows after n).
"""

from __future__ import annotations

import numpy as np


def rows_needed(num_accepted):
    """Rows each request must read: n + 1 (rows 0..n)."""
    return np.asarray(num_accepted, dtype=np.int64) + 1


def bytes_bounds(num_accepted, K, V, elem_bytes):
    """(least bytes any correct early exit reads, bytes of every row)."""
    n = np.asarray(num_accepted, dtype=np.int64)
    lo = int(rows_needed(n).sum()) * V * elem_bytes
    hi = int(n.size) * (K + 1) * V * elem_bytes
    return lo, hi
