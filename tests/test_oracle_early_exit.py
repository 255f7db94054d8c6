"""Pins of oracle/early_exit.py: hand counts, and the fact it rests on --
the greedy oracle's outputs do not depend on rows after the first mismatch."""

import numpy as np

from oracle import early_exit as E
from oracle import spec_oracle as O


def test_rows_and_byte_bounds_by_hand():
    assert E.rows_needed([0, 3, 5]).tolist() == [1, 4, 6]
    # K = 5, V = 10, bf16: at least (1 + 4 + 6) rows of 20 bytes, at most 3 * 6 rows
    assert E.bytes_bounds([0, 3, 5], 5, 10, 2) == (220, 360)


def test_rows_after_the_first_mismatch_do_not_change_greedy_outputs():
    rng = np.random.default_rng(11)
    B, K, V = 40, 12, 17
    x = rng.normal(0, 2, (B, K + 1, V))
    am = np.argmax(x[:, :K], axis=-1)
    d = np.where(rng.random((B, K)) < 0.7, am, (am + 1 + rng.integers(0, V - 1, (B, K))) % V)
    ref = O.verify_greedy(x, d)
    y = x.copy()
    for b in range(B):
        n = int(ref["num_accepted"][b])
        y[b, n + 1:] = rng.normal(0, 5, (K - n, V))      # scramble every row the decision never reads
    got = O.verify_greedy(y, d)
    for k in ("tokens", "num_accepted", "logprob", "mu", "status"):
        assert np.array_equal(got[k], ref[k]), k
    # while scrambling row n itself does change them
    z = x.copy()
    for b in range(B):
        z[b, int(ref["num_accepted"][b])] = rng.normal(0, 5, V)
    assert not np.array_equal(O.verify_greedy(z, d)["logprob"], ref["logprob"])
