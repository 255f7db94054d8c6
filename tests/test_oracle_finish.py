"""Pins of oracle/finish.py: stop-set and cap truncation worked by hand, and
the spec-decode README run numbers recovered through the counters."""

import json
import os

import numpy as np
import pytest

from oracle import finish as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "spec_decode_readme_numbers.json")


def _one(tokens, n, nodes=None):
    W = len(tokens)
    out = dict(tokens=np.array([tokens], dtype=np.int64), num_accepted=np.array([n]),
               logprob=np.full((1, W), -0.5), mu=np.full((1, W), 0.25), status=np.array([0]))
    for j in range(n + 1, W):
        out["logprob"][0, j] = 0.0
        out["mu"][0, j] = 0.0
    if nodes is not None:
        out["nodes"] = np.array([nodes], dtype=np.int64)
    return out


def test_stop_token_inside_the_emitted_run_is_kept_and_ends_it():
    o = _one([5, 9, 2, 7], 3)
    r, L, c = F.finish(o, stop_ids=[2])
    assert L[0] == 3
    assert r["tokens"][0].tolist() == [5, 9, 2, -1]
    assert r["logprob"][0].tolist() == [-0.5, -0.5, -0.5, 0.0]
    assert r["mu"][0].tolist() == [0.25, 0.25, 0.25, 0.0]
    assert r["status"][0] == F.STATUS_STOPPED
    assert c[0].tolist() == [1, 0, 3, 3]
    assert o["tokens"][0].tolist() == [5, 9, 2, 7]          # input untouched


def test_stop_at_the_first_position_and_after_the_run():
    r, L, _ = F.finish(_one([2, 9, 4], 2), stop_ids=[2])
    assert L[0] == 1 and r["tokens"][0].tolist() == [2, -1, -1]
    r, L, _ = F.finish(_one([5, 9, -1, -1], 1), stop_ids=[7, -1])   # -1 slots are not emitted
    assert L[0] == 2 and r["status"][0] == 0


def test_the_first_of_several_stop_ids_wins():
    r, L, _ = F.finish(_one([5, 9, 7, 3], 3), stop_ids=[7, 9])
    assert L[0] == 2 and r["tokens"][0].tolist() == [5, 9, -1, -1]


def test_cap_truncates_and_flags():
    r, L, c = F.finish(_one([5, 9, 2, 7], 3), max_new=[2], offered=4)
    assert L[0] == 2 and r["tokens"][0].tolist() == [5, 9, -1, -1]
    assert r["status"][0] == F.STATUS_CAPPED
    assert c[0].tolist() == [1, 4, 3, 2]
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3), max_new=[0])
    assert L[0] == 0 and r["tokens"][0].tolist() == [-1, -1, -1, -1]
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3), max_new=[-3])      # clamped at zero
    assert L[0] == 0
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3), max_new=[4])
    assert L[0] == 4 and r["status"][0] == 0


def test_stop_and_cap_together():
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3), stop_ids=[2], max_new=[2])
    assert L[0] == 2 and r["status"][0] == F.STATUS_CAPPED        # the stop token was cut
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3), stop_ids=[2], max_new=[3])
    assert L[0] == 3 and r["status"][0] == F.STATUS_STOPPED       # kept exactly up to it


def test_tree_nodes_are_cleared_with_the_tokens():
    r, L, _ = F.finish(_one([5, 9, 2, 7], 3, nodes=[0, 3, 11, 40]), stop_ids=[9])
    assert L[0] == 2 and r["nodes"][0].tolist() == [0, 3, -1, -1]


def test_counters_accumulate_and_give_the_readme_run():
    g = json.load(open(GOLDEN))["run"]
    passes, tokens, k = g["target_passes"], g["tokens"], g["k"]
    # a run of `passes` calls, nothing truncated, that emitted `tokens` in all:
    # each call keeps n + 1 tokens, so the accepted drafts total tokens - passes
    rng = np.random.default_rng(3)
    n = np.full(passes, (tokens - passes) // passes)
    n[rng.choice(passes, (tokens - passes) - int(n.sum()), replace=False)] += 1
    assert n.sum() == tokens - passes and n.max() <= k
    cnt = np.zeros((1, 4), dtype=np.int64)
    for ni in n:
        o = _one([1] * (k + 1), int(ni))
        _, _, cnt = F.finish(o, counters=cnt, offered=k)
    assert cnt[0].tolist() == [passes, passes * k, tokens - passes, tokens]
    tau, alpha = F.tau_alpha(cnt)
    assert round(tau, 3) == g["tokens_per_pass"]
    assert round(alpha, 3) == g["acceptance_rate"]
