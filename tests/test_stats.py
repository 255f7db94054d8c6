"""Host-side acceptance statistics against the numbers the pages print."""

import json
import os

import numpy as np

from speculative_decoding_verification_72_gb300 import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_spec_decode_cli_numbers():
    with open(os.path.join(GOLDEN, "spec_decode_readme_numbers.json")) as f:
        g = json.load(f)["run"]
    tpp = stats.tokens_per_pass(g["tokens"], g["target_passes"])
    assert round(tpp, 3) == g["tokens_per_pass"]
    rate = stats.acceptance_rate_from_tokens_per_pass(round(tpp, 3), g["k"])
    assert round(rate, 3) == g["acceptance_rate"]
    sp = stats.speedup(round(tpp, 3), g["k"], g["draft_cost"])
    assert round(sp, 2) == g["speedup"]


def test_perfect_draft_gives_k_plus_one_per_pass():
    s = stats.acceptance_stats(np.full(100, 4), K=4)
    assert s["tokens_per_pass"] == 5.0 and s["acceptance_rate"] == 1.0


def test_mini_sglang_forward_counts_follow_from_acceptance():
    with open(os.path.join(GOLDEN, "mini_sglang_acceptance.json")) as f:
        g = json.load(f)
    n_new = g["new_tokens"]
    for kind, acc in g["per_round_acceptance"].items():
        # one verify forward per round of (accepted + 1) tokens, plus prefill
        forwards = n_new / (acc + 1.0) + 1.0
        assert abs(forwards - g["target_forwards"][kind]) <= 1.5, kind
    assert n_new / 1.0 + 1.0 == g["target_forwards"]["non_speculative"]


def test_acceptance_stats_fields():
    s = stats.acceptance_stats([0, 1, 2, 3], K=4)
    assert s["rounds"] == 4 and s["tokens"] == 10.0
    assert s["mean_accepted"] == 1.5 and s["acceptance_rate"] == 0.375
