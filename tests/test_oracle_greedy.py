"""Pins for the oracle's greedy chain rule (mini-sglang PR #134,
Modifications / verify.py and the Accuracy Tests scenario list) and the
greedy tree walk (nanospec README, tree configuration)."""

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import log_softmax

from oracle import spec_oracle as O
from speculative_decoding_verification_72_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_scenarios():
    rows = []
    with open(os.path.join(GOLDEN, "verify_drafts_scenarios.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, V, am, drafts, n, toks = [s.strip() for s in line.split("|")]
            am = [int(t) for t in am.split()]
            drafts = [] if drafts == "-" else [int(t) for t in drafts.split()]
            rows.append((name, int(V), am, drafts, int(n), [int(t) for t in toks.split()]))
    return rows


SCENARIOS = load_scenarios()


def one_hot_logits(V, argmaxes, hot=4.0):
    x = np.zeros((len(argmaxes), V))
    for i, a in enumerate(argmaxes):
        x[i, a] = hot
    return x


@pytest.mark.parametrize("scn", SCENARIOS, ids=[s[0] for s in SCENARIOS])
def test_verify_drafts_scenarios(scn):
    name, V, am, drafts, n, toks = scn
    K = len(drafts)
    assert len(am) == K + 1
    x = one_hot_logits(V, am)[None]
    out = O.verify_greedy(x, np.array([drafts], dtype=np.int64).reshape(1, K))
    assert out["num_accepted"][0] == n
    expect = toks + [-1] * (K + 1 - len(toks))
    assert list(out["tokens"][0]) == expect
    # closed form: log_softmax at the hot index = 4 - ln(e^4 + V - 1)
    lp = 4.0 - math.log(math.exp(4.0) + V - 1)
    assert np.allclose(out["logprob"][0, : n + 1], lp, atol=1e-14)
    assert (out["logprob"][0, n + 1:] == 0).all()
    assert (out["mu"][0, : n + 1] == 1).all() and (out["mu"][0, n + 1:] == 0).all()
    assert out["status"][0] == 0


def test_greedy_ties_go_to_lowest_index():
    x = np.zeros((1, 3, 6))
    x[0, 0, [2, 5]] = 1.0            # tie between 2 and 5
    x[0, 1, 4] = 1.0
    x[0, 2, [0, 1]] = 2.0            # bonus tie
    out = O.verify_greedy(x, np.array([[5, 4]]))
    assert out["num_accepted"][0] == 0 and out["tokens"][0, 0] == 2
    out = O.verify_greedy(x, np.array([[2, 4]]))
    assert out["num_accepted"][0] == 2 and list(out["tokens"][0]) == [2, 4, 0]


def test_greedy_logprob_is_log_softmax():
    ci = workloads.greedy_chain(B=6, K=5, V=300, dtype=torch.float32, seed=9)
    x = ci.target.double().numpy()
    out = O.verify_greedy(x, ci.draft_tokens.numpy())
    ref = log_softmax(x, axis=-1)
    for b in range(6):
        n = out["num_accepted"][b]
        for j in range(n + 1):
            assert abs(out["logprob"][b, j] - ref[b, j, out["tokens"][b, j]]) < 1e-12
        # the accepted prefix really matches the argmax, and the next draft does not
        for j in range(n):
            assert ci.draft_tokens[b, j] == np.argmax(x[b, j])
        if n < 5:
            assert ci.draft_tokens[b, n] != np.argmax(x[b, n])


def test_greedy_bad_token_and_nonfinite_row():
    x = np.zeros((2, 3, 5))
    x[:, :, 1] = 1.0
    out = O.verify_greedy(x, np.array([[1, 7], [-1, 1]]))
    assert out["num_accepted"][0] == 1 and out["status"][0] == O.STATUS_BAD_TOKEN
    assert list(out["tokens"][0]) == [1, 1, -1]
    assert out["num_accepted"][1] == 0 and out["status"][1] == O.STATUS_BAD_TOKEN
    x[1, 2, :] = -np.inf
    out = O.verify_greedy(x, np.array([[1, 1], [1, 1]]))
    assert out["status"][1] & O.STATUS_NONFINITE_ROW
    # a row after the first mismatch is not read, so it is not flagged
    out = O.verify_greedy(x, np.array([[1, 1], [0, 1]]))
    assert out["status"][1] == 0 and out["num_accepted"][1] == 0


def test_greedy_chain_equals_chain_shaped_tree():
    ci = workloads.greedy_chain(B=8, K=6, V=50, dtype=torch.float32, p_match=0.85, seed=4)
    x = ci.target.double().numpy()
    d = ci.draft_tokens.numpy().astype(np.int64)
    chain = O.verify_greedy(x, d)
    B, R, _ = x.shape
    parents = np.tile(np.arange(-1, R - 1), (B, 1))
    toks = np.concatenate([np.zeros((B, 1), np.int64), d], axis=1)
    tree = O.verify_tree(x, toks, parents, max_depth=R - 1, temperature=0.0)
    for key in ("tokens", "num_accepted", "status"):
        assert np.array_equal(chain[key], tree[key]), key
    assert np.allclose(chain["logprob"], tree["logprob"], atol=1e-12)
    assert np.array_equal(tree["nodes"][:, 0], np.zeros(B))


def _brute_force_greedy_tree(x, tok, par):
    """Deepest node whose every edge (parent -> child) carries the parent row's
    argmax; with distinct sibling tokens that node is unique."""
    N = len(par)
    best, best_depth = 0, 0
    for n in range(1, N):
        path, c, ok = [], n, True
        while c != 0:
            pc = par[c]
            if tok[c] != np.argmax(x[pc]):
                ok = False
                break
            path.append(c)
            c = pc
        if ok and len(path) > best_depth:
            best, best_depth = n, len(path)
    return best, best_depth


def test_greedy_tree_matches_brute_force():
    ti = workloads.eagle_tree(B=6, V=40, dtype=torch.float32, seed=12)
    x = ti.target.double().numpy()
    tok = ti.node_tokens.numpy().astype(np.int64)
    par = ti.parents.numpy().astype(np.int64)
    out = O.verify_tree(x, tok, par, max_depth=5, temperature=0.0)
    for b in range(6):
        node, depth = _brute_force_greedy_tree(x[b], tok[b], par[b])
        assert out["num_accepted"][b] == depth
        last = out["nodes"][b, depth]
        assert last == node
        assert out["tokens"][b, depth] == np.argmax(x[b, node])
        # path tokens are the accepted nodes' tokens
        for j in range(depth):
            assert out["tokens"][b, j] == tok[b, out["nodes"][b, j + 1]]
            assert par[b, out["nodes"][b, j + 1]] == out["nodes"][b, j]


def test_tree_shape_generator_is_ancestor_closed_bfs():
    rng = np.random.default_rng(0)
    for _ in range(20):
        par = workloads.tree_shape(rng)
        assert len(par) == 64 and par[0] == -1
        assert all(0 <= par[n] < n for n in range(1, 64))
        depth = np.zeros(64, int)
        for n in range(1, 64):
            depth[n] = depth[par[n]] + 1
        assert depth.max() <= 5 and (np.diff(depth) >= 0).all()
