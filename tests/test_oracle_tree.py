"""Pins for the oracle's stochastic tree walk (nanospec README: tree
configuration; exact / relaxed / power rules; mu per emitted token).

* Telescoping, in exact rationals: with deterministic drafts and the exact
  rule, the law of the token a node emits is p (oracle.exact.tree_node_law).
* Monte Carlo on the float64 oracle: the frequency of each token a node emits
  equals the mu the oracle reports, for all three rules, and equals p for the
  exact rule.
* Structure: bad parent links, the depth cap, duplicate sibling tokens.
"""

import math
import random
from collections import Counter
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import exact as E
from oracle import spec_oracle as O
from speculative_decoding_verification_72_gb300 import workloads


def test_rational_tree_node_law_telescopes_to_p():
    rng = random.Random(8)
    for _ in range(300):
        V = rng.randint(2, 9)
        w = [rng.randint(0, 6) for _ in range(V)]
        if sum(w) == 0:
            w[0] = 1
        p = [Fraction(a, sum(w)) for a in w]
        m = rng.randint(1, V)
        kids = rng.sample(range(V), m)
        assert E.tree_node_law(p, kids) == p


def _star_tree(V, kids_tokens):
    m = len(kids_tokens)
    parents = np.array([-1] + [0] * m)
    toks = np.array([0] + list(kids_tokens))
    return parents, toks


@pytest.mark.parametrize("rule,alpha,tau", [(O.RULE_EXACT, 1.0, 0.0),
                                            (O.RULE_POWER, 0.3, 0.0),
                                            (O.RULE_RELAXED, 1.0, 0.12)])
def test_node_emission_frequency_is_mu(rule, alpha, tau):
    rng = np.random.default_rng(31 + rule)
    V, runs = 7, 40000
    x_root = rng.normal(0, 1.2, V)
    order = np.argsort(-x_root)
    kids = [int(order[0]), int(order[2]), int(order[4])]
    parents, toks = _star_tree(V, kids)
    N = len(toks)
    x = rng.normal(0, 1.0, (N, V))
    x[0] = x_root
    u = rng.random((runs, N))
    out = O.verify_tree(np.broadcast_to(x, (runs, N, V)), np.broadcast_to(toks, (runs, N)),
                        np.broadcast_to(parents, (runs, N)), max_depth=3, temperature=1.0,
                        uniforms=u, rule=rule, alpha=alpha, tau=tau)
    first = out["tokens"][:, 0]
    mus = out["mu"][:, 0]
    seen = Counter(int(t) for t in first)
    p = O.target_probs(x_root)
    for t in seen:
        vals = set(np.round(mus[first == t], 12))
        assert len(vals) == 1
        mu = vals.pop()
        f = seen[t] / runs
        assert abs(f - mu) <= 5 * math.sqrt(max(mu * (1 - mu), 1e-12) / runs) + 1e-9
        if rule == O.RULE_EXACT:
            assert abs(mu - p[t]) < 1e-12
    if rule == O.RULE_RELAXED:
        acc = out["num_accepted"] >= 1
        assert (out["mu"][acc, 0] == 1.0).all()


def test_exact_tree_mu_equals_probability():
    ti = workloads.eagle_tree(B=5, V=30, dtype=torch.float32, seed=41)
    x = ti.target.double().numpy()
    out = O.verify_tree(x, ti.node_tokens.numpy(), ti.parents.numpy(), 5, 1.0,
                        ti.uniforms.double().numpy())
    em = out["tokens"] >= 0
    assert np.allclose(out["mu"][em], np.exp(out["logprob"][em]), atol=1e-12)
    for b in range(5):
        n = out["num_accepted"][b]
        assert (out["tokens"][b, : n + 1] >= 0).all() and (out["tokens"][b, n + 1:] == -1).all()
        for j in range(n):   # the accepted path is a real root-to-node path
            c = out["nodes"][b, j + 1]
            assert ti.parents[b, c] == out["nodes"][b, j]
            assert out["tokens"][b, j] == ti.node_tokens[b, c]


def test_bad_parent_links_are_flagged_and_excluded():
    V = 6
    x = np.zeros((1, 4, V))
    x[0, 0, 2] = 5.0
    x[0, 1, 3] = 5.0
    x[0, 2, 4] = 5.0
    toks = np.array([[0, 2, 3, 4]])
    par = np.array([[-1, 0, 3, 1]])          # node 2 points forward: invalid
    out = O.verify_tree(x, toks, par, 3, 0.0)
    assert out["status"][0] & O.STATUS_BAD_PARENT
    assert out["num_accepted"][0] == 1       # node 2 is not a child of node 1
    assert list(out["tokens"][0, :2]) == [2, 3]


def test_depth_cap_and_duplicates():
    V = 5
    x = np.zeros((1, 4, V))
    for n in range(4):
        x[0, n, 1] = 6.0
    toks = np.array([[0, 1, 1, 1]])
    par = np.array([[-1, 0, 1, 2]])
    out = O.verify_tree(x, toks, par, 2, 0.0)
    assert out["num_accepted"][0] == 2 and out["status"][0] & O.STATUS_DEPTH_EXCEEDED
    assert list(out["tokens"][0]) == [1, 1, 1]
    # duplicate sibling tokens: once token 3 is rejected its duplicate cannot pass
    x = np.zeros((1, 3, V))
    toks = np.array([[0, 3, 3]])
    par = np.array([[-1, 0, 0]])
    u = np.array([[0.5, 0.99, 0.0]])         # node 1 rejected, node 2 would pass
    out = O.verify_tree(x, toks, par, 2, 1.0, u)
    assert out["num_accepted"][0] == 0
    assert out["tokens"][0, 0] != 3          # drawn from p with token 3 zeroed
    assert abs(out["mu"][0, 0] - 0.2) < 1e-12   # uniform p: (1 - 0.2) * 0.2 / 0.8
