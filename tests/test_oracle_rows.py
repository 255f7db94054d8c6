"""Pins for the oracle's row-level pieces: log-sum-exp, the residual, the
closed-form induced distribution and the inverse-CDF draw.

The identity test follows the spec-decode README, "Provably exact": the law of
the first emitted token, q(t) min(1, p(t)/q(t)) + (rejection mass)
residual(p, q)(t), equals p; the README's own check reports a maximum total
variation of 2.21e-16 over random pairs. Here the bound is 1e-12 over 6000
pairs, including zeros in p or q, equal and disjoint supports.
"""

import json
import math
import os

import numpy as np

from oracle import spec_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax(z):
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _pair(rng, k):
    V = int(rng.integers(2, 65))
    kind = k % 6
    if kind == 0:
        p = rng.dirichlet(np.full(V, 0.3))
        q = rng.dirichlet(np.full(V, 0.3))
    elif kind == 1:
        p = _softmax(rng.normal(0, 2, V))
        q = _softmax(rng.normal(0, 2, V))
    elif kind == 2:                      # zeros in q
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        q[rng.random(V) < 0.4] = 0.0
        if q.sum() == 0:
            q[0] = 1.0
        q /= q.sum()
    elif kind == 3:                      # zeros in p
        p = rng.dirichlet(np.ones(V))
        q = rng.dirichlet(np.ones(V))
        p[rng.random(V) < 0.4] = 0.0
        if p.sum() == 0:
            p[-1] = 1.0
        p /= p.sum()
    elif kind == 4:                      # disjoint supports
        cut = int(rng.integers(1, V))
        p = np.zeros(V)
        q = np.zeros(V)
        p[:cut] = rng.dirichlet(np.ones(cut))
        q[cut:] = rng.dirichlet(np.ones(V - cut))
    else:                                # p == q
        p = rng.dirichlet(np.ones(V))
        q = p.copy()
    return p, q


def test_induced_distribution_equals_target():
    with open(os.path.join(GOLDEN, "spec_decode_readme_numbers.json")) as f:
        printed = json.load(f)["verify_max_tv"]
    rng = np.random.default_rng(20240601)
    worst = 0.0
    for k in range(6000):
        p, q = _pair(rng, k)
        induced = O.induced_from_dists(p, q)
        tv = 0.5 * np.abs(induced - p).sum()
        worst = max(worst, tv)
    assert worst < 1e-12, worst
    # the README's figure is the same order as ours (double rounding only)
    assert printed < 1e-12


def test_induced_distribution_detects_a_wrong_residual():
    # A residual of relu(q - p) instead of relu(p - q) must break the identity.
    rng = np.random.default_rng(3)
    p, q = _softmax(rng.normal(0, 2, 16)), _softmax(rng.normal(0, 2, 16))
    wrong = np.maximum(q - p, 0)
    wrong /= wrong.sum()
    accepted = np.minimum(p, q)
    bad = accepted + (1 - accepted.sum()) * wrong
    assert 0.5 * np.abs(bad - p).sum() > 1e-3
    assert 0.5 * np.abs(O.induced_from_dists(p, q) - p).sum() < 1e-14


def test_residual_mass_is_total_variation():
    # sum relu(p - q) = 1 - sum min(p, q) = TV(p, q): a closed form.
    rng = np.random.default_rng(5)
    for k in range(500):
        p, q = _pair(rng, k)
        w = np.maximum(p - q, 0)
        tv = 0.5 * np.abs(p - q).sum()
        assert abs(w.sum() - tv) < 1e-14
        res = O.residual(p, q)
        if tv > 0:
            assert abs(res.sum() - 1) < 1e-14 and (res[p <= q] == 0).all()
        else:
            assert res is None


def test_log_sum_exp_against_fsum():
    rng = np.random.default_rng(11)
    for V in (2, 7, 32, 1000, 50257):
        for T in (1.0, 0.7, 2.5):
            x = rng.normal(0, 3, V)
            if V > 10:
                x[rng.integers(0, V, 3)] = -np.inf
            ref = math.log(math.fsum(math.exp(v / T) for v in x))
            assert abs(O.log_sum_exp(x, T) - ref) < 1e-12 * max(1.0, abs(ref))
            p = O.target_probs(x, T)
            assert abs(math.fsum(p) - 1.0) < 1e-12


def test_first_argmax_takes_lowest_index_on_ties():
    x = np.array([0.5, 3.0, -1.0, 3.0, 3.0])
    assert O.first_argmax(x) == 1
    assert O.rank_of(x, 0) == 3 and O.rank_of(x, 3) == 0 and O.rank_of(x, 2) == 4


def test_inverse_cdf_has_law_w_over_sum():
    # Over a fine grid of u the draw frequencies equal w / S to within 1/M.
    rng = np.random.default_rng(17)
    M = 20000
    us = (np.arange(M) + 0.5) / M
    for V in (1, 2, 5, 40):
        w = rng.random(V) * (rng.random(V) < 0.7)
        if w.sum() == 0:
            w[-1] = 0.5
        counts = np.zeros(V)
        for u in us:
            j = O.inverse_cdf(w, u)[0]
            counts[j] += 1
        assert np.all(np.abs(counts / M - w / w.sum()) <= 1.0 / M + 1e-12)
        assert counts[w == 0].sum() == 0


def test_inverse_cdf_edges_and_margin():
    w = np.array([0.0, 0.25, 0.0, 0.75])
    assert O.inverse_cdf(w, 0.0)[0] == 1          # u = 0: first positive index
    assert O.inverse_cdf(w, 0.2499)[0] == 1
    assert O.inverse_cdf(w, 0.25)[0] == 3         # boundary goes to the next cell
    j, margin, lo, hi = O.inverse_cdf(w, 0.5)
    assert j == 3 and abs(margin - 0.25) < 1e-15 and lo == hi == 3
    assert O.inverse_cdf(np.array([0.0, 2.0]), 1 - 2 ** -53)[0] == 1
    # the band: cells within 1e-5 * S of u * S
    w = np.array([0.5, 1e-6, 1e-6, 0.5 - 2e-6])
    j, margin, lo, hi = O.inverse_cdf(w, 0.5 + 0.5e-6)
    assert j == 1 and lo == 0 and hi == 3 and margin < 1e-5
    j, margin, lo, hi = O.inverse_cdf(w, 0.25)
    assert j == lo == hi == 0
