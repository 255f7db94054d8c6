"""Pins for the oracle's stochastic chain rule.

1. Exact rationals (oracle.exact): the law of the first M = K+1 emitted tokens
   over repeated rounds equals the target's autoregressive joint, for V=4 and
   K=1..3 on context-dependent toy models (spec-decode README, "Provably
   exact" and "Design decisions").
2. Monte Carlo on the float64 oracle itself, driven by the same toy models:
   its emitted-token law matches that exact joint within 5 sigma.
3. mu (nanospec README: "the probability the speculative sampler emitted
   it"): the empirical frequency of each emitted token equals the mu the
   oracle reports, for the exact, power and relaxed rules, with and without
   draft logits.
4. Special cases: power alpha=1 is exact; relaxed tau=0 accepts everything
   (spec100m README's accept-all mode); relaxed tau>1 without top-k accepts
   nothing; relaxed mu = 1 on accepted drafts; exact mu = exp(logprob); a
   perfect draft emits exactly k+1 tokens per pass (spec-decode README,
   "Speedup (measured)"); deterministic drafts equal the chain-shaped tree.
"""

import itertools
import math
from collections import Counter

import numpy as np
import pytest

from oracle import exact as E
from oracle import spec_oracle as O


def _log(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray([float(a) for a in p]))


@pytest.mark.parametrize("K", [1, 2, 3])
@pytest.mark.parametrize("seed", [1, 2])
def test_rational_speculative_law_is_target_joint(K, seed):
    target = E.RationalMarkov(4, seed=100 + seed)
    draft = E.RationalMarkov(4, seed=200 + seed)
    M = K + 1
    spec = E.speculative_law(target, draft, (), M, K)
    joint = E.target_joint(target, (), M)
    assert set(k for k, v in spec.items() if v) == set(joint)
    for s, pr in joint.items():
        assert spec[s] == pr


def test_rational_law_detects_a_wrong_rule():
    # Accepting with min(1, q/p) instead of min(1, p/q) is not lossless.
    from fractions import Fraction
    target = E.RationalMarkov(4, seed=101)
    draft = E.RationalMarkov(4, seed=201)
    joint = E.target_joint(target, (), 2)
    # first-token law of one K=1 round with the swapped ratio:
    p, q = target.next_dist(()), draft.next_dist(())
    law = [Fraction(0)] * 4
    res = E.residual(p, q)
    for d in range(4):
        if q[d] == 0:
            continue
        r = min(Fraction(1), q[d] / p[d]) if p[d] else Fraction(1)
        law[d] += q[d] * r
        for a in range(4):
            if res and res[a]:
                law[a] += q[d] * (1 - r) * res[a]
    first = [sum(v for s, v in joint.items() if s[0] == a) for a in range(4)]
    assert law != first


def _run_rounds(target, draft, K, M, runs, rng, rule=O.RULE_EXACT, alpha=1.0, tau=0.0):
    """Drive oracle.verify_sample round after round with a toy model until M
    tokens are emitted; returns a Counter of the first M tokens."""
    V = target.V
    states = [tuple() for _ in range(runs)]
    done = Counter()
    while states:
        B = len(states)
        x = np.zeros((B, K + 1, V))
        y = np.zeros((B, K, V))
        d = np.zeros((B, K), dtype=np.int64)
        for b, ctx in enumerate(states):
            c = ctx
            for i in range(K):
                q = np.array([float(a) for a in draft.next_dist(c)])
                d[b, i] = rng.choice(V, p=q / q.sum())
                x[b, i] = _log(target.next_dist(c))
                y[b, i] = _log(draft.next_dist(c))
                c = c + (int(d[b, i]),)
            x[b, K] = _log(target.next_dist(c))
        u = rng.random((B, K + 1))
        out = O.verify_sample(x, y, d, 1.0, u, rule=rule, alpha=alpha, tau=tau)
        nxt = []
        for b, ctx in enumerate(states):
            n = out["num_accepted"][b]
            ctx = ctx + tuple(int(t) for t in out["tokens"][b, : n + 1])
            if len(ctx) >= M:
                done[ctx[:M]] += 1
            else:
                nxt.append(ctx)
        states = nxt
    return done


def test_monte_carlo_oracle_matches_exact_target_joint():
    rng = np.random.default_rng(77)
    K, M, runs = 2, 3, 30000
    target = E.RationalMarkov(4, seed=103)
    draft = E.RationalMarkov(4, seed=203)
    joint = E.target_joint(target, (), M)
    counts = _run_rounds(target, draft, K, M, runs, rng)
    assert sum(counts.values()) == runs
    for s in itertools.product(range(4), repeat=M):
        pi = float(joint.get(s, 0))
        f = counts.get(s, 0) / runs
        sigma = math.sqrt(max(pi * (1 - pi), 1e-12) / runs)
        assert abs(f - pi) <= 5 * sigma + 1e-9, (s, f, pi)


def _softmax(z):
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _check_mu_frequencies(tokens_at, mus_at, runs):
    """Tokens emitted at one position: the reported mu of each token is one
    value, and its empirical frequency matches it within 5 sigma."""
    by_tok = {}
    for t, m in zip(tokens_at, mus_at):
        by_tok.setdefault(int(t), set()).add(round(float(m), 12))
    for t, ms in by_tok.items():
        assert len(ms) == 1, (t, ms)
    total = len(tokens_at)
    seen = Counter(int(t) for t in tokens_at)
    mass = 0.0
    for t, ms in by_tok.items():
        mu = next(iter(ms))
        mass += mu
        f = seen[t] / total
        sigma = math.sqrt(max(mu * (1 - mu), 1e-12) / total)
        assert abs(f - mu) <= 5 * sigma + 1e-9, (t, f, mu)
    assert mass <= 1 + 1e-9


@pytest.mark.parametrize("rule,alpha,tau,top_k", [(O.RULE_EXACT, 1.0, 0.0, 0),
                                                  (O.RULE_POWER, 0.3, 0.0, 0),
                                                  (O.RULE_RELAXED, 1.0, 0.15, 0),
                                                  (O.RULE_RELAXED, 1.0, 0.3, 2)])
def test_mu_is_emission_probability_with_draft_logits(rule, alpha, tau, top_k):
    rng = np.random.default_rng(5 + rule + top_k)
    V, K, runs = 6, 2, 40000
    x = rng.normal(0, 1.5, (K + 1, V))
    y = x[:K] + rng.normal(0, 1.0, (K, V))
    q = np.stack([_softmax(y[i]) for i in range(K)])
    d = np.stack([rng.choice(V, size=runs, p=q[i]) for i in range(K)], axis=1)
    u = rng.random((runs, K + 1))
    out = O.verify_sample(np.broadcast_to(x, (runs, K + 1, V)),
                          np.broadcast_to(y, (runs, K, V)), d, 1.0, u,
                          rule=rule, alpha=alpha, tau=tau, top_k=top_k)
    _check_mu_frequencies(out["tokens"][:, 0], out["mu"][:, 0], runs)
    later = out["num_accepted"] >= 1     # rows are context-free here
    _check_mu_frequencies(out["tokens"][later, 1], out["mu"][later, 1], int(later.sum()))
    if rule == O.RULE_EXACT:
        emitted = out["tokens"] >= 0
        assert np.allclose(out["mu"][emitted], np.exp(out["logprob"][emitted]), atol=1e-12)


@pytest.mark.parametrize("rule,alpha,tau", [(O.RULE_EXACT, 1.0, 0.0),
                                            (O.RULE_POWER, 0.3, 0.0),
                                            (O.RULE_RELAXED, 1.0, 0.1)])
def test_mu_is_emission_probability_deterministic_drafts(rule, alpha, tau):
    rng = np.random.default_rng(9 + rule)
    V, K, runs = 5, 1, 40000
    x = rng.normal(0, 1.5, (K + 1, V))
    d = np.full((runs, K), int(np.argsort(x[0])[-2]))   # second-best token
    u = rng.random((runs, K + 1))
    out = O.verify_sample(np.broadcast_to(x, (runs, K + 1, V)), None, d, 1.0, u,
                          rule=rule, alpha=alpha, tau=tau)
    _check_mu_frequencies(out["tokens"][:, 0], out["mu"][:, 0], runs)
    if rule == O.RULE_RELAXED:
        acc = out["num_accepted"] >= 1
        assert (out["mu"][acc, 0] == 1.0).all()


def _random_chain(rng, B, K, V, std=2.0):
    x = rng.normal(0, std, (B, K + 1, V))
    y = x[:, :K] + rng.normal(0, 1.0, (B, K, V))
    d = np.zeros((B, K), dtype=np.int64)
    for b in range(B):
        for i in range(K):
            d[b, i] = rng.choice(V, p=_softmax(y[b, i]))
    u = rng.random((B, K + 1))
    return x, y, d, u


def test_power_alpha_one_is_exact():
    rng = np.random.default_rng(21)
    x, y, d, u = _random_chain(rng, 50, 4, 12)
    for drafts in (y, None):
        a = O.verify_sample(x, drafts, d, 1.0, u, rule=O.RULE_EXACT)
        b = O.verify_sample(x, drafts, d, 1.0, u, rule=O.RULE_POWER, alpha=1.0)
        for key in ("tokens", "num_accepted", "status"):
            assert np.array_equal(a[key], b[key])
        assert np.allclose(a["mu"], b["mu"], atol=1e-12)
        assert np.allclose(a["logprob"], b["logprob"], atol=1e-12)


def test_relaxed_extremes():
    rng = np.random.default_rng(22)
    x, y, d, u = _random_chain(rng, 40, 4, 12)
    for drafts in (y, None):
        allin = O.verify_sample(x, drafts, d, 1.0, u, rule=O.RULE_RELAXED, tau=0.0)
        assert (allin["num_accepted"] == 4).all()
        assert np.array_equal(allin["tokens"][:, :4], d)
        none = O.verify_sample(x, drafts, d, 1.0, u, rule=O.RULE_RELAXED, tau=1.5, top_k=0)
        assert (none["num_accepted"] == 0).all()
    # top-k alone: the argmax draft (rank 0) is accepted with top_k = 1
    am = np.argmax(x[:, :4], axis=-1)
    tk = O.verify_sample(x, None, am, 1.0, u, rule=O.RULE_RELAXED, tau=2.0, top_k=1)
    assert (tk["num_accepted"] == 4).all() and (tk["mu"][:, :4] == 1.0).all()


def test_relaxed_top_k_counts_strictly_greater_logits_with_ties():
    # one row with repeated values; the draft at each token in turn, tau out of
    # reach: accepted iff fewer than k logits are strictly above it
    row = np.array([1.0, 3.0, 2.0, 3.0, 0.5, 2.0, 3.0])
    greater = [5, 0, 3, 0, 6, 3, 0]   # logits strictly above row[t], counted by hand
    for k in (1, 3, 4, 6, 7):
        for t in range(row.size):
            x = np.stack([row, row])[None]        # K = 1: row 0 tests the draft
            out = O.verify_sample(x, None, np.array([[t]]), 1.0, np.array([[0.5, 0.5]]),
                                  rule=O.RULE_RELAXED, tau=2.0, top_k=k)
            assert int(out["num_accepted"][0]) == (1 if greater[t] < k else 0), (k, t)


def test_perfect_draft_emits_k_plus_one():
    rng = np.random.default_rng(23)
    x, _, _, u = _random_chain(rng, 30, 4, 10)
    y = x[:, :4].copy()
    d = np.zeros((30, 4), dtype=np.int64)
    for b in range(30):
        for i in range(4):
            d[b, i] = rng.choice(10, p=_softmax(y[b, i]))
    out = O.verify_sample(x, y, d, 1.0, u)
    assert (out["num_accepted"] == 4).all()
    assert ((out["tokens"] >= 0).sum(axis=1) == 5).all()


def test_temperature_scales_both_distributions():
    rng = np.random.default_rng(24)
    x, y, d, u = _random_chain(rng, 20, 3, 9)
    hot = O.verify_sample(x, y, d, 2.0, u)
    same = O.verify_sample(x / 2.0, y / 2.0, d, 1.0, u)
    for key in ("tokens", "num_accepted"):
        assert np.array_equal(hot[key], same[key])
    assert np.allclose(hot["logprob"], same["logprob"], atol=1e-12)


def test_deterministic_chain_equals_chain_tree():
    rng = np.random.default_rng(25)
    B, K, V = 60, 4, 10
    x, _, _, u = _random_chain(rng, B, K, V)
    d = rng.integers(0, V, (B, K))
    am = np.argmax(x[:, :K], axis=-1)
    d = np.where(rng.random((B, K)) < 0.6, am, d)
    parents = np.tile(np.arange(-1, K), (B, 1))
    toks = np.concatenate([np.zeros((B, 1), np.int64), d], axis=1)
    ut = np.concatenate([u[:, K:], u[:, :K]], axis=1)
    for rule, alpha, tau in ((O.RULE_EXACT, 1, 0), (O.RULE_POWER, 0.3, 0), (O.RULE_RELAXED, 1, 0.2)):
        c = O.verify_sample(x, None, d, 1.0, u, rule=rule, alpha=alpha, tau=tau)
        t = O.verify_tree(x, toks, parents, K, 1.0, ut, rule=rule, alpha=alpha, tau=tau)
        for key in ("tokens", "num_accepted", "status"):
            assert np.array_equal(c[key], t[key]), (rule, key)
        assert np.allclose(c["mu"], t["mu"], atol=1e-12)
        assert np.allclose(c["logprob"], t["logprob"], atol=1e-12)


def test_zero_mass_and_zero_q_cases():
    V = 4
    x = np.log(np.array([[[0.5, 0.5, 0.0, 0.0]] * 2]))
    y = np.log(np.array([[[0.0, 1.0, 0.0, 0.0]]]))
    with np.errstate(divide="ignore"):
        # q(0) = 0 < p(0): ratio 1, always accepted
        out = O.verify_sample(x, y, np.array([[0]]), 1.0, np.array([[0.999, 0.3]]))
        assert out["num_accepted"][0] == 1 and out["status"][0] == 0
        # p(2) = q(2) = 0: rejected, status flagged
        out = O.verify_sample(x, y, np.array([[2]]), 1.0, np.array([[0.0, 0.3]]))
        assert out["num_accepted"][0] == 0 and out["status"][0] == O.STATUS_ZERO_MASS
        assert out["tokens"][0, 0] == 0      # residual relu(p - q) = mass on token 0
    del V


def test_bad_draft_token_is_rejected():
    rng = np.random.default_rng(26)
    x, y, d, u = _random_chain(rng, 3, 3, 8)
    d[0, 1] = 8
    d[1, 0] = -3
    u[:] = 0.0                           # u = 0 accepts every valid draft with a > 0
    out = O.verify_sample(x, y, d, 1.0, u)
    assert out["num_accepted"][0] == 1 and out["status"][0] & O.STATUS_BAD_TOKEN
    assert out["num_accepted"][1] == 0 and out["status"][1] & O.STATUS_BAD_TOKEN
    assert out["num_accepted"][2] == 3 and out["status"][2] == 0
