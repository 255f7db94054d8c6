"""Exact-rational brute force of speculative sampling on tiny vocabularies.

TEST INFRASTRUCTURE (see oracle/__init__.py). Used only to pin
oracle.spec_oracle: nothing here is timed or compared with the GPU directly.

A model is a function next_dist(prefix) -> tuple of Fractions, as in the
spec-decode README, "Design decisions" (a model is next_dist(prefix); toy
Markov models stand in for networks). The functions below enumerate every
draft sequence and every accept / reject branch analytically:

  target_joint          law of the first M tokens sampled one at a time from
                        the target (the distribution the method must keep);
  speculative_round     law of one draft-K / verify-once round, spec-decode
                        README "How it works" (accept with min(1, p/q), residual
                        normalize(relu(p - q)) at the first rejection, bonus
                        sample from p when all K are accepted);
  speculative_law       law of the first M tokens over repeated rounds;
  tree_node_law         law of the token emitted at one tree node with
                        deterministic draft children under the exact rule
                        (telescoping: it must equal p).

Parity status: speculative_law == target_joint and tree_node_law == p are the
losslessness the spec-decode README ("Provably exact") states; the tests assert
both as exact rational equalities.
"""

from __future__ import annotations

import random
from collections import defaultdict
from fractions import Fraction


class RationalMarkov:
    """Context-dependent toy model over V tokens with rational probabilities.

    The next-token law depends on the last token and on the prefix length
    modulo 3; some entries are zero so that zero-mass cases are exercised.
    """

    def __init__(self, V, seed, zero_rate=0.2):
        rng = random.Random(seed)
        self.V = V
        self.table = {}
        for phase in range(3):
            for last in range(-1, V):
                w = [0 if rng.random() < zero_rate else rng.randint(1, 9) for _ in range(V)]
                if sum(w) == 0:
                    w[rng.randrange(V)] = 1
                s = sum(w)
                self.table[(phase, last)] = tuple(Fraction(a, s) for a in w)

    def next_dist(self, prefix):
        last = prefix[-1] if prefix else -1
        return self.table[(len(prefix) % 3, last)]


def residual(p, q):
    w = [max(pi - qi, Fraction(0)) for pi, qi in zip(p, q)]
    s = sum(w)
    if s == 0:
        return None
    return [wi / s for wi in w]


def target_joint(target, prefix, M):
    """P(t_0..t_{M-1}) = prod_j p(prefix + t_<j)(t_j)."""
    law = {(): Fraction(1)}
    for _ in range(M):
        nxt = {}
        for seq, pr in law.items():
            p = target.next_dist(tuple(prefix) + seq)
            for a, pa in enumerate(p):
                if pa:
                    nxt[seq + (a,)] = pr * pa
        law = nxt
    return law


def speculative_round(target, draft, prefix, K):
    """Law of the tokens one round emits (n accepted drafts + 1)."""
    out = defaultdict(Fraction)
    V = target.V

    def walk(i, ctx, emitted, prob):
        p = target.next_dist(ctx)
        if i == K:
            for a in range(V):
                if p[a]:
                    out[emitted + (a,)] += prob * p[a]
            return
        q = draft.next_dist(ctx)
        res = residual(p, q)
        for d in range(V):
            if q[d] == 0:
                continue
            r = min(Fraction(1), p[d] / q[d])
            if r > 0:
                walk(i + 1, ctx + (d,), emitted + (d,), prob * q[d] * r)
            if r < 1:
                rej = prob * q[d] * (1 - r)
                for a in range(V):
                    if res[a]:
                        out[emitted + (a,)] += rej * res[a]

    walk(0, tuple(prefix), (), Fraction(1))
    return dict(out)


def speculative_law(target, draft, prefix, M, K):
    """Law of the first M tokens emitted by repeated speculative rounds."""
    law = defaultdict(Fraction)
    frontier = {(): Fraction(1)}
    while frontier:
        shortest = min(len(s) for s in frontier)
        batch = {s: pr for s, pr in frontier.items() if len(s) == shortest}
        for s in batch:
            del frontier[s]
        for emitted, pr in batch.items():
            for seq, pr_round in speculative_round(target, draft, tuple(prefix) + emitted, K).items():
                nxt = emitted + seq
                if len(nxt) >= M:
                    law[nxt[:M]] += pr * pr_round
                else:
                    frontier[nxt] = frontier.get(nxt, Fraction(0)) + pr * pr_round
    return dict(law)


def tree_node_law(p, child_tokens):
    """Law of the token emitted at a node whose children carry the distinct
    tokens child_tokens (tested in order) under the exact rule with one-hot
    drafts: a_j = p(c_j) / rest_j, rest_{j+1} = rest_j - p(c_j); when all are
    rejected the draw is from p with the children's tokens zeroed."""
    V = len(p)
    law = [Fraction(0)] * V
    rest = Fraction(1)
    reach = Fraction(1)
    for t in child_tokens:
        a = min(Fraction(1), p[t] / rest) if rest > 0 else Fraction(1)
        law[t] += reach * a
        reach *= (1 - a)
        rest -= p[t]
    w = [Fraction(0) if a in child_tokens else p[a] for a in range(V)]
    s = sum(w)
    if s > 0:
        for a in range(V):
            law[a] += reach * w[a] / s
    return law
