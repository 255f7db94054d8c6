"""Pins of oracle/tree_build.py: a tree worked by hand, the topk = 1 chain,
keep-everything, and invariants checked by an independent walk."""

import numpy as np

from oracle import tree_build as T


def test_hand_worked_tree():
    # V = 5, depth 2, topk 2, 5 nodes. Logits are log-probs, so softmax returns them.
    p = np.array([[0.5, 0.3, 0.1, 0.05, 0.05],     # root row
                  [0.1, 0.5, 0.3, 0.05, 0.05],     # row of the best level-1 node (token 0)
                  [0.7, 0.1, 0.1, 0.05, 0.05]])    # row of the second (token 1); tokens 1, 2 tie
    out = T.build_tree(np.log(p)[None], depth=2, topk=2, n_nodes=5)
    # candidates: t0 .5, t1 .3 | under t0: t1 .25, t2 .15 | under t1: t0 .21, t1 .03 (tie -> lower id)
    # keep the 4 best: .5, .3, .25, .21; BFS by level then score
    assert out["tokens"][0].tolist() == [-1, 0, 1, 1, 0]
    assert out["parents"][0].tolist() == [-1, 0, 0, 1, 2]
    assert np.allclose(out["scores"][0], np.log([1, 0.5, 0.3, 0.25, 0.21]))
    assert not out["near_tie"][0]


def test_topk_one_is_the_argmax_chain():
    rng = np.random.default_rng(1)
    y = rng.normal(0, 3, (3, 5, 50))                 # depth 5, topk 1: rows 0..4
    out = T.build_tree(y, depth=5, topk=1, n_nodes=6)
    for b in range(3):
        assert out["parents"][b].tolist() == [-1, 0, 1, 2, 3, 4]
        assert out["tokens"][b, 1:].tolist() == [int(np.argmax(y[b, r])) for r in range(5)]


def test_keeping_every_candidate_and_structure():
    rng = np.random.default_rng(2)
    depth, k = 3, 3
    R = 1 + (depth - 1) * k
    total = k + (depth - 1) * k * k
    y = rng.normal(0, 2, (4, R, 40))
    full = T.build_tree(y, depth, k, 1 + total)
    for b in range(4):
        assert sorted(np.bincount(_depths(full["parents"][b]))[1:].tolist()) == [k, k * k, k * k]
    out = T.build_tree(y, depth, k, 12)
    for b in range(4):
        par, tok, sc = out["parents"][b], out["tokens"][b], out["scores"][b]
        dep = _depths(par)
        assert all(par[n] < n for n in range(1, 12)) and dep.max() <= depth
        assert all(dep[n] >= dep[n - 1] for n in range(2, 12))               # BFS order
        # every kept score >= every dropped candidate's score
        kept = set(np.round(sc[1:], 12).tolist())
        allsc = np.sort(full["scores"][b, 1:])[::-1]
        assert min(sc[1:]) >= allsc[11] - 1e-12
        assert len(kept) == 11
        # scores re-derived along each path: the row of a level-d node's parent is
        # found by ranking the parent's level, independently of the builder's order
        for n in range(1, 12):
            assert sc[n] <= (sc[par[n]] if par[n] > 0 else 0.0) + 1e-12
        lvl1 = [n for n in range(1, 12) if dep[n] == 1]
        assert sorted(tok[n] for n in lvl1) == sorted(T.top_tokens(y[b, 0], k)[:len(lvl1)])
        for n in lvl1:
            assert abs(sc[n] - T.log_softmax(y[b, 0])[tok[n]]) < 1e-12


def _depths(par):
    d = np.zeros(len(par), dtype=np.int64)
    for n in range(1, len(par)):
        d[n] = d[par[n]] + 1
    return d


def test_tied_logits_take_the_lower_token():
    # depth 2, topk 1: the root row's top logit is shared by tokens 2 and 4,
    # the next row's by tokens 1 and 5; the lower id wins each time
    y = np.zeros((1, 2, 6))
    y[0, 0, [4, 2]] = 3.0
    y[0, 1, [5, 1]] = 1.5
    out = T.build_tree(y, depth=2, topk=1, n_nodes=3)
    assert out["tokens"][0].tolist() == [-1, 2, 1]


def test_temperature_limits():
    # a very hot softmax is uniform: a depth-d node scores -d log V; a very
    # cold one puts all mass on the argmax: the argmax chain scores ~0
    rng = np.random.default_rng(5)
    V = 50
    y = rng.normal(0, 3, (2, 4, V))                  # depth 2, topk 3: rows 0..3
    hot = T.build_tree(y, 2, 3, 13, temperature=1e6)
    for b in range(2):
        dep = _depths(hot["parents"][b])
        assert np.allclose(hot["scores"][b, 1:], -dep[1:] * np.log(V), atol=1e-4)
    cold = T.build_tree(y, 2, 3, 13, temperature=1e-3)
    for b in range(2):
        best = int(np.argmax(cold["scores"][b, 1:])) + 1
        assert cold["scores"][b, best] > -1e-6
        assert cold["tokens"][b, 1] == int(np.argmax(y[b, 0]))
