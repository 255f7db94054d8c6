"""Float64 CPU oracle for EAGLE-style draft-tree construction: top-k
expansion level by level, then a rerank of all candidates to n_nodes.

TEST INFRASTRUCTURE: only tests/ (and bench.py's oracle legs) use this
module; it shares no code with the CUDA library.

Source: nanospec README, introduction and bench configurations (EAGLE-3
tree speculation, "tree (depth 5, topk 4)"; the task's workload prunes it to
64 nodes). The page names the parameters, not the procedure; the reading
taken here (the usual EAGLE construction):
  * a node's score is the cumulative draft log-prob of its path:
    score(child) = score(parent) + log_softmax(y / T)[token], root score 0;
  * level 1 = the topk tokens of the root's draft row; for every later level
    the topk best nodes of the level above (score descending, earlier
    candidate first on ties) are expanded, each into the topk tokens of its
    own draft row; a row's top tokens are taken by raw logit, lower token id
    first on ties;
  * draft rows arrive in that order: row 0 is the root's, row
    1 + (d - 2) * topk + r belongs to the r-th best node of level d - 1
    (d = 2..depth), so 1 + (depth - 1) * topk rows per request;
  * the n_nodes - 1 best candidates (score descending, earlier candidate
    first) are kept with the root; since log-probs are <= 0 a parent always
    ranks before its child, so the kept set is ancestor-closed;
  * output order is BFS: root first, then by level, within a level by score
    descending (earlier candidate first), as workloads.tree_shape orders its
    trees; the root's token is -1 and its parent -1.
A request is flagged near_tie when a decision above compares two distinct
scores closer than NEAR (1e-4): the order of a level's best topk + 1 nodes, the
keep boundary, or the order of two kept nodes of one level; the device
path, summing in fp32, may then legitimately order them differently.

Parity status: pinned by tests/test_oracle_tree_build.py (a hand-worked
tree, the topk = 1 chain, keep-everything, and structural invariants).
"""

from __future__ import annotations

import numpy as np

NEAR = 1e-4


def log_softmax(y, temperature=1.0):
    z = np.asarray(y, dtype=np.float64) / float(temperature)
    m = np.max(z)
    return z - (m + np.log(np.sum(np.exp(z - m))))


def top_tokens(y, k):
    """The k tokens with the largest raw logits, lower id first on ties."""
    y = np.asarray(y, dtype=np.float64)
    order = np.lexsort((np.arange(y.size), -y))
    return [int(t) for t in order[:k]]


def _close(a, b):
    # equal scores are ordered by creation on any device (they come from equal
    # logits of one row, computed identically); only distinct, close scores
    # are ambiguous under rounding
    return a != b and abs(a - b) < NEAR


def build_tree(draft_logits, depth, topk, n_nodes, temperature=1.0):
    y = np.asarray(draft_logits, dtype=np.float64)
    B, R, V = y.shape
    assert R == 1 + (depth - 1) * topk and topk <= V
    total = topk + (depth - 1) * topk * topk
    assert 1 <= n_nodes <= 1 + total
    out = dict(tokens=np.full((B, n_nodes), -1, dtype=np.int64),
               parents=np.full((B, n_nodes), -1, dtype=np.int64),
               scores=np.zeros((B, n_nodes), dtype=np.float64),
               near_tie=np.zeros(B, dtype=bool))
    for b in range(B):
        lp = [log_softmax(y[b, r], temperature) for r in range(R)]
        cands = []          # dicts: depth, score, parent (candidate index or -1), token
        tie = False
        level = []
        for t in top_tokens(y[b, 0], topk):
            cands.append(dict(depth=1, score=float(lp[0][t]), parent=-1, token=t))
            level.append(len(cands) - 1)
        for d in range(2, depth + 1):
            ranked = sorted(level, key=lambda c: (-cands[c]["score"], c))
            s = [cands[c]["score"] for c in ranked[:topk + 1]]
            tie |= any(_close(s[i], s[i + 1]) for i in range(len(s) - 1))
            nxt = []
            for r, node in enumerate(ranked[:topk]):
                row = 1 + (d - 2) * topk + r
                for t in top_tokens(y[b, row], topk):
                    cands.append(dict(depth=d, score=cands[node]["score"] + float(lp[row][t]),
                                      parent=node, token=t))
                    nxt.append(len(cands) - 1)
            level = nxt
        ranked = sorted(range(len(cands)), key=lambda c: (-cands[c]["score"], c))
        keep = ranked[:n_nodes - 1]
        if 0 < n_nodes - 1 < len(cands):
            tie |= _close(cands[ranked[n_nodes - 2]]["score"], cands[ranked[n_nodes - 1]]["score"])
        keep_set = set(keep)
        assert all(cands[c]["parent"] == -1 or cands[c]["parent"] in keep_set for c in keep)
        order = sorted(keep, key=lambda c: (cands[c]["depth"], -cands[c]["score"], c))
        for i in range(len(order) - 1):
            a, c = order[i], order[i + 1]
            if cands[a]["depth"] == cands[c]["depth"] and _close(cands[a]["score"], cands[c]["score"]):
                tie = True
        new_id = {c: i + 1 for i, c in enumerate(order)}
        for c in order:
            n = new_id[c]
            out["tokens"][b, n] = cands[c]["token"]
            out["parents"][b, n] = 0 if cands[c]["parent"] == -1 else new_id[cands[c]["parent"]]
            out["scores"][b, n] = cands[c]["score"]
        out["near_tie"][b] = tie
    return out
