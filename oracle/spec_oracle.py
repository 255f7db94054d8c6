"""Float64 CPU oracle for batched speculative-decoding verification.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / --impl reference legs use this module. It shares no code with
the CUDA library and never imports it.

Everything here is plain NumPy in float64, one request at a time, written to be
checked by eye against the pages:

[NS] nanospec README, acceptance-rules paragraph: every emitted token carries
     its target log-prob and mu(a|s), the probability that the speculative
     sampler emitted it. Rules: exact (lossless); relaxed (accept iff
     p >= tau or the token is in the top-k; deterministic, so mu = 1 on an
     accepted draft); power (accept with probability min(1, p/rest)**alpha).
     Chain and tree (depth 5, topk 4) EAGLE-3 configurations.
[MS] mini-sglang PR #134 "[Feature] Vanilla speculative decoding",
     Modifications (verify.py): verify_drafts(draft_tokens, target_logits)
     accepts the argmax-matching prefix of the K drafts against the K+1
     verify-pass logits and appends the target's bonus token.
[SD] spec-decode README, "How it works" flowchart: accept each draft in order
     with min(1, p/q); on the first rejection emit a sample from
     normalize(relu(p - q)) and stop; if all are accepted emit a bonus token.
     "Provably exact": induced(t) = q(t) min(1, p(t)/q(t)) +
     (rejection mass) residual(p, q)(t), which equals p.

Readings taken where the pages are silent:
  * argmax breaks ties toward the lowest vocabulary index, on raw logits;
  * greedy log-probs are log_softmax(x) at temperature 1; sampled log-probs
    are log p_T with p_T = softmax(x / T), the distribution sampled from;
  * a draft is accepted iff u < a (strict), u the caller's uniform for it;
  * chain uniforms: column i tests draft i, column K drives the single final
    draw; tree uniforms: column c tests node c, column 0 drives the final draw;
  * the final draw is inverse-CDF in ascending vocabulary order: the smallest j
    whose inclusive prefix sum exceeds u * S (S the total weight); if rounding
    leaves none, the last index with positive weight;
  * q(t) = 0 < p(t) gives ratio 1; p(t) = q(t) = 0 rejects and sets
    STATUS_ZERO_MASS; zero residual mass falls back to drawing from p;
  * deterministic drafts (no draft logits, and every tree) use q = one-hot:
    children c_1..c_m of a node are tested in increasing node index with
    rest_1 = 1, rest_{j+1} = rest_j - p(c_j) over rejected, distinct, valid
    tokens; exact a_j = min(1, p/rest_j), power a_j = min(1, p/rest_j)**alpha,
    relaxed a_j = [p >= tau or rank < top_k] (rank = number of logits strictly
    greater); a duplicate of a rejected sibling's token has a_j = 0; when all
    are rejected the draw is from p with the rejected tokens zeroed, and mu is
    the probability of that whole branch;
  * with draft logits, power and relaxed use acc(t) = min(1, p/q)**alpha or
    [p >= tau or rank < top_k], the residual stays normalize(relu(p - q)), and
    mu(a) = q(a) acc(a) + (1 - sum_s q(s) acc(s)) res(a); exact gives mu = p;
  * a tree walk accepts at most max_depth nodes; at that depth a node with
    children is treated as a leaf and STATUS_DEPTH_EXCEEDED is set;
  * STATUS_NONFINITE_ROW is set for a row the decision reads (chain rows
    0..n, draft rows 0..min(n, K-1), the tree path's rows) whose maximum is
    not finite or which holds a NaN; rows after the decision are not read.

Parity status: every function below is pinned by tests/test_oracle_*.py
(closed forms, exact-rational brute force, scenario fixtures, Monte Carlo
against mu and the target law, special-case reductions).
"""

from __future__ import annotations

import numpy as np

STATUS_BAD_TOKEN = 1
STATUS_BAD_PARENT = 2
STATUS_NONFINITE_ROW = 4
STATUS_ZERO_MASS = 8
STATUS_DEPTH_EXCEEDED = 16

RULE_EXACT = 0
RULE_RELAXED = 1
RULE_POWER = 2

# An accept test with |u - a| < 1e-5 (or |p - tau| < 1e-5) is a near tie: an
# fp32 implementation may take the other branch there. For the final draw the
# same band around u * S gives the range of tokens that rounding can select.
NEAR_TIE = 1e-5


# ---------------------------------------------------------------- row math

def log_sum_exp(x, temperature=1.0):
    """log sum_j exp(x_j / T), max-shifted, float64 (NumPy pairwise sum)."""
    z = np.asarray(x, dtype=np.float64) / float(temperature)
    m = np.max(z)
    return float(m + np.log(np.sum(np.exp(z - m))))


def target_probs(x, temperature=1.0):
    """p_T = softmax(x / T) in float64."""
    z = np.asarray(x, dtype=np.float64) / float(temperature)
    return np.exp(z - log_sum_exp(x, temperature))


def first_argmax(x):
    """argmax with ties to the lowest index (NumPy returns the first maximum)."""
    return int(np.argmax(x))


def rank_of(x, t):
    """Number of logits strictly greater than x[t] (raw logits)."""
    return int(np.count_nonzero(x > x[t]))


def row_is_finite(x):
    """A row is usable when it has no NaN and its maximum is finite."""
    return bool(np.isfinite(np.max(x))) and not bool(np.isnan(x).any())


def residual(p, q):
    """normalize(relu(p - q)) [SD "How it works"]; None if the mass is zero."""
    w = np.maximum(p - q, 0.0)
    s = w.sum()
    if not s > 0.0:
        return None
    return w / s


def induced_from_dists(p, q):
    """Closed-form law of the first emitted token [SD "Provably exact"]:
    q(t) min(1, p(t)/q(t)) + (rejection mass) residual(p, q)(t)."""
    p = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    ratio = np.ones_like(p)
    pos = q > 0
    ratio[pos] = np.minimum(1.0, p[pos] / q[pos])
    accepted = q * ratio
    rejection_mass = 1.0 - accepted.sum()
    res = residual(p, q)
    if res is None:
        return accepted
    return accepted + rejection_mass * res


def inverse_cdf(w, u, band=NEAR_TIE):
    """Smallest j with C_j > u * S (C the inclusive prefix sum of w in index
    order, S = C[-1]); falls back to the last positive index.

    Also returns the relative distance from u * S to the chosen cell's nearer
    boundary, and the index range [j_lo, j_hi] of the cells that meet the
    band u * S +- band * S: a draw computed with a slightly different rounding
    of the prefix sums lands in that range."""
    w = np.asarray(w, dtype=np.float64)
    c = np.cumsum(w)
    s = c[-1]
    thr = u * s

    def first_above(t):
        hits = np.nonzero(c > t)[0]
        return int(hits[0]) if hits.size else int(np.nonzero(w > 0)[0][-1])

    j = first_above(thr)
    lo = c[j - 1] if j > 0 else 0.0
    margin = min(abs(thr - lo), abs(c[j] - thr)) / s
    return j, margin, first_above(thr - band * s), first_above(thr + band * s)


def _acceptance_vs_rest(rule, p_t, rest, rank, tau, top_k, alpha):
    """a_j for a deterministic draft token (q one-hot), see module header."""
    if rule == RULE_RELAXED:
        return 1.0 if (p_t >= tau or rank < top_k) else 0.0
    ratio = 1.0 if rest <= 0.0 else min(1.0, p_t / rest)
    if rule == RULE_POWER:
        return ratio ** alpha
    return ratio


def _acceptance_vs_q(rule, p, q, x, t, tau, top_k, alpha):
    """acc(t) for a draft token sampled from q, see module header."""
    if rule == RULE_RELAXED:
        return 1.0 if (p[t] >= tau or rank_of(x, t) < top_k) else 0.0
    ratio = 1.0 if q[t] == 0.0 else min(1.0, p[t] / q[t])
    if rule == RULE_POWER:
        return ratio ** alpha
    return ratio


def _acceptance_vector_vs_q(rule, p, q, x, tau, top_k, alpha):
    """acc(s) for every token s of a row (used for mu under power/relaxed)."""
    if rule == RULE_RELAXED:
        ranks = np.array([rank_of(x, s) for s in range(x.size)]) if top_k > 0 else None
        acc = (p >= tau).astype(np.float64)
        if ranks is not None:
            acc = np.maximum(acc, (ranks < top_k).astype(np.float64))
        return acc
    ratio = np.ones_like(p)
    pos = q > 0
    ratio[pos] = np.minimum(1.0, p[pos] / q[pos])
    if rule == RULE_POWER:
        return ratio ** alpha
    return ratio


def _empty_outputs(B, width):
    return dict(tokens=np.full((B, width), -1, dtype=np.int64),
                num_accepted=np.zeros(B, dtype=np.int64),
                logprob=np.zeros((B, width), dtype=np.float64),
                mu=np.zeros((B, width), dtype=np.float64),
                status=np.zeros(B, dtype=np.int64),
                tie_pos=np.full(B, -1, dtype=np.int64),
                draw_band=np.full((B, 2), -1, dtype=np.int64))


# ------------------------------------------------------------- greedy chain

def verify_greedy(target_logits, draft_tokens):
    """Greedy chain verification [MS Modifications, verify.py].

    target_logits [B, K+1, V], draft_tokens [B, K]. The accepted count n is the
    first i < K whose draft is out of range or differs from argmax(row i), else
    K; tokens = d_0..d_{n-1}, argmax(row n), then -1. logprob_j = x_j[tok_j] -
    lse(x_j) at T = 1, mu_j = 1 for the n + 1 emitted tokens, 0 after.
    """
    x = np.asarray(target_logits, dtype=np.float64)
    d = np.asarray(draft_tokens, dtype=np.int64)
    B, R, V = x.shape
    K = R - 1
    assert d.shape == (B, K)
    out = _empty_outputs(B, R)
    for b in range(B):
        n = K
        for i in range(K):
            t = d[b, i]
            if t < 0 or t >= V:
                out["status"][b] |= STATUS_BAD_TOKEN
                n = i
                break
            if t != first_argmax(x[b, i]):
                n = i
                break
        for j in range(n):
            out["tokens"][b, j] = d[b, j]
        out["tokens"][b, n] = first_argmax(x[b, n])
        for i in range(n + 1):          # the rows the decision read
            if not row_is_finite(x[b, i]):
                out["status"][b] |= STATUS_NONFINITE_ROW
        for j in range(n + 1):
            tok = out["tokens"][b, j]
            out["logprob"][b, j] = x[b, j, tok] - log_sum_exp(x[b, j], 1.0)
            out["mu"][b, j] = 1.0
        out["num_accepted"][b] = n
    return out


# --------------------------------------------------------- stochastic chain

def verify_sample(target_logits, draft_logits, draft_tokens, temperature,
                  uniforms, rule=RULE_EXACT, tau=0.0, top_k=0, alpha=1.0):
    """Stochastic chain verification [SD "How it works"; NS rules].

    target_logits [B, K+1, V]; draft_logits [B, K, V] or None (deterministic
    drafts, q = one-hot); draft_tokens [B, K]; uniforms [B, K+1] in [0, 1).
    Returns tokens / logprob / mu [B, K+1], num_accepted [B], status [B],
    tie_pos [B] (first position whose accept test was a near tie, else -1)
    and draw_band [B, 2] (tokens the final draw may take under rounding).
    """
    x = np.asarray(target_logits, dtype=np.float64)
    y = None if draft_logits is None else np.asarray(draft_logits, dtype=np.float64)
    d = np.asarray(draft_tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float64)
    B, R, V = x.shape
    K = R - 1
    T = float(temperature)
    assert T > 0.0 and d.shape == (B, K) and u.shape == (B, R)
    out = _empty_outputs(B, R)

    for b in range(B):
        status = 0
        tie = -1
        n = K
        final_w = None
        final_scale = 1.0   # probability of reaching the final draw's branch
        final_mu = None     # callable a -> mu under power/relaxed with q
        for i in range(K):
            t = d[b, i]
            p = target_probs(x[b, i], T)
            bad = t < 0 or t >= V
            if bad:
                status |= STATUS_BAD_TOKEN
            if y is None:
                # one candidate per position, rest_1 = 1 (module header)
                if bad:
                    a, margin = 0.0, np.inf
                else:
                    a = _acceptance_vs_rest(rule, p[t], 1.0, rank_of(x[b, i], t),
                                            tau, top_k, alpha)
                    margin = abs(p[t] - tau) if rule == RULE_RELAXED else abs(u[b, i] - a)
                if margin < NEAR_TIE and tie < 0:
                    tie = i
                if u[b, i] < a:
                    out["tokens"][b, i] = t
                    out["logprob"][b, i] = np.log(p[t])
                    out["mu"][b, i] = a
                    continue
                n = i
                w = p.copy()
                if not bad:
                    w[t] = 0.0
                if not w.sum() > 0.0:
                    w = p.copy()
                final_w = w
                final_scale = 1.0 - a
                break
            q = target_probs(y[b, i], T)
            if bad:
                a, margin = 0.0, np.inf
            elif p[t] == 0.0 and q[t] == 0.0:
                status |= STATUS_ZERO_MASS
                a, margin = 0.0, np.inf
            else:
                a = _acceptance_vs_q(rule, p, q, x[b, i], t, tau, top_k, alpha)
                margin = abs(p[t] - tau) if rule == RULE_RELAXED else abs(u[b, i] - a)
            if margin < NEAR_TIE and tie < 0:
                tie = i
            res = residual(p, q)
            if res is None:
                res = p
            if rule == RULE_EXACT:
                mu_of = (lambda a_, p_=p: p_[a_])
            else:
                acc = _acceptance_vector_vs_q(rule, p, q, x[b, i], tau, top_k, alpha)
                keep = float(np.sum(q * acc))
                mu_of = (lambda a_, q_=q, acc_=acc, keep_=keep, res_=res:
                         q_[a_] * acc_[a_] + (1.0 - keep_) * res_[a_])
            if u[b, i] < a:
                out["tokens"][b, i] = t
                out["logprob"][b, i] = np.log(p[t])
                out["mu"][b, i] = mu_of(t)
                continue
            n = i
            final_w = res
            final_mu = mu_of
            break
        if n == K:
            final_w = target_probs(x[b, K], T)
            final_mu = None
            final_scale = 1.0
        j, _, j_lo, j_hi = inverse_cdf(final_w, u[b, K])
        out["draw_band"][b] = (j_lo, j_hi)
        p_row = target_probs(x[b, n], T)
        out["tokens"][b, n] = j
        out["logprob"][b, n] = np.log(p_row[j])
        if final_mu is not None:
            out["mu"][b, n] = final_mu(j)
        elif y is None and n < K:
            out["mu"][b, n] = final_scale * final_w[j] / final_w.sum()
        else:
            out["mu"][b, n] = p_row[j]
        for i in range(n + 1):          # the rows the decision read
            if not row_is_finite(x[b, i]):
                status |= STATUS_NONFINITE_ROW
            if y is not None and i < K and not row_is_finite(y[b, i]):
                status |= STATUS_NONFINITE_ROW
        out["num_accepted"][b] = n
        out["status"][b] = status
        out["tie_pos"][b] = tie
    return out


# ---------------------------------------------------------------- tree walk

def tree_children(parents):
    """children[n] = nodes c with a valid link parents[c] = n, in increasing
    index; also returns whether every link was valid (parents[0] = -1 and
    0 <= parents[c] < c)."""
    N = len(parents)
    children = [[] for _ in range(N)]
    ok = int(parents[0]) == -1
    for c in range(1, N):
        pc = int(parents[c])
        if 0 <= pc < c:
            children[pc].append(c)
        else:
            ok = False
    return children, ok


def verify_tree(target_logits, node_tokens, parents, max_depth, temperature,
                uniforms=None, rule=RULE_EXACT, tau=0.0, top_k=0, alpha=1.0):
    """Tree verification [NS chain/tree configurations and rules].

    target_logits [B, N, V]: row n is the target's next-token logits after the
    path root..n. node_tokens [B, N] (node 0 is the root, its token unused),
    parents [B, N]. temperature == 0 selects the greedy walk (uniforms unused);
    otherwise uniforms [B, N]. Returns tokens / nodes / logprob / mu
    [B, max_depth + 1] (nodes[j] is the path node whose row scored token j),
    num_accepted, status, tie_pos.
    """
    x = np.asarray(target_logits, dtype=np.float64)
    tok = np.asarray(node_tokens, dtype=np.int64)
    par = np.asarray(parents, dtype=np.int64)
    B, N, V = x.shape
    greedy = float(temperature) == 0.0
    T = 1.0 if greedy else float(temperature)
    u = None if greedy else np.asarray(uniforms, dtype=np.float64)
    W = max_depth + 1
    out = _empty_outputs(B, W)
    out["nodes"] = np.full((B, W), -1, dtype=np.int64)

    for b in range(B):
        status = 0
        children, links_ok = tree_children(par[b])
        if not links_ok:
            status |= STATUS_BAD_PARENT
        tie = -1
        cur = 0
        depth = 0
        while True:
            cands = children[cur]
            if depth == max_depth and cands:
                status |= STATUS_DEPTH_EXCEEDED
                cands = []
            out["nodes"][b, depth] = cur
            if greedy:
                a = first_argmax(x[b, cur])
                nxt = None
                for c in cands:
                    t = tok[b, c]
                    if t < 0 or t >= V:
                        status |= STATUS_BAD_TOKEN
                        continue
                    if t == a:
                        nxt = c
                        break
                lp = x[b, cur, a] - log_sum_exp(x[b, cur], 1.0)
                out["tokens"][b, depth] = a
                out["logprob"][b, depth] = lp
                out["mu"][b, depth] = 1.0
                if nxt is None:
                    break
                cur = nxt
                depth += 1
                continue

            p = target_probs(x[b, cur], T)
            rest = 1.0
            prod = 1.0
            rejected = []
            accepted = None
            for c in cands:
                t = tok[b, c]
                if t < 0 or t >= V:
                    status |= STATUS_BAD_TOKEN
                    a, margin = 0.0, np.inf
                elif t in rejected:
                    a, margin = 0.0, np.inf
                else:
                    a = _acceptance_vs_rest(rule, p[t], rest, rank_of(x[b, cur], t),
                                            tau, top_k, alpha)
                    margin = abs(p[t] - tau) if rule == RULE_RELAXED else abs(u[b, c] - a)
                if margin < NEAR_TIE and tie < 0:
                    tie = depth
                if u[b, c] < a:
                    accepted = c
                    out["tokens"][b, depth] = t
                    out["logprob"][b, depth] = np.log(p[t])
                    out["mu"][b, depth] = prod * a
                    break
                prod *= (1.0 - a)
                if 0 <= t < V and t not in rejected:
                    rest -= p[t]
                    rejected.append(t)
            if accepted is not None:
                cur = accepted
                depth += 1
                continue
            w = p.copy()
            if rejected:
                w[rejected] = 0.0
            if not w.sum() > 0.0:
                w = p.copy()
            j, _, j_lo, j_hi = inverse_cdf(w, u[b, 0])
            out["draw_band"][b] = (j_lo, j_hi)
            out["tokens"][b, depth] = j
            out["logprob"][b, depth] = np.log(p[j])
            out["mu"][b, depth] = prod * w[j] / w.sum()
            break
        for j in range(depth + 1):      # the rows the walk read
            if not row_is_finite(x[b, out["nodes"][b, j]]):
                status |= STATUS_NONFINITE_ROW
        out["num_accepted"][b] = depth
        out["status"][b] = status
        out["tie_pos"][b] = tie
    return out
