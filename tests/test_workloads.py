"""The seeded input generators produce the shapes, distributions and
structure the workload recipes state (CPU): logits N(0, std^2) in the stated
dtype, greedy drafts equal to the row argmax at the stated rate and another
id otherwise, stochastic drafts sampled from the draft softmax, draft logits
= target + N(0, 1), EAGLE-style trees (64 nodes, depth 5, BFS order, valid
parents, distinct sibling tokens, first child = parent argmax at the stated
rate), and determinism under a seed."""

import numpy as np
import torch

from speculative_decoding_verification_72_gb300 import workloads as W


def test_greedy_chain_recipe():
    B, K, V = 64, 5, 4096
    ci = W.greedy_chain(B=B, K=K, V=V, seed=11)
    assert ci.target.shape == (B, K + 1, V) and ci.target.dtype == torch.bfloat16
    assert ci.draft_tokens.shape == (B, K) and ci.draft_tokens.dtype == torch.int32
    assert ci.uniforms.shape == (B, K + 1)
    x = ci.target.float()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 3.0) < 0.01
    am = torch.argmax(ci.target[:, :K], dim=-1)
    match = (ci.draft_tokens.long() == am).float().mean().item()
    assert abs(match - 0.8) < 0.05                      # argmax w.p. 0.8 (B*K = 320 draws)
    assert ((ci.draft_tokens >= 0) & (ci.draft_tokens < V)).all()
    u = ci.uniforms
    assert (u >= 0).all() and (u < 1).all()


def test_long_chain_match_rate():
    ci = W.greedy_chain(B=2, K=2047, V=257, p_match=0.95, seed=12)
    am = torch.argmax(ci.target[:, :-1], dim=-1)
    match = (ci.draft_tokens.long() == am).float().mean().item()
    assert abs(match - 0.95) < 0.015


def test_stochastic_chain_recipe():
    B, K, V = 64, 4, 2000
    ci = W.stochastic_chain(B=B, K=K, V=V, seed=13)
    assert ci.target.dtype == torch.float32 and ci.draft_logits.shape == (B, K, V)
    noise = (ci.draft_logits - ci.target[:, :K]).double()
    assert abs(float(noise.mean())) < 0.01 and abs(float(noise.std()) - 1.0) < 0.01
    # drafts are samples of softmax(draft logits): the mean of q(d) over the
    # draws estimates E_q[q] = sum q^2 (far above the uniform 1 / V)
    q = torch.softmax(ci.draft_logits.double(), -1)
    picked = q.gather(-1, ci.draft_tokens.long().unsqueeze(-1)).squeeze(-1)
    expect = float((q * q).sum(-1).mean())
    sem = float(picked.std()) / (B * K) ** 0.5
    assert abs(float(picked.mean()) - expect) < 4 * sem + 1e-3
    assert expect > 20.0 / V


def test_toy_chain_recipe():
    ci = W.toy_chain()
    assert ci.target.shape == (4, 5, 32) and ci.draft_logits.shape == (4, 4, 32)
    q = torch.exp(ci.draft_logits.double())
    assert torch.allclose(q.sum(-1), torch.ones(4, 4, dtype=torch.float64), atol=1e-6)
    p = torch.softmax(ci.target[:, :4].double(), -1)
    assert (q >= 0.8 * p - 1e-6).all()                  # q = 0.8 p + 0.2 (something >= 0)


def test_eagle_tree_recipe():
    B, V = 8, 500
    ti = W.eagle_tree(B=B, V=V, dtype=torch.float32, seed=14)
    par, tok = ti.parents.numpy(), ti.node_tokens.numpy()
    assert par.shape == (B, 64) and (par[:, 0] == -1).all()
    am = torch.argmax(ti.target, dim=-1).numpy()
    first_hits = first_total = 0
    for b in range(B):
        depth = np.zeros(64, dtype=np.int64)
        for n in range(1, 64):
            assert 0 <= par[b, n] < n                    # parents precede children
            depth[n] = depth[par[b, n]] + 1
        assert depth.max() <= 5 and (np.diff(depth[1:]) >= 0).all()   # BFS order
        assert (depth == 1).sum() == 4                   # the root's topk children
        for n in range(64):
            kids = [c for c in range(1, 64) if par[b, c] == n]
            toks = tok[b, kids]
            assert len(set(toks.tolist())) == len(kids)  # distinct siblings
            assert len(kids) <= 4
            if kids:
                first_total += 1
                first_hits += int(toks[0] == am[b, n])
                assert (toks[1:] != am[b, n]).all()
    assert abs(first_hits / first_total - 0.8) < 0.12


def test_tree_shape_keeps_best_and_is_closed():
    rng = np.random.default_rng(3)
    for _ in range(20):
        par = W.tree_shape(rng)
        assert len(par) == 64 and par[0] == -1
        assert all(0 <= par[n] < n for n in range(1, 64))


def test_generators_are_deterministic():
    a = W.stochastic_chain(B=3, K=2, V=100, seed=5)
    b = W.stochastic_chain(B=3, K=2, V=100, seed=5)
    assert torch.equal(a.target, b.target) and torch.equal(a.draft_tokens, b.draft_tokens)
    assert torch.equal(a.uniforms, b.uniforms) and torch.equal(a.draft_logits, b.draft_logits)
    c = W.eagle_tree(B=2, V=50, seed=6)
    d = W.eagle_tree(B=2, V=50, seed=6)
    assert torch.equal(c.parents, d.parents) and torch.equal(c.node_tokens, d.node_tokens)
    e = W.draft_tree_rows(B=2, V=64, seed=7)
    assert e.shape == (2, 17, 64) and torch.equal(e, W.draft_tree_rows(B=2, V=64, seed=7))
